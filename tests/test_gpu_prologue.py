"""GPU parity of the fused prologue: un-normalised q/k rows (per-row norms from
about 1.4 to 91) normalised inside the kernels (``qk_l2norm``), against the
oracle's fp64 normalisation followed by its token loop; and the packed conv
layout (q, k, v as column views of one bf16 tensor; g and beta as column
views of one fp32 tensor with row stride 2*nv)."""
import numpy as np
import pytest

import gdn_synth
import oracle
from tests.gpu_helpers import DeviceProblem, assert_parity, to_torch_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_17_gb300 import build

    build.build()
    oracle.build()


@pytest.mark.parametrize("T,nk,nv", [(64, 1, 1), (300, 2, 4), (1000, 4, 8)])
def test_prefill_prologue_dense(T, nk, nv):
    p = gdn_synth.make_problem(seed=6100 + T, B=2, T=T, nk=nk, nv=nv, h0_std=0.02, qk_raw=True)
    dp = DeviceProblem(p)
    dp.run()
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.token_loop(p, qk_l2norm=True)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label=f"prologue T={T} nk={nk} nv={nv}")


def test_prefill_prologue_varlen_state_table():
    p = gdn_synth.make_problem(seed=6200, B=4, lengths=[1, 65, 200, 127], nk=2, nv=4, h0_std=0.02,
                               qk_raw=True, pad_qk=8, pad_v=16, gb_stride=8)
    dp = DeviceProblem(p, state_table=True)
    dp.run()
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.token_loop(p, qk_l2norm=True)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="prologue varlen, state table")


def test_prefill_prologue_weak_decay():
    # weak decay carries the un-normalised scale through many chunks if it leaked
    p = gdn_synth.make_problem(seed=6300, B=1, T=1500, nk=2, nv=4, h0_std=0.02, gate_mu=-6.0,
                               gate_sigma=0.5, qk_raw=True)
    dp = DeviceProblem(p)
    dp.run()
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.token_loop(p, qk_l2norm=True)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="prologue weak decay")


@pytest.mark.parametrize("norm", [False, True])
def test_flag_honoured_on_half_length_rows(norm):
    # unit rows halved (exact in bf16): a stable recurrence either way, whose result
    # depends on whether the prologue restores the unit length
    p = gdn_synth.make_problem(seed=6400, B=1, T=200, nk=1, nv=2, h0_std=0.02)
    for name in ("q", "k"):
        setattr(p, name, gdn_synth.f32_to_bf16_bits(gdn_synth.bf16_bits_to_f32(getattr(p, name)) * np.float32(0.5)))
    dp = DeviceProblem(p, qk_l2norm=norm)
    dp.run()
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.token_loop(p, qk_l2norm=norm)
    o_other, _ = oracle.token_loop(p, qk_l2norm=not norm)
    assert np.linalg.norm(o_other - o_ref) > 0.1 * np.linalg.norm(o_ref)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label=f"half-length rows, qk_l2norm={norm}")


def test_decode_prologue_repeated_steps():
    import gated_delta_rule_17_gb300 as gdn

    p = gdn_synth.make_problem(seed=6500, B=3, T=30, nk=2, nv=4, h0_std=0.02, qk_raw=True)
    dp = DeviceProblem(p)

    def rows(x, t):
        return x.view(p.B, p.T, *x.shape[1:])[:, t]

    for t in range(p.T):
        gdn.decode(rows(dp.q, t), rows(dp.k, t), rows(dp.v, t), rows(dp.g, t), rows(dp.beta, t), dp.state,
                   rows(dp.out, t), nk=p.nk, nv=p.nv, qk_l2norm=True)
    torch.cuda.synchronize()
    gdn.check()
    o_ref, s_ref = oracle.token_loop(p, qk_l2norm=True)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="decode prologue x30")


@pytest.mark.parametrize("norm", [False, True])
def test_packed_conv_layout(norm):
    # q | k | v side by side in one bf16 row of conv_dim = 2 nk dk + nv dv columns,
    # g | beta side by side in one fp32 row of 2 nv columns
    import gated_delta_rule_17_gb300 as gdn

    B, T, nk, nv = 2, 200, 2, 4
    p = gdn_synth.make_problem(seed=6600, B=B, T=T, nk=nk, nv=nv, h0_std=0.02, qk_raw=norm)
    rows, qd, vd = p.rows, nk * 128, nv * 128
    conv = np.zeros((rows, 2 * qd + vd), dtype=np.uint16)
    conv[:, :qd], conv[:, qd:2 * qd], conv[:, 2 * qd:] = p.q[:, :qd], p.k[:, :qd], p.v[:, :vd]
    gb = np.zeros((rows, 2 * nv), dtype=np.float32)
    gb[:, :nv], gb[:, nv:] = p.g[:, :nv], p.beta[:, :nv]
    conv_d = to_torch_bf16(conv, "cuda")
    gb_d = torch.from_numpy(gb).cuda()
    state = torch.from_numpy(p.h0.copy()).cuda()
    out = torch.full((rows, vd), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdn.prefill(conv_d[:, :qd], conv_d[:, qd:2 * qd], conv_d[:, 2 * qd:], gb_d[:, :nv], gb_d[:, nv:], state, out,
                nk=nk, nv=nv, B=B, T=T, qk_l2norm=norm)
    torch.cuda.synchronize()
    gdn.check()
    o_ref, s_ref = oracle.token_loop(p, qk_l2norm=norm)
    o = out.float().cpu().numpy().astype(np.float64).reshape(rows, nv, 128)
    assert_parity(o, state.cpu().numpy().astype(np.float64), o_ref, s_ref, label=f"packed conv layout norm={norm}")
