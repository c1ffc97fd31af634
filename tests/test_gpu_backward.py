"""GPU parity of the backward (gdn_prefill_backward) against the oracle's fp64
backward (itself pinned by finite differences): every gradient -- q, k, v, g,
beta and the initial state -- on dense GQA batches with and without a final-state
cotangent, sequences spanning several 64-token recompute blocks with a ragged
tail, a varlen batch with an empty sequence and a state table, and nk = nv."""
import numpy as np
import pytest

import gdn_synth
import oracle
from tests.gpu_helpers import to_torch_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

REL_L2 = 2e-3  # fp32 accumulation over up to ~1000 reverse steps from bf16 inputs


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_17_gb300 import build

    build.build()
    oracle.build()


def run_backward(p, seed, with_dst=True, state_table=False, workspace=True):
    import gated_delta_rule_17_gb300 as gdn

    rng = np.random.default_rng(seed)
    dout = rng.standard_normal((p.rows, p.nv, p.dv)).astype(np.float32)
    dst = rng.standard_normal((p.B, p.nv, p.dk, p.dv)).astype(np.float32) if with_dst else None
    dev = "cuda"
    q, k, v = (to_torch_bf16(x, dev) for x in (p.q, p.k, p.v))
    g, beta = torch.from_numpy(p.g).to(dev), torch.from_numpy(p.beta).to(dev)
    if state_table:
        states = [torch.from_numpy(p.h0[s].copy()).to(dev) for s in range(p.B)]
        h0 = torch.tensor([t.data_ptr() for t in states], dtype=torch.int64, device=dev)
    else:
        h0 = torch.from_numpy(p.h0.copy()).to(dev)
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"dq": torch.full((p.rows, p.nk * p.dk), float("nan"), **f32),
           "dk": torch.full((p.rows, p.nk * p.dk), float("nan"), **f32),
           "dv": torch.full((p.rows, p.nv * p.dv), float("nan"), **f32),
           "dg": torch.full((p.rows, p.nv), float("nan"), **f32),
           "dbeta": torch.full((p.rows, p.nv), float("nan"), **f32),
           "dh0": torch.full((p.B, p.nv, p.dk, p.dv), float("nan"), **f32)}
    cu = None if p.cu_seqlens is None else torch.from_numpy(p.cu_seqlens).to(dev)
    ws = None
    if workspace:
        ws = torch.empty(gdn.backward_workspace_bytes(p.B, p.T, p.nv, p.varlen), dtype=torch.uint8, device=dev)
    gdn.backward(q, k, v, g, beta, h0, torch.from_numpy(dout.reshape(p.rows, -1)).to(dev), out["dq"], out["dk"],
                 out["dv"], out["dg"], out["dbeta"], nk=p.nk, nv=p.nv, B=p.B, T=p.T, cu_seqlens=cu,
                 dST=None if dst is None else torch.from_numpy(dst).to(dev), dh0=out["dh0"],
                 state_is_table=state_table, workspace=ws)
    torch.cuda.synchronize()
    gdn.check()
    assert gdn.last_launch_count() == 2
    ref = oracle.token_loop_backward(p, dout.astype(np.float64), None if dst is None else dst.astype(np.float64))
    return {n: t.cpu().numpy().astype(np.float64) for n, t in out.items()}, ref


def assert_grads(got, ref, label):
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        a = got[name].reshape(-1)
        b = ref[name].reshape(-1)
        assert np.isfinite(a).all(), f"{label}: {name} has non-finite values"
        rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
        assert rel <= REL_L2, f"{label}: {name} rel L2 {rel:.3e}"


@pytest.mark.parametrize("T", [1, 64, 200])
def test_backward_dense_gqa(T):
    p = gdn_synth.make_problem(seed=8100 + T, B=2, T=T, nk=2, nv=4, h0_std=0.02)
    got, ref = run_backward(p, 8100 + T)
    assert_grads(got, ref, f"dense T={T}")


def test_backward_long_ragged_no_final_cotangent():
    # 1000 tokens: 16 recompute blocks, the last one 40 tokens; dL/dS_T = 0
    p = gdn_synth.make_problem(seed=8200, B=1, T=1000, nk=1, nv=2, h0_std=0.02)
    got, ref = run_backward(p, 8200, with_dst=False)
    assert_grads(got, ref, "dense T=1000 no dS_T")


def test_backward_weak_decay():
    p = gdn_synth.make_problem(seed=8300, B=1, T=700, nk=1, nv=1, h0_std=0.02, gate_mu=-4.0, gate_sigma=0.5)
    got, ref = run_backward(p, 8300)
    assert_grads(got, ref, "weak decay")


def test_backward_varlen_state_table_allocating():
    p = gdn_synth.make_problem(seed=8400, B=4, lengths=[65, 0, 130, 7], nk=2, nv=4, h0_std=0.02)
    got, ref = run_backward(p, 8400, state_table=True, workspace=False)
    assert_grads(got, ref, "varlen state table")


def test_backward_one_head_per_key():
    p = gdn_synth.make_problem(seed=8500, B=3, T=90, nk=3, nv=3, h0_std=0.02)
    got, ref = run_backward(p, 8500)
    assert_grads(got, ref, "nk = nv")


@pytest.mark.parametrize("B,cols", [(4, 2), (5, 4)])
def test_backward_wide_batches_use_wider_column_blocks(B, cols):
    # 128 chains take 2 CTAs of 64 columns per (sequence, head), 160 chains one CTA of
    # 128 columns (the kernel variants with 2 and 4 columns per thread); a ragged last
    # recompute block
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    chains = B * 32
    expect = 1 if chains * 4 <= 3 * sms else (2 if chains * 2 <= 2 * sms else 4)
    assert expect == cols, "the case must select the intended variant on this device"
    p = gdn_synth.make_problem(seed=8600 + B, B=B, T=70, nk=16, nv=32, h0_std=0.02)
    got, ref = run_backward(p, 8600 + B)
    assert_grads(got, ref, f"B={B} nv=32 ({cols} columns per thread)")
