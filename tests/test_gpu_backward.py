"""GPU parity of the chunked backward (gdn_prefill_backward) against the oracle's
fp64 token-by-token backward (itself pinned by finite differences): every
gradient -- q, k, v, g, beta and the initial state -- on dense GQA batches with
and without a final-state cotangent, sequences of many chunks with a ragged last
chunk, weak decay over long sequences (where errors would build up along both
chains), a varlen batch with an empty sequence and a state table, nk = nv, more
(sequence, head) chains than SMs, and one key-head group of the benchmark
workload."""
import numpy as np
import pytest

import gdn_synth
import oracle
from tests.gpu_helpers import to_torch_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# fp16 tensor-core operands (2^-11 relative rounding) for every contraction; the two
# chains carry fp32 states split into fp16 hi + lo. Each gradient is a sum of a few
# such products, so errors of a few 1e-4 are expected; the bound leaves margin.
REL_L2 = 3e-3
# Element-wise bound as well, so that a local error (one head, one chunk, a few rows)
# cannot hide inside a small whole-tensor norm. Per gradient and element,
#     |error| <= MAX_OVER_RMS * rms(oracle gradient) + MAX_REL * |oracle element|:
# the rms term bounds the error of ordinary elements, the relative term admits the
# fp16-operand rounding (~1e-3 relative) of the few elements tens of rms in size (dk
# of the B=4 T=8192 workload has such elements). A wrong head, chunk or row gives
# errors of the order of the elements themselves and fails it.
MAX_OVER_RMS = 5e-2
MAX_REL = 1e-2


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
    assert gdn.last_launch_count() == (5 if p.varlen else 4)
    ref = oracle.token_loop_backward(p, dout.astype(np.float64), None if dst is None else dst.astype(np.float64))
    return {n: t.cpu().numpy().astype(np.float64) for n, t in out.items()}, ref


def assert_grads(got, ref, label):
    rels, maxs = {}, {}
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        a = got[name].reshape(-1)
        b = ref[name].reshape(-1)
        assert np.isfinite(a).all(), f"{label}: {name} has non-finite values"
        rels[name] = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
        rms = max(np.sqrt(np.mean(b * b)), 1e-30)
        err = np.abs(a - b)
        i = int(err.argmax())
        maxs[name] = err[i] / rms
        excess = err - (MAX_OVER_RMS * rms + MAX_REL * np.abs(b))
        worst = int(excess.argmax())
        print(f"{label}: {name} rel L2 {rels[name]:.2e}, max |err|/rms {maxs[name]:.2e} at flat index {i} "
              f"(|ref|/rms {abs(b[i]) / rms:.1f}, rel err there {err[i] / max(abs(b[i]), 1e-30):.2e}), "
              f"{int((err > MAX_OVER_RMS * rms).sum())} elements above {MAX_OVER_RMS} rms")
        assert rels[name] <= REL_L2, f"{label}: {name} rel L2 {rels[name]:.3e}"
        assert excess[worst] <= 0, (f"{label}: {name} element {worst}: |err| {err[worst]:.3e} above "
                                    f"{MAX_OVER_RMS} rms + {MAX_REL} |ref| (rms {rms:.3e}, ref {b[worst]:.3e})")


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


@pytest.mark.parametrize("group", [4, 8])
def test_backward_wide_gqa_groups(group):
    # 4 and 8 value heads per key head: the per-chunk gradient kernel walks the whole group
    # in one CTA, accumulating dq and dk over it, with a ragged last chunk
    p = gdn_synth.make_problem(seed=8550 + group, B=2, T=150, nk=2, nv=2 * group, h0_std=0.02)
    got, ref = run_backward(p, 8550 + group)
    assert_grads(got, ref, f"{group} value heads per key head")


@pytest.mark.parametrize("B", [4, 5])
def test_backward_many_chains(B):
    # 128 and 160 (sequence, head) chains (more than the SMs: a second wave) of 70 tokens
    p = gdn_synth.make_problem(seed=8600 + B, B=B, T=70, nk=16, nv=32, h0_std=0.02)
    got, ref = run_backward(p, 8600 + B)
    assert_grads(got, ref, f"B={B} nv=32")


def test_backward_weak_decay_long():
    # 2000 tokens (32 chunks) with gates near zero: both chains carry their state far
    p = gdn_synth.make_problem(seed=8700, B=1, T=2000, nk=1, nv=2, h0_std=0.02, gate_mu=-5.0, gate_sigma=0.5)
    got, ref = run_backward(p, 8700)
    assert_grads(got, ref, "weak decay T=2000")


@pytest.mark.parametrize("config,khs", [(2, (0, 5)), (4, (11, 15))])
def test_backward_large_workloads_two_key_heads(config, khs):
    # The B=4 T=8192 nk=16 nv=32 workload (the benchmark's launch configuration) and the
    # B=1 T=65536 long-context one (1024 chunks of gates near zero: errors could build up
    # along both chains); the oracle runs two key heads' groups (two value heads each),
    # which fixes dq and dk of those key heads and every gradient of those value heads.
    import gated_delta_rule_17_gb300 as gdn

    p = gdn_synth.config_problem(config)
    rng = np.random.default_rng(8800 + config)
    dout = rng.standard_normal((p.rows, p.nv, p.dv)).astype(np.float32)
    dst = rng.standard_normal((p.B, p.nv, p.dk, p.dv)).astype(np.float32)
    dev = "cuda"
    q, k, v = (to_torch_bf16(x, dev) for x in (p.q, p.k, p.v))
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"dq": torch.empty((p.rows, p.nk * p.dk), **f32), "dk": torch.empty((p.rows, p.nk * p.dk), **f32),
           "dv": torch.empty((p.rows, p.nv * p.dv), **f32), "dg": torch.empty((p.rows, p.nv), **f32),
           "dbeta": torch.empty((p.rows, p.nv), **f32), "dh0": torch.empty((p.B, p.nv, p.dk, p.dv), **f32)}
    gdn.backward(q, k, v, torch.from_numpy(p.g).to(dev), torch.from_numpy(p.beta).to(dev),
                 torch.from_numpy(p.h0.copy()).to(dev), torch.from_numpy(dout.reshape(p.rows, -1)).to(dev),
                 out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"], nk=p.nk, nv=p.nv, B=p.B, T=p.T,
                 dST=torch.from_numpy(dst).to(dev), dh0=out["dh0"])
    torch.cuda.synchronize()
    gdn.check()
    got = {n: t.cpu().numpy().astype(np.float64) for n, t in out.items()}
    del out, q, k, v
    grp = p.nv // p.nk
    d = p.dk
    # both key heads' groups in one oracle call: key heads khs as a 2-key-head problem
    kcols = np.concatenate([np.arange(kh * d, (kh + 1) * d) for kh in khs])
    heads = np.concatenate([np.arange(kh * grp, (kh + 1) * grp) for kh in khs])
    vcols = np.concatenate([np.arange(h * d, (h + 1) * d) for h in heads])
    sub = gdn_synth.Problem(B=p.B, T=p.T, nk=len(khs), nv=len(heads), dk=d, dv=d,
                            q=np.ascontiguousarray(p.q[:, kcols]), k=np.ascontiguousarray(p.k[:, kcols]),
                            v=np.ascontiguousarray(p.v[:, vcols]), g=np.ascontiguousarray(p.g[:, heads]),
                            beta=np.ascontiguousarray(p.beta[:, heads]), h0=np.ascontiguousarray(p.h0[:, heads]))
    ref = oracle.token_loop_backward(sub, dout[:, heads].astype(np.float64), dst[:, heads].astype(np.float64))
    mine = {"dq": got["dq"][:, kcols], "dk": got["dk"][:, kcols], "dv": got["dv"][:, vcols],
            "dg": got["dg"][:, heads], "dbeta": got["dbeta"][:, heads], "dh0": got["dh0"][:, heads]}
    assert_grads(mine, ref, f"{gdn_synth.CONFIG_NAMES[config]}, key heads {khs}")
