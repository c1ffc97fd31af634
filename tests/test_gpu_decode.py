"""GPU parity of the single-token decode step (gdn_decode) against the fp64
oracle: one token per sequence, repeated steps against the oracle's token loop
over the whole sequence, GQA, state tables, padded strides and the batch a
serving step would use."""
import pytest

import gdn_synth
import oracle
from tests.gpu_helpers import DeviceProblem, assert_parity

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_17_gb300 import build

    build.build()
    oracle.build()


def _decode_rows(dp, t):
    """Views of token t of every sequence of a dense problem (rows b*T + t)."""
    p = dp.p

    def rows(x):
        return x.view(p.B, p.T, *x.shape[1:])[:, t]

    return rows(dp.q), rows(dp.k), rows(dp.v), rows(dp.g), rows(dp.beta), rows(dp.out)


def run_decode_steps(dp):
    import gated_delta_rule_17_gb300 as gdn

    p = dp.p
    for t in range(p.T):
        q, k, v, g, beta, out = _decode_rows(dp, t)
        gdn.decode(q, k, v, g, beta, dp.state, out, nk=p.nk, nv=p.nv, state_is_table=dp.table)
    torch.cuda.synchronize()
    gdn.check()


@pytest.mark.parametrize("B,nk,nv", [(1, 1, 1), (7, 2, 4), (16, 16, 32)])
def test_single_step_matches_oracle(B, nk, nv):
    p = gdn_synth.make_problem(seed=5100 + B, B=B, T=1, nk=nk, nv=nv, h0_std=0.02)
    dp = DeviceProblem(p)
    run_decode_steps(dp)
    o_ref, s_ref = oracle.token_loop(p)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label=f"decode B={B} nk={nk} nv={nv}")


@pytest.mark.parametrize("gate", ["default", "zero"])
def test_repeated_steps_follow_the_recurrence(gate):
    # 40 decode steps from a non-zero state = the oracle's token loop over 40 tokens
    kw = dict(gate_zero=True) if gate == "zero" else {}
    p = gdn_synth.make_problem(seed=5200, B=3, T=40, nk=2, nv=4, h0_std=0.02, **kw)
    dp = DeviceProblem(p)
    run_decode_steps(dp)
    o_ref, s_ref = oracle.token_loop(p)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label=f"decode x40 ({gate} gates)")


def test_decode_continues_a_prefill():
    # prefill of the first 100 tokens, then 20 decode steps: the oracle's 120-token loop
    import gated_delta_rule_17_gb300 as gdn

    full = gdn_synth.make_problem(seed=5300, B=2, T=120, nk=2, nv=4, h0_std=0.02)
    dp = DeviceProblem(full)
    p = full
    q, k, v, g, beta, out = (x.view(p.B, p.T, *x.shape[1:]) for x in (dp.q, dp.k, dp.v, dp.g, dp.beta, dp.out))
    pre = [x[:, :100].contiguous().view(p.B * 100, *x.shape[2:]) for x in (q, k, v, g, beta)]
    pre_out = torch.empty((p.B * 100, p.nv * p.dv), dtype=torch.bfloat16, device="cuda")
    gdn.prefill(*pre, dp.state, pre_out, nk=p.nk, nv=p.nv, B=p.B, T=100)
    for t in range(100, 120):
        gdn.decode(q[:, t], k[:, t], v[:, t], g[:, t], beta[:, t], dp.state, out[:, t], nk=p.nk, nv=p.nv)
    torch.cuda.synchronize()
    gdn.check()
    out[:, :100] = pre_out.view(p.B, 100, -1)
    o_ref, s_ref = oracle.token_loop(full)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="prefill 100 + decode 20")


def test_state_table_and_padded_strides():
    p = gdn_synth.make_problem(seed=5400, B=5, T=3, nk=2, nv=6, h0_std=0.02)
    dp = DeviceProblem(p, state_table=True, out_pad=24)
    run_decode_steps(dp)
    o_ref, s_ref = oracle.token_loop(p)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="decode, state table, padded out rows")


def test_serving_batch():
    # a serving-sized step: 128 sequences x 32 heads
    p = gdn_synth.make_problem(seed=5500, B=128, T=1, nk=16, nv=32, h0_std=0.02)
    dp = DeviceProblem(p)
    run_decode_steps(dp)
    o_ref, s_ref = oracle.token_loop(p)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="decode B=128 nv=32")
