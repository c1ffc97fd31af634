"""GPU parity of the segment-parallel schedule for long sequences with few chains.

A dense batch with few (sequence, head) chains and enough chunks is cut into G
segments: the affine state maps of segments 0 .. G-2 (M from S = I with v = 0, N
from S = 0) are computed by output-free runs in parallel, the combine steps chain
X_{g+1} = M_g X_g + N_g from the carried-in state, and every segment then runs from
its entry state. Every case is checked against the oracle's token loop over the
whole sequence, and against the serial schedule (the allocation-free entry point,
which never segments)."""
import numpy as np
import pytest

import gdn_synth
import oracle
from tests.gpu_helpers import DeviceProblem, assert_parity, compare

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_17_gb300 import build

    build.build()
    oracle.build()


def _segments(p):
    """(G, L) the library's plan takes for a dense problem on this device."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    chains = p.B * p.nv
    nchunks = (p.T + 63) // 64
    if chains * 2 > sms:
        return 0, 0
    G = min(sms // (2 * chains) + 1, nchunks // 8, 8)
    if G < 2:
        return 0, 0
    L = (nchunks + G - 1) // G
    G = (nchunks + L - 1) // L
    return (G, L) if G >= 2 else (0, 0)


def run_serial(dp):
    import gated_delta_rule_17_gb300 as gdn

    p = dp.p
    gdn.prefill_noalloc(dp.q, dp.k, dp.v, dp.g, dp.beta, dp.state, dp.out, nk=p.nk, nv=p.nv, B=p.B, T=p.T,
                        state_is_table=dp.table, qk_l2norm=dp.qk_l2norm)


@pytest.mark.parametrize("T", [4096, 4096 + 37, 1500, 1024])
def test_segmented_matches_oracle_and_serial(T):
    import gated_delta_rule_17_gb300 as gdn

    p = gdn_synth.make_problem(seed=7100 + T, B=1, T=T, nk=2, nv=4, h0_std=0.02)
    G, _ = _segments(p)
    assert G >= 2, "the case must take the segment schedule"
    dp = DeviceProblem(p)
    dp.run()
    torch.cuda.synchronize()
    gdn.check()
    assert gdn.last_launch_count() == 3 + G  # WY, setup, phase 1, G-1 combines, phase 2
    o_ref, s_ref = oracle.token_loop(p)
    out_seg, st_seg = dp.out_np(), dp.state_np()
    assert_parity(out_seg, st_seg, o_ref, s_ref, label=f"segmented T={T} G={G}")
    ser = DeviceProblem(p)
    run_serial(ser)
    torch.cuda.synchronize()
    gdn.check()
    assert gdn.last_launch_count() == 2
    out_ser, st_ser = ser.out_np(), ser.state_np()
    assert_parity(out_ser, st_ser, o_ref, s_ref, label=f"serial T={T}")
    # the two schedules agree with each other as closely as each agrees with the oracle
    r_seg = compare(out_seg, st_seg, o_ref, s_ref)
    r_x = compare(out_seg, st_seg, out_ser, st_ser)
    assert r_x[0] <= 2 * max(r_seg[0], 1e-4) and r_x[2] <= 2 * max(r_seg[2], 1e-5)


def test_segmented_weak_decay_long_range():
    # near-zero log-gates (the long-context workload's distribution): the state carries
    # across every segment boundary
    p = gdn_synth.make_problem(seed=7200, B=2, T=3000, nk=1, nv=2, h0_std=0.02, gate_mu=-3.0, gate_sigma=0.5)
    assert _segments(p)[0] >= 2
    dp = DeviceProblem(p)
    dp.run()
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.token_loop(p)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="segmented weak decay B=2")


def test_segmented_state_table_and_prologue():
    p = gdn_synth.make_problem(seed=7300, B=2, T=2048 + 5, nk=2, nv=4, h0_std=0.02, qk_raw=True)
    assert _segments(p)[0] >= 2
    dp = DeviceProblem(p, state_table=True)
    dp.run()
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.token_loop(p, qk_l2norm=True)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="segmented state table + qk_l2norm")


def test_segmented_zero_gates():
    # g = 0: no decay at all, so the segment maps M are far from the identity's decayed
    # multiple and errors would accumulate over the combine chain
    p = gdn_synth.make_problem(seed=7400, B=1, T=4096, nk=1, nv=4, h0_std=0.02, gate_zero=True)
    assert _segments(p)[0] >= 2
    dp = DeviceProblem(p)
    dp.run()
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.token_loop(p)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="segmented zero gates")


def test_workspace_entry_point_segments_or_not():
    # gdn_prefill_ex on a dense batch: with the plan's workspace it segments, without it
    # it runs the serial schedule; both match the oracle
    import gated_delta_rule_17_gb300 as gdn

    p = gdn_synth.make_problem(seed=7500, B=1, T=2000, nk=1, nv=2, h0_std=0.02)
    G, _ = _segments(p)
    assert G >= 2
    nbytes = gdn.workspace_bytes(p.B, p.T, p.nv, varlen=False)
    assert nbytes > 0
    o_ref, s_ref = oracle.token_loop(p)
    dp = DeviceProblem(p)
    dp.run(workspace=torch.empty(nbytes, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert gdn.last_launch_count() == 3 + G
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="ex with workspace")
    dp2 = DeviceProblem(p)
    dp2.run(workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert gdn.last_launch_count() == 2
    assert_parity(dp2.out_np(), dp2.state_np(), o_ref, s_ref, label="ex without workspace")


def test_long_context_config_segmented_all_heads():
    # the T=65536 long-context workload itself: 1024 chunks per chain in 3 segments,
    # every head compared with the oracle
    import gated_delta_rule_17_gb300 as gdn

    p = gdn_synth.config_problem(4)
    assert _segments(p)[0] == 3
    dp = DeviceProblem(p)
    dp.run()
    torch.cuda.synchronize()
    gdn.check()
    o_ref, s_ref = oracle.token_loop(p)
    assert_parity(dp.out_np(), dp.state_np(), o_ref, s_ref, label="config 4 segmented")
