"""GPU tests of the end-to-end entry point from page-locked host memory
(``gdn_prefill_host``): the copies in, the op and the copies out in one call,
pipelined over chunk ranges for long dense batches. Its results must equal the
device entry point's bit for bit, and the oracle's within the tolerances."""
import ctypes

import numpy as np
import pytest

import gdn_synth
import oracle
from tests.gpu_helpers import DeviceProblem, assert_parity, to_torch_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_17_gb300 import build

    build.build()
    oracle.build()


class HostProblem:
    """Page-locked host copies of a problem's inputs, state and output rows."""

    def __init__(self, p):
        self.p = p
        self.q = to_torch_bf16(p.q, "cpu").pin_memory()
        self.k = to_torch_bf16(p.k, "cpu").pin_memory()
        self.v = to_torch_bf16(p.v, "cpu").pin_memory()
        self.g = torch.from_numpy(p.g).pin_memory()
        self.beta = torch.from_numpy(p.beta).pin_memory()
        self.state = torch.from_numpy(p.h0.copy()).pin_memory()
        self.cu = None if p.cu_seqlens is None else torch.from_numpy(p.cu_seqlens).pin_memory()
        self.out = torch.full((p.rows, p.nv * p.dv), float("nan"), dtype=torch.bfloat16).pin_memory()

    def run(self, scratch=None, qk_l2norm=None):
        import gated_delta_rule_17_gb300 as gdn

        p = self.p
        gdn.prefill_host(self.q, self.k, self.v, self.g, self.beta, self.state, self.out, nk=p.nk, nv=p.nv,
                         B=p.B, T=p.T, cu_seqlens=self.cu, scratch=scratch,
                         qk_l2norm=p.meta.get("qk_raw", False) if qk_l2norm is None else qk_l2norm)

    def out_np(self):
        return self.out.float().numpy().astype(np.float64).reshape(self.p.rows, self.p.nv, self.p.dv)

    def state_np(self):
        return self.state.numpy().astype(np.float64)


def _device_run(p, workspace):
    import gated_delta_rule_17_gb300 as gdn

    dp = DeviceProblem(p)
    dp.run(workspace=workspace)
    torch.cuda.synchronize()
    gdn.check()
    return dp


def test_pipelined_ranges_equal_device_path_and_oracle():
    # 96 chains of 41 chunks (ragged last chunk): no segment schedule, so the call cuts
    # the sequences into 2 chunk ranges whose copies overlap the op
    import gated_delta_rule_17_gb300 as gdn

    p = gdn_synth.make_problem(seed=3900, B=3, T=40 * 64 + 17, nk=16, nv=32, h0_std=0.02)
    hp = HostProblem(p)
    hp.run()
    torch.cuda.synchronize()
    gdn.check()
    assert gdn.last_launch_count() == 4  # a WY solve and a spine per range
    dp = _device_run(p, torch.empty(0, dtype=torch.uint8, device="cuda"))
    np.testing.assert_array_equal(hp.out_np(), dp.out_np())
    np.testing.assert_array_equal(hp.state_np(), dp.state_np())
    o_ref, s_ref = oracle.token_loop(p)
    assert_parity(hp.out_np(), hp.state_np(), o_ref, s_ref, label="host entry point, 2 ranges")


def test_given_scratch_fused_norms_repeated_calls():
    # caller scratch, raw q/k rows normalised in the kernels, and a second call that
    # carries the state on: both calls equal the device path's
    import gated_delta_rule_17_gb300 as gdn

    p = gdn_synth.make_problem(seed=3901, B=2, T=48 * 64, nk=20, nv=40, h0_std=0.02, qk_raw=True)
    scratch = torch.empty(gdn.host_scratch_bytes(p.B, p.T, p.nk, p.nv, False), dtype=torch.uint8, device="cuda")
    hp = HostProblem(p)
    dp = DeviceProblem(p)
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        hp.run(scratch=scratch)
        dp.run(workspace=empty)
        torch.cuda.synchronize()
        gdn.check()
        np.testing.assert_array_equal(hp.out_np(), dp.out_np())
        np.testing.assert_array_equal(hp.state_np(), dp.state_np())


@pytest.mark.parametrize("case", ["varlen", "segments"])
def test_single_pass_cases_equal_device_path(case):
    # varlen batches and dense batches that take the segment schedule run as one pass:
    # everything in, the op, everything out
    import gated_delta_rule_17_gb300 as gdn

    if case == "varlen":
        p = gdn_synth.make_problem(seed=3902, B=3, lengths=[100, 5, 3000], nk=2, nv=4, h0_std=0.02)
        dp = _device_run(p, None)
    else:
        p = gdn_synth.make_problem(seed=3903, B=1, T=4096, nk=2, nv=4, h0_std=0.02)
        dp = _device_run(p, None)  # with the queried workspace: the segment schedule
    hp = HostProblem(p)
    hp.run()
    torch.cuda.synchronize()
    gdn.check()
    assert gdn.last_launch_count() >= 2
    np.testing.assert_array_equal(hp.out_np(), dp.out_np())
    np.testing.assert_array_equal(hp.state_np(), dp.state_np())
    o_ref, s_ref = oracle.token_loop(p)
    assert_parity(hp.out_np(), hp.state_np(), o_ref, s_ref, label=f"host entry point, {case}")


def test_rejects_pageable_host_memory_before_launch():
    import gated_delta_rule_17_gb300 as gdn

    p = gdn_synth.make_problem(seed=3904, B=1, T=128, nk=1, nv=1)
    hp = HostProblem(p)
    pageable = hp.q.clone()  # not page-locked
    assert not pageable.is_pinned()
    with pytest.raises(gdn.GdnError) as ei:
        gdn.prefill_host(pageable, hp.k, hp.v, hp.g, hp.beta, hp.state, hp.out, nk=1, nv=1, B=1, T=128)
    assert ei.value.code == gdn.GDN_ERR_ARG
    # the C entry point checks the memory type itself
    lib = gdn.load()
    st = gdn.Strides(128, 128, 128, 1, 1, 128, 0, 0)
    rc = lib.gdn_prefill_host(pageable.data_ptr(), hp.k.data_ptr(), hp.v.data_ptr(), hp.g.data_ptr(),
                              hp.beta.data_ptr(), hp.state.data_ptr(), hp.out.data_ptr(), 1, 128, 1, 1, 128, 128,
                              ctypes.byref(st), None, None, 0, torch.cuda.current_stream().cuda_stream)
    assert rc == gdn.GDN_ERR_ARG
    assert "page-locked" in lib.gdn_last_error().decode()
    assert lib.gdn_last_launch_count() == 0
    assert torch.isnan(hp.out.float()).all()  # nothing was written
