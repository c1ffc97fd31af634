"""The allocation-free entry point, gdn_prefill_noalloc, called through the C ABI.

It is meant for callers that cannot allocate device memory in the middle of a
call (a serving process whose memory is reserved up front by its own
allocator, or a latency-bound loop where cudaMalloc could block or fail).
Its results must match gdn_prefill's on the same inputs, call after call,
even though every call reuses one static scratch array. This file is
collected last so that a failure here never hides another test's result.
"""
import ctypes

import numpy as np
import pytest

import gdn_synth
from tests.gpu_helpers import DeviceProblem, compare, OUT_REL_L2, OUT_MAX_OVER_RMS, STATE_REL_L2

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_17_gb300 import build

    build.build()
    import gated_delta_rule_17_gb300 as gdn

    return gdn.load()


def _call(lib, fn, dp):
    p = dp.p
    import gated_delta_rule_17_gb300 as gdn

    st = gdn.Strides(dp.q.stride(0), dp.k.stride(0), dp.v.stride(0), dp.g.stride(0), dp.beta.stride(0),
                     dp.out.stride(0), 1 if dp.table else 0)
    stream = torch.cuda.current_stream().cuda_stream
    rc = getattr(lib, fn)(dp.q.data_ptr(), dp.k.data_ptr(), dp.v.data_ptr(), dp.g.data_ptr(), dp.beta.data_ptr(),
                          dp.state.data_ptr(), dp.out.data_ptr(), p.B, p.T, p.nk, p.nv, 128, 128,
                          ctypes.byref(st), None if dp.cu is None else dp.cu.data_ptr(), stream)
    assert rc == 0, lib.gdn_last_error().decode()
    torch.cuda.synchronize()
    assert lib.gdn_prefill_check(stream) == 0, lib.gdn_last_error().decode()
    return dp.out_np(), dp.state_np()


def _check_close(a, b):
    out_rel, out_max, st_rel = compare(a[0], a[1], b[0], b[1])
    assert out_rel <= OUT_REL_L2 and out_max <= OUT_MAX_OVER_RMS and st_rel <= STATE_REL_L2, (out_rel, out_max, st_rel)


@pytest.mark.parametrize("problems", ["varlen", "dense+varlen"])
def test_noalloc_matches_gdn_prefill_on_consecutive_calls(lib, problems):
    # two calls in a row that reuse the shared schedule array with different batch shapes
    first = gdn_synth.make_problem(seed=4100, B=5, lengths=[300, 1, 0, 129, 64], nk=2, nv=4, h0_std=0.02)
    if problems == "dense+varlen":
        first = gdn_synth.make_problem(seed=4101, B=2, T=200, nk=1, nv=2, h0_std=0.02)
    second = gdn_synth.make_problem(seed=4102, B=3, lengths=[70, 500, 33], nk=1, nv=2, h0_std=0.02)
    for p in (first, second):
        ref = DeviceProblem(p)
        want = _call(lib, "gdn_prefill", ref)
        got_dp = DeviceProblem(p)
        got = _call(lib, "gdn_prefill_noalloc", got_dp)
        _check_close(got, want)
        assert lib.gdn_last_launch_count() == (3 if p.varlen else 2)


def test_noalloc_rejects_too_many_sequences(lib):
    import gated_delta_rule_17_gb300 as gdn

    n = gdn.NOALLOC_MAX_SEQS + 1
    p16 = ctypes.c_void_p(256)
    rc = lib.gdn_prefill_noalloc(p16, p16, p16, p16, p16, p16, p16, n, 4 * n, 1, 1, 128, 128, None, p16, None)
    assert rc == gdn.GDN_ERR_UNSUPPORTED
    assert "at most" in lib.gdn_last_error().decode()
