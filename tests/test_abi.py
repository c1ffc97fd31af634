"""C ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every function the header declares; host-side validation rejects bad
arguments with named reasons before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn_prefill.h")


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_17_gb300 import build

    build.build()
    import gated_delta_rule_17_gb300 as gdn

    return gdn.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(gdn_[a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gdn_prefill", "gdn_prefill_ex", "gdn_prefill_workspace_bytes", "gdn_prefill_check",
              "gdn_last_error", "gdn_last_launch_count", "gdn_prefill_noalloc", "gdn_set_timing_events",
              "gdn_decode", "gdn_prefill_backward", "gdn_prefill_backward_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_no_cpu_fallback_symbols(lib):
    # the library is CUDA-only: its product path links nothing from oracle/
    data = open(lib._name, "rb").read()
    assert b"gdn_oracle_run" not in data and b"gdn_oracle_backward" not in data


def _call(lib, B=1, T=64, nk=1, nv=1, dk=128, dv=128, strides=None, ptr=16, cu=None):
    import gated_delta_rule_17_gb300 as gdn

    p = ctypes.c_void_p(ptr) if ptr else None
    st = ctypes.byref(strides) if strides is not None else None
    rc = lib.gdn_prefill(p, p, p, p, p, p, p, B, T, nk, nv, dk, dv, st, cu, None)
    return rc, lib.gdn_last_error().decode()


def test_rejects_head_dims(lib):
    import gated_delta_rule_17_gb300 as gdn

    rc, msg = _call(lib, dk=64)
    assert rc == gdn.GDN_ERR_UNSUPPORTED and "128" in msg


def test_rejects_gqa_mismatch(lib):
    import gated_delta_rule_17_gb300 as gdn

    rc, msg = _call(lib, nk=3, nv=4)
    assert rc == gdn.GDN_ERR_UNSUPPORTED and "multiple of nk" in msg


def test_rejects_negative_sizes(lib):
    import gated_delta_rule_17_gb300 as gdn

    assert _call(lib, B=-1)[0] == gdn.GDN_ERR_ARG
    assert _call(lib, T=-5)[0] == gdn.GDN_ERR_ARG
    assert _call(lib, nk=0)[0] == gdn.GDN_ERR_ARG


def test_rejects_null_and_misaligned_pointers(lib):
    import gated_delta_rule_17_gb300 as gdn

    rc, msg = _call(lib, ptr=0)
    assert rc == gdn.GDN_ERR_ARG and "NULL" in msg
    rc, msg = _call(lib, ptr=18)
    assert rc == gdn.GDN_ERR_ARG and "aligned" in msg


def test_rejects_bad_strides(lib):
    import gated_delta_rule_17_gb300 as gdn

    st = gdn.Strides(132, 128, 128, 1, 1, 128, 0)  # q stride not a multiple of 8
    rc, msg = _call(lib, strides=st)
    assert rc == gdn.GDN_ERR_ARG and "q row stride" in msg
    st = gdn.Strides(128, 128, 64, 1, 1, 128, 0)  # v stride below nv*dv
    rc, msg = _call(lib, strides=st)
    assert rc == gdn.GDN_ERR_ARG and "v row stride" in msg
    st = gdn.Strides(128, 128, 128, 0, 1, 128, 0)  # g stride below nv
    assert _call(lib, strides=st)[0] == gdn.GDN_ERR_ARG
    st = gdn.Strides(128, 128, 128, 1, 1, 128, 2)  # bad table flag
    assert _call(lib, strides=st)[0] == gdn.GDN_ERR_ARG


def test_empty_problem_is_a_no_op(lib):
    import gated_delta_rule_17_gb300 as gdn

    assert _call(lib, B=0, ptr=0)[0] == gdn.GDN_OK
    assert lib.gdn_last_launch_count() == 0
    assert _call(lib, T=0, ptr=0)[0] == gdn.GDN_OK


def test_workspace_sizes(lib):
    assert lib.gdn_prefill_workspace_bytes(4, 8192, 32, 128, 128, 0) == 0
    assert lib.gdn_prefill_workspace_bytes(8, 64000, 48, 128, 128, 1) == 256
    assert lib.gdn_prefill_workspace_bytes(100, 64000, 48, 128, 128, 1) == 1024
    # dense batches with few chains and long sequences: the segment schedule's tables
    # (4 x 256-byte-aligned regions) and 3 (G-1) per-sequence states, here G = 3 on the
    # 152 SMs assumed without a visible GPU
    assert lib.gdn_prefill_workspace_bytes(1, 65536, 32, 128, 128, 0) == 1024 + 3 * 2 * 32 * 128 * 128 * 4
    # G = 2 (B * nv = 64 chains): 3 states per sequence
    assert lib.gdn_prefill_workspace_bytes(2, 65536, 32, 128, 128, 0) == 1024 + 3 * 2 * 32 * 128 * 128 * 4
    # too many chains, or too few chunks, for 2 segments: none
    assert lib.gdn_prefill_workspace_bytes(3, 65536, 32, 128, 128, 0) == 0
    assert lib.gdn_prefill_workspace_bytes(1, 64 * 15, 4, 128, 128, 0) == 0


def test_ex_rejects_small_workspace(lib):
    import gated_delta_rule_17_gb300 as gdn

    p = ctypes.c_void_p(256)
    cu = ctypes.c_void_p(512)
    rc = lib.gdn_prefill_ex(p, p, p, p, p, p, p, 4, 100, 1, 1, 128, 128, None, cu, p, 8, None)
    assert rc == gdn.GDN_ERR_ARG and "workspace" in lib.gdn_last_error().decode()


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import gated_delta_rule_17_gb300 as gdn

    monkeypatch.setattr(gdn, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(gdn, "_lib", None)
    with pytest.raises(gdn.GdnError):
        gdn.load()


def test_backward_workspace_sizes(lib):
    # varlen schedule (2B + 1 int32), then T, u and du' (16-bit, rows x nv x 128 each)
    # and each chunk slot's S0 and dS_end (fp16 128 x 128 per head, rows / 64 + B + 1
    # slots)
    def a256(x):
        return (x + 255) // 256 * 256

    for B, T, nv, varlen in ((1, 4096, 32, 0), (3, 1000, 8, 1)):
        rows = T if varlen else B * T
        row16 = rows * nv * 128 * 2
        state16 = (rows // 64 + B + 1) * nv * 128 * 128 * 2
        off = a256((2 * B + 1) * 4 if varlen else 0)
        off = a256(off + row16)
        off = a256(off + row16)
        off = a256(off + row16)
        off = a256(off + state16)
        off = a256(off + state16)
        assert lib.gdn_prefill_backward_workspace_bytes(B, T, nv, 128, 128, varlen) == off
    assert lib.gdn_prefill_backward_workspace_bytes(0, T, nv, 128, 128, 0) == 0


def _bwd(lib, B=1, T=64, nk=1, nv=1, dk=128, dv=128, strides=None, ptr=16, grad=16):
    p = ctypes.c_void_p(ptr) if ptr else None
    gp = ctypes.c_void_p(grad) if grad else None
    st = ctypes.byref(strides) if strides is not None else None
    rc = lib.gdn_prefill_backward(p, p, p, p, p, p, p, None, gp, gp, gp, gp, gp, None, B, T, nk, nv, dk, dv, st,
                                  None, None, 0, None)
    return rc, lib.gdn_last_error().decode()


def test_backward_host_checks(lib):
    # every rejection below happens before the device is touched
    import gated_delta_rule_17_gb300 as gdn

    rc, msg = _bwd(lib, strides=gdn.Strides(128, 128, 128, 1, 1, 128, 0, 1))
    assert rc == gdn.GDN_ERR_UNSUPPORTED and "normalised" in msg
    rc, msg = _bwd(lib, grad=0)
    assert rc == gdn.GDN_ERR_ARG and "gradient output pointer is NULL" in msg
    rc, msg = _bwd(lib, grad=24)
    assert rc == gdn.GDN_ERR_ARG and "16-byte aligned" in msg
    rc, msg = _bwd(lib, dk=64)
    assert rc == gdn.GDN_ERR_UNSUPPORTED and "128" in msg
    rc, msg = _bwd(lib, nk=3, nv=4)
    assert rc == gdn.GDN_ERR_UNSUPPORTED and "multiple of nk" in msg
    assert _bwd(lib, B=-1)[0] == gdn.GDN_ERR_ARG
    assert _bwd(lib, B=0, ptr=0, grad=0)[0] == gdn.GDN_OK
    assert lib.gdn_last_launch_count() == 0


def _dec(lib, B=1, nk=1, nv=1, dk=128, dv=128, strides=None, ptr=16):
    p = ctypes.c_void_p(ptr) if ptr else None
    st = ctypes.byref(strides) if strides is not None else None
    rc = lib.gdn_decode(p, p, p, p, p, p, p, B, nk, nv, dk, dv, st, None)
    return rc, lib.gdn_last_error().decode()


def test_decode_host_checks(lib):
    # the decode step shares the prefill's argument rules; each rejection happens on the host
    import gated_delta_rule_17_gb300 as gdn

    rc, msg = _dec(lib, dv=64)
    assert rc == gdn.GDN_ERR_UNSUPPORTED and "128" in msg
    rc, msg = _dec(lib, nk=2, nv=3)
    assert rc == gdn.GDN_ERR_UNSUPPORTED and "multiple of nk" in msg
    assert _dec(lib, B=-2)[0] == gdn.GDN_ERR_ARG
    rc, msg = _dec(lib, ptr=0)
    assert rc == gdn.GDN_ERR_ARG and "NULL" in msg
    rc, msg = _dec(lib, ptr=18)
    assert rc == gdn.GDN_ERR_ARG and "aligned" in msg
    rc, msg = _dec(lib, strides=gdn.Strides(132, 128, 128, 1, 1, 128, 0))
    assert rc == gdn.GDN_ERR_ARG and "q row stride" in msg
    assert _dec(lib, B=0, ptr=0)[0] == gdn.GDN_OK
    assert lib.gdn_last_launch_count() == 0


def test_binding_rejects_host_tensors_and_wrong_types(lib):
    # every entry point of the binding checks element types and device placement before
    # the library sees an address (a host pointer would otherwise reach a kernel)
    import torch

    import gated_delta_rule_17_gb300 as gdn

    rows, nk, nv = 64, 1, 1
    bf = dict(dtype=torch.bfloat16)
    f32 = dict(dtype=torch.float32)
    q, k, v, out = (torch.zeros((rows, 128), **bf) for _ in range(4))
    g, beta = torch.zeros((rows, nv), **f32), torch.zeros((rows, nv), **f32)
    state = torch.zeros((1, nv, 128, 128), **f32)
    calls = {
        "prefill": lambda **kw: gdn.prefill(q, k, v, g, beta, state, out, nk=nk, nv=nv, B=1, T=rows, **kw),
        "prefill_noalloc": lambda **kw: gdn.prefill_noalloc(q, k, v, g, beta, state, out, nk=nk, nv=nv, B=1,
                                                            T=rows, **kw),
        "decode": lambda **kw: gdn.decode(q, k, v, g, beta, state, out, nk=nk, nv=nv, **kw),
        "backward": lambda **kw: gdn.backward(q, k, v, g, beta, state, torch.zeros((rows, 128), **f32),
                                              *(torch.zeros((rows, 128), **f32) for _ in range(3)),
                                              torch.zeros((rows, nv), **f32), torch.zeros((rows, nv), **f32),
                                              nk=nk, nv=nv, B=1, T=rows, **kw),
    }
    for name, call in calls.items():
        with pytest.raises(gdn.GdnError, match="CUDA tensor"):
            call()
    with pytest.raises(gdn.GdnError, match="must be torch.bfloat16"):
        gdn.prefill(q.float(), k, v, g, beta, state, out, nk=nk, nv=nv, B=1, T=rows)
    with pytest.raises(gdn.GdnError, match="got torch.float16"):
        gdn.prefill_noalloc(q.half(), k, v, g, beta, state, out, nk=nk, nv=nv, B=1, T=rows)


def _call_host(lib, B=1, T=64, nk=1, nv=1, dk=128, dv=128, strides=None, ptr=16):
    p = ctypes.c_void_p(ptr) if ptr else None
    st = ctypes.byref(strides) if strides is not None else None
    rc = lib.gdn_prefill_host(p, p, p, p, p, p, p, B, T, nk, nv, dk, dv, st, None, None, 0, None)
    return rc, lib.gdn_last_error().decode()


def test_host_entry_point_rejects_before_any_device_call(lib):
    # argument checks of gdn_prefill_host that run before it touches CUDA
    import gated_delta_rule_17_gb300 as gdn

    rc, msg = _call_host(lib, dk=64)
    assert rc == gdn.GDN_ERR_UNSUPPORTED and "128" in msg
    st = gdn.Strides(128, 128, 128, 1, 1, 128, 1, 0)  # a state table
    rc, msg = _call_host(lib, strides=st)
    assert rc == gdn.GDN_ERR_UNSUPPORTED and "contiguous state" in msg
    st = gdn.Strides(256, 128, 128, 1, 1, 128, 0, 0)  # padded q rows
    rc, msg = _call_host(lib, strides=st)
    assert rc == gdn.GDN_ERR_UNSUPPORTED and "packed rows" in msg
    assert _call_host(lib, ptr=0)[0] == gdn.GDN_ERR_ARG
    assert _call_host(lib, B=0, ptr=0)[0] == gdn.GDN_OK
    assert lib.gdn_last_launch_count() == 0


def test_host_scratch_sizes(lib):
    # packed staging of q, k, v, g, beta, the state and out (each 256-byte aligned),
    # cu_seqlens for varlen batches, then the op's own workspace
    def up(x):
        return (x + 255) // 256 * 256

    B, T, nk, nv = 4, 8192, 16, 32
    rows = B * T
    qk, vo, gb, st = rows * nk * 256, rows * nv * 256, rows * nv * 4, B * nv * 128 * 128 * 4
    dense = up(qk) * 2 + up(vo) + up(gb) * 2 + up(st) + up(vo)
    assert lib.gdn_prefill_host_scratch_bytes(B, T, nk, nv, 128, 128, 0) == dense
    B, T, nk, nv = 3, 405, 2, 4
    parts = [T * nk * 256] * 2 + [T * nv * 256, T * nv * 4, T * nv * 4, B * nv * 128 * 128 * 4, T * nv * 256,
                                  (B + 1) * 4]
    want = sum(up(x) for x in parts) + lib.gdn_prefill_workspace_bytes(B, T, nv, 128, 128, 1)
    assert lib.gdn_prefill_host_scratch_bytes(B, T, nk, nv, 128, 128, 1) == want
    assert lib.gdn_prefill_host_scratch_bytes(B, T, nk, nv, 64, 128, 1) == 0
