"""GB300-native chunked gated-delta-rule (GDN) prefill forward.

A thin ctypes binding over the C ABI in ``include/gdn_prefill.h``; every step
of the computation runs in the library's CUDA kernels. PyTorch only supplies
device memory and the current stream. There is no fallback: if the compiled
library is missing, importing works but every call raises ``GdnError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["prefill", "prefill_noalloc", "prefill_host", "host_scratch_bytes", "NOALLOC_MAX_SEQS", "workspace_bytes", "check", "last_launch_count",
           "backward", "backward_workspace_bytes",
           "set_timing_events", "set_test_hooks", "decode", "lib_path", "load", "GdnError",
           "Strides", "GDN_OK", "GDN_ERR_ARG", "GDN_ERR_UNSUPPORTED", "GDN_ERR_CUDA",
           "GDN_ERR_DEVICE_STATUS", "GDN_ERR_TIMEOUT", "GDN_ERR_RANGE"]

(GDN_OK, GDN_ERR_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_DEVICE_STATUS, GDN_ERR_TIMEOUT,
 GDN_ERR_RANGE) = range(7)
NOALLOC_MAX_SEQS = 16384  # GDN_NOALLOC_MAX_SEQS in include/gdn_prefill.h

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libgdn_gb300.so")
_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"gdn error {code}: {message}")
        self.code = code


class Strides(ctypes.Structure):
    _fields_ = [("q", ctypes.c_int64), ("k", ctypes.c_int64), ("v", ctypes.c_int64),
                ("g", ctypes.c_int64), ("beta", ctypes.c_int64), ("out", ctypes.c_int64),
                ("state_is_table", ctypes.c_int32), ("qk_l2norm", ctypes.c_int32)]


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load the compiled library (raises GdnError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise GdnError(GDN_ERR_UNSUPPORTED, f"CUDA library not built: {_LIB_PATH} is missing "
                                                    "(run __graft_entry__.build())")
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
            common = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.POINTER(Strides), vp]
            lib.gdn_prefill.argtypes = common + [vp]
            lib.gdn_prefill.restype = i
            lib.gdn_prefill_ex.argtypes = common + [vp, sz, vp]
            lib.gdn_prefill_ex.restype = i
            lib.gdn_prefill_workspace_bytes.argtypes = [i, i, i, i, i, i]
            lib.gdn_prefill_workspace_bytes.restype = sz
            lib.gdn_prefill_check.argtypes = [vp]
            lib.gdn_prefill_check.restype = i
            lib.gdn_last_error.argtypes = []
            lib.gdn_last_error.restype = ctypes.c_char_p
            lib.gdn_last_launch_count.argtypes = []
            lib.gdn_last_launch_count.restype = i
            lib.gdn_prefill_noalloc.argtypes = common + [vp]
            lib.gdn_prefill_noalloc.restype = i
            lib.gdn_prefill_host.argtypes = common + [vp, sz, vp]
            lib.gdn_prefill_host.restype = i
            lib.gdn_prefill_host_scratch_bytes.argtypes = [i, i, i, i, i, i, i]
            lib.gdn_prefill_host_scratch_bytes.restype = sz
            lib.gdn_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.POINTER(Strides), vp]
            lib.gdn_decode.restype = i
            lib.gdn_prefill_backward_workspace_bytes.argtypes = [i, i, i, i, i, i]
            lib.gdn_prefill_backward_workspace_bytes.restype = sz
            lib.gdn_prefill_backward.argtypes = [vp] * 14 + [i] * 6 + [ctypes.POINTER(Strides), vp, vp, sz, vp]
            lib.gdn_prefill_backward.restype = i
            lib.gdn_set_timing_events.argtypes = [vp, vp, vp]
            lib.gdn_set_timing_events.restype = None
            lib.gdn_set_test_hooks.argtypes = [i64, i64, i]
            lib.gdn_set_test_hooks.restype = i
            _lib = lib
    return _lib


def _raise(code):
    msg = load().gdn_last_error().decode(errors="replace")
    raise GdnError(code, msg)


def _row_stride(t, name, inner):
    """Row stride (elements) of a [rows, ...] tensor whose per-row part is contiguous."""
    if t.dim() < 2:
        raise GdnError(GDN_ERR_ARG, f"{name} must be at least 2-D ([rows, ...])")
    per_row = 1
    for d in t.shape[1:]:
        per_row *= d
    expect = 1
    for d in range(t.dim() - 1, 0, -1):
        if t.shape[d] != 1 and t.stride(d) != expect:
            raise GdnError(GDN_ERR_ARG, f"{name}: the part of each row must be contiguous")
        expect *= t.shape[d]
    if per_row < inner:
        raise GdnError(GDN_ERR_ARG, f"{name}: rows hold {per_row} elements, need {inner}")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), per_row)


def workspace_bytes(B, T, nv, varlen, dk=128, dv=128) -> int:
    return int(load().gdn_prefill_workspace_bytes(B, T, nv, dk, dv, 1 if varlen else 0))


# The library takes raw device addresses, so a host tensor or a wrong element type
# handed to it would reach a kernel; these checks turn that into a GdnError first.
def _check_rows(torch, named):
    for name, t, dt in named:
        if t.dtype != dt:
            raise GdnError(GDN_ERR_ARG, f"{name} must be {dt}, got {t.dtype}")
        if not t.is_cuda:
            raise GdnError(GDN_ERR_ARG, f"{name} must be a CUDA tensor")


def _check_state(torch, state, state_is_table, name="state"):
    if not state.is_cuda:
        raise GdnError(GDN_ERR_ARG, f"{name} must be a CUDA tensor")
    if state_is_table:
        if state.dtype != torch.int64 or not state.is_contiguous():
            raise GdnError(GDN_ERR_ARG, f"a {name} table must be a contiguous int64 tensor of device addresses")
    elif state.dtype != torch.float32 or not state.is_contiguous():
        raise GdnError(GDN_ERR_ARG, f"{name} must be a contiguous fp32 tensor [B, nv, dk, dv]")


def _check_aux(torch, cu_seqlens, workspace):
    if cu_seqlens is not None and (cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda
                                   or not cu_seqlens.is_contiguous()):
        raise GdnError(GDN_ERR_ARG, "cu_seqlens must be a contiguous int32 CUDA tensor")
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise GdnError(GDN_ERR_ARG, "workspace must be a contiguous CUDA tensor")


def _io_rows(torch, q, k, v, g, beta, last):
    return (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
            ("g", g, torch.float32), ("beta", beta, torch.float32), last)


def prefill(q, k, v, g, beta, state, out, *, nk: int, nv: int, B: int | None = None, T: int | None = None,
            cu_seqlens=None, state_is_table: bool = False, workspace=None, stream=None, dk: int = 128,
            dv: int = 128, qk_l2norm: bool = False) -> None:
    """Enqueue one GDN prefill on ``stream`` (default: torch's current stream).

    q, k: bf16 CUDA tensors [rows, nk*dk] (or [rows, nk, dk]); v: bf16 [rows, nv*dv];
    g, beta: fp32 [rows, nv]; out: bf16 [rows, nv*dv]. ``state``: fp32 CUDA tensor
    [B, nv, dk, dv] updated in place, or (``state_is_table``) an int64 CUDA tensor of
    B device addresses of [nv, dk, dv] fp32 states. Dense batches give ``B`` and ``T``
    (rows = B*T); varlen batches give ``cu_seqlens`` (int32 CUDA [B+1]).
    ``workspace`` (uint8 CUDA tensor) passes caller-provided scratch (``gdn_prefill_ex``).
    ``qk_l2norm`` normalises every q and k head row inside the kernels (fused prologue).
    """
    import torch

    lib = load()
    _check_rows(torch, _io_rows(torch, q, k, v, g, beta, ("out", out, torch.bfloat16)))
    _check_state(torch, state, state_is_table)
    _check_aux(torch, cu_seqlens, workspace)
    rows = q.shape[0]
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
        T = rows
    elif B is None or T is None:
        raise GdnError(GDN_ERR_ARG, "dense batches need B and T")
    st = Strides(_row_stride(q, "q", nk * dk), _row_stride(k, "k", nk * dk), _row_stride(v, "v", nv * dv),
                 _row_stride(g, "g", nv), _row_stride(beta, "beta", nv), _row_stride(out, "out", nv * dv),
                 1 if state_is_table else 0, 1 if qk_l2norm else 0)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(), state.data_ptr(),
            out.data_ptr(), B, T, nk, nv, dk, dv, ctypes.byref(st),
            None if cu_seqlens is None else cu_seqlens.data_ptr()]
    if workspace is None:
        rc = lib.gdn_prefill(*args, stream)
    else:
        rc = lib.gdn_prefill_ex(*args, workspace.data_ptr() if workspace.numel() else None,
                                workspace.numel() * workspace.element_size(), stream)
    if rc != GDN_OK:
        _raise(rc)


def prefill_noalloc(q, k, v, g, beta, state, out, *, nk: int, nv: int, B: int | None = None,
                    T: int | None = None, cu_seqlens=None, state_is_table: bool = False, stream=None,
                    dk: int = 128, dv: int = 128, qk_l2norm: bool = False) -> None:
    """``prefill`` through ``gdn_prefill_noalloc``: the library allocates no device
    memory during the call (its varlen schedule lives in a static device array of
    ``NOALLOC_MAX_SEQS`` entries). For callers that cannot allocate mid-call.
    Calls that overlap on the GPU race on that shared array."""
    import torch

    lib = load()
    _check_rows(torch, _io_rows(torch, q, k, v, g, beta, ("out", out, torch.bfloat16)))
    _check_state(torch, state, state_is_table)
    _check_aux(torch, cu_seqlens, None)
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
        T = q.shape[0]
    elif B is None or T is None:
        raise GdnError(GDN_ERR_ARG, "dense batches need B and T")
    st = Strides(_row_stride(q, "q", nk * dk), _row_stride(k, "k", nk * dk), _row_stride(v, "v", nv * dv),
                 _row_stride(g, "g", nv), _row_stride(beta, "beta", nv), _row_stride(out, "out", nv * dv),
                 1 if state_is_table else 0, 1 if qk_l2norm else 0)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = lib.gdn_prefill_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(),
                                 state.data_ptr(), out.data_ptr(), B, T, nk, nv, dk, dv, ctypes.byref(st),
                                 None if cu_seqlens is None else cu_seqlens.data_ptr(), stream)
    if rc != GDN_OK:
        _raise(rc)


def host_scratch_bytes(B, T, nk, nv, varlen, dk=128, dv=128) -> int:
    """Device scratch of ``prefill_host`` (``gdn_prefill_host_scratch_bytes``)."""
    return int(load().gdn_prefill_host_scratch_bytes(B, T, nk, nv, dk, dv, 1 if varlen else 0))


def prefill_host(q, k, v, g, beta, state, out, *, nk: int, nv: int, B: int | None = None, T: int | None = None,
                 cu_seqlens=None, scratch=None, stream=None, dk: int = 128, dv: int = 128,
                 qk_l2norm: bool = False) -> None:
    """``gdn_prefill_host``: the prefill over page-locked host tensors (``pin_memory()``),
    packed as for ``prefill`` (q, k [rows, nk*dk] bf16; v, out [rows, nv*dv] bf16; g, beta
    [rows, nv] fp32; state [B, nv, dk, dv] fp32, updated in place; cu_seqlens int32 [B+1]).
    Enqueued on ``stream`` (default: torch's current CUDA stream); the host tensors must
    stay untouched until that stream passes the call. ``scratch``: optional uint8 CUDA
    tensor of ``host_scratch_bytes(...)`` bytes (else allocated stream-ordered)."""
    import torch

    lib = load()
    named = [("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16), ("g", g, torch.float32),
             ("beta", beta, torch.float32), ("state", state, torch.float32), ("out", out, torch.bfloat16)]
    if cu_seqlens is not None:
        named.append(("cu_seqlens", cu_seqlens, torch.int32))
    for name, t, dt in named:
        if t.device.type != "cpu" or not t.is_pinned():
            raise GdnError(GDN_ERR_ARG, f"{name} must be a page-locked CPU tensor (pin_memory())")
        if t.dtype != dt or not t.is_contiguous():
            raise GdnError(GDN_ERR_ARG, f"{name} must be a contiguous {dt} tensor")
    if scratch is not None and (not scratch.is_cuda or scratch.dtype != torch.uint8):
        raise GdnError(GDN_ERR_ARG, "scratch must be a uint8 CUDA tensor")
    rows = q.shape[0]
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
        T = rows
    elif B is None or T is None:
        raise GdnError(GDN_ERR_ARG, "dense batches need B and T")
    st = Strides(nk * dk, nk * dk, nv * dv, nv, nv, nv * dv, 0, 1 if qk_l2norm else 0)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = lib.gdn_prefill_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(),
                              state.data_ptr(), out.data_ptr(), B, T, nk, nv, dk, dv, ctypes.byref(st),
                              None if cu_seqlens is None else cu_seqlens.data_ptr(),
                              None if scratch is None or not scratch.numel() else scratch.data_ptr(),
                              0 if scratch is None else scratch.numel(), stream)
    if rc != GDN_OK:
        _raise(rc)


def decode(q, k, v, g, beta, state, out, *, nk: int, nv: int, state_is_table: bool = False, stream=None,
           dk: int = 128, dv: int = 128, qk_l2norm: bool = False) -> None:
    """Enqueue one single-token decode step for every row (sequence) b of q/k/v/g/beta/out:
    the state of sequence b (``state[b]``, or the b-th pointer of a table) is advanced by
    that token and the token's output written to ``out[b]``. Same layouts as ``prefill``."""
    import torch

    lib = load()
    _check_rows(torch, _io_rows(torch, q, k, v, g, beta, ("out", out, torch.bfloat16)))
    _check_state(torch, state, state_is_table)
    st = Strides(_row_stride(q, "q", nk * dk), _row_stride(k, "k", nk * dk), _row_stride(v, "v", nv * dv),
                 _row_stride(g, "g", nv), _row_stride(beta, "beta", nv), _row_stride(out, "out", nv * dv),
                 1 if state_is_table else 0, 1 if qk_l2norm else 0)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = lib.gdn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(), state.data_ptr(),
                        out.data_ptr(), q.shape[0], nk, nv, dk, dv, ctypes.byref(st), stream)
    if rc != GDN_OK:
        _raise(rc)


def backward_workspace_bytes(B, T, nv, varlen, dk=128, dv=128) -> int:
    return int(load().gdn_prefill_backward_workspace_bytes(B, T, nv, dk, dv, 1 if varlen else 0))


def backward(q, k, v, g, beta, h0, dout, dq, dk, dv, dg, dbeta, *, nk: int, nv: int, dST=None, dh0=None,
             B: int | None = None, T: int | None = None, cu_seqlens=None, state_is_table: bool = False,
             workspace=None, stream=None, dk_dim: int = 128, dv_dim: int = 128) -> None:
    """Enqueue the backward of ``prefill`` (``gdn_prefill_backward``): the chunked form
    on the tensor cores, 4 launches (5 with ``cu_seqlens``).

    q, k, v, g, beta, cu_seqlens, state_is_table: as ``prefill``; ``h0`` is the initial
    state the forward started from. ``dout`` fp32 [rows, nv*dv] (dL/do), ``dST`` fp32
    [B, nv, dk, dv] or None. Outputs (fp32): dq, dk [rows, nk*dk], dv [rows, nv*dv],
    dg, dbeta [rows, nv], dh0 [B, nv, dk, dv] or None.
    """
    import torch

    lib = load()
    _check_rows(torch, _io_rows(torch, q, k, v, g, beta, ("dout", dout, torch.float32)))
    _check_state(torch, h0, state_is_table, name="h0")
    _check_aux(torch, cu_seqlens, workspace)
    for name, t in (("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv), ("dg", dg), ("dbeta", dbeta),
                    ("dST", dST), ("dh0", dh0)):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda):
            raise GdnError(GDN_ERR_ARG, f"{name} must be a contiguous fp32 CUDA tensor")
    rows = q.shape[0]
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
        T = rows
    elif B is None or T is None:
        raise GdnError(GDN_ERR_ARG, "dense batches need B and T")
    st = Strides(_row_stride(q, "q", nk * dk_dim), _row_stride(k, "k", nk * dk_dim), _row_stride(v, "v", nv * dv_dim),
                 _row_stride(g, "g", nv), _row_stride(beta, "beta", nv), nv * dv_dim,
                 1 if state_is_table else 0, 0)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream

    def ptr(t):
        return None if t is None else t.data_ptr()

    ws_ptr, ws_size = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    rc = lib.gdn_prefill_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(), h0.data_ptr(),
                                  dout.data_ptr(), ptr(dST), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dg.data_ptr(),
                                  dbeta.data_ptr(), ptr(dh0), B, T, nk, nv, dk_dim, dv_dim, ctypes.byref(st),
                                  ptr(cu_seqlens), ws_ptr, ws_size, stream)
    if rc != GDN_OK:
        _raise(rc)


def check(stream=None) -> None:
    """Synchronise the stream and raise if a kernel reported a device-side error."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = load().gdn_prefill_check(stream)
    if rc != GDN_OK:
        _raise(rc)


def last_launch_count() -> int:
    return int(load().gdn_last_launch_count())


def set_timing_events(before_wy=None, before_spine=None, after_spine=None) -> None:
    """Have later calls on this thread record these torch.cuda.Events (or None) before
    the WY-solve kernel, between the kernels and after the spine kernel. torch creates
    an event's CUDA handle on its first record, so record each once beforehand."""
    def handle(e):
        return None if e is None else e.cuda_event
    load().gdn_set_timing_events(handle(before_wy), handle(before_spine), handle(after_spine))


def set_test_hooks(wait_limit_ns: int = 0, consumer_delay_ns: int = 0, skip_hand_off_chunk: int = -1) -> None:
    """Test hooks (``gdn_set_test_hooks``) for later prefill calls on this thread: a
    short wait limit, a consumer delay before the hand-off wait of odd chunks, and a
    skipped hand-off arrival. All defaults switch them off."""
    rc = load().gdn_set_test_hooks(int(wait_limit_ns), int(consumer_delay_ns), int(skip_hand_off_chunk))
    if rc != GDN_OK:
        _raise(rc)
