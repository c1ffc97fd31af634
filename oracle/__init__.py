"""CPU ORACLE -- test infrastructure for the GDN prefill, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. It shares no code with the CUDA library: the
token-by-token fp64 recurrence lives in ``gdn_token_loop.c`` (compiled here
with gcc + OpenMP), and an independent chunked-WY evaluation in numpy lives in
``chunked_wy.py``.

The backward (``token_loop_backward``) is the same recurrence differentiated
by hand, token by token in reverse, in the same C file.

Parity pins: every function here is checked by ``tests/test_oracle.py``
against closed forms (pure decay, exact overwrite with orthonormal keys,
strong decay), exact rational brute force, dense transition-matrix products
and the chunked evaluation; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from gdn_synth import Problem

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_token_loop.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libgdn_oracle.so")
_lock = threading.Lock()
_handle = None

DT_BF16, DT_F32, DT_F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc -O2 -fopenmp); returns the library path."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            lib = ctypes.CDLL(build())
            lib.gdn_oracle_run.restype = ctypes.c_int
            lib.gdn_oracle_max_threads.restype = ctypes.c_int
            lib.gdn_oracle_backward.restype = ctypes.c_int
            _handle = lib
    return _handle


def max_threads() -> int:
    return int(_lib().gdn_oracle_max_threads())


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return DT_BF16
    if a.dtype == np.float32:
        return DT_F32
    if a.dtype == np.float64:
        return DT_F64
    raise TypeError(f"unsupported oracle input dtype {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def token_loop_raw(q, k, v, g, beta, h0, *, B, T, nk, nv, dk, dv,
                   cu_seqlens=None, heads=None, threads=0):
    """Token-by-token fp64 recurrence on raw 2-D row arrays.

    q, k: [rows, >= nk*dk]; v: [rows, >= nv*dv] (bf16 bits, fp32 or fp64);
    g, beta: [rows, >= nv] (fp32 or fp64); h0: [B, nv, dk, dv] or None.
    Returns (out [rows, nv, dv] fp64, hT [B, nv, dk, dv] fp64).
    """
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    g = np.ascontiguousarray(g)
    beta = np.ascontiguousarray(beta)
    assert q.dtype == k.dtype == v.dtype and g.dtype == beta.dtype
    rows = q.shape[0]
    out = np.zeros((rows, nv, dv))
    hT = np.zeros((B, nv, dk, dv))
    h0c = None if h0 is None else np.ascontiguousarray(h0)
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    hs = None if heads is None else np.ascontiguousarray(heads, dtype=np.int32)
    rc = _lib().gdn_oracle_run(
        _ptr(q), _ptr(k), _ptr(v), ctypes.c_int(_dtype_code(q)),
        _ptr(g), _ptr(beta), ctypes.c_int(_dtype_code(g)),
        _ptr(h0c), ctypes.c_int(_dtype_code(h0c) if h0c is not None else DT_F32),
        _ptr(out), _ptr(hT),
        ctypes.c_int(B), ctypes.c_int(T), ctypes.c_int(nk), ctypes.c_int(nv),
        ctypes.c_int(dk), ctypes.c_int(dv),
        ctypes.c_int64(q.shape[1]), ctypes.c_int64(k.shape[1]), ctypes.c_int64(v.shape[1]),
        ctypes.c_int64(g.shape[1]), ctypes.c_int64(beta.shape[1]),
        _ptr(cu), _ptr(hs), ctypes.c_int(0 if hs is None else len(hs)), ctypes.c_int(threads))
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    return out, hT


def token_loop_backward(p: Problem, dout, dST=None, threads=0):
    """Backward of the token recurrence in fp64 (the training pass).

    dout: [rows, nv, dv] (dL/do); dST: [B, nv, dk, dv] (dL/dS_T) or None.
    Returns a dict with dq, dk [rows, nk, dk], dv [rows, nv, dv], dg, dbeta
    [rows, nv] and dh0 [B, nv, dk, dv], all fp64 (rows outside every sequence
    are zero).
    """
    rows = p.rows
    dout = np.ascontiguousarray(dout, dtype=np.float64).reshape(rows, p.nv, p.dv)
    dst = None if dST is None else np.ascontiguousarray(dST, dtype=np.float64)
    q = np.ascontiguousarray(p.q)
    k = np.ascontiguousarray(p.k)
    v = np.ascontiguousarray(p.v)
    g = np.ascontiguousarray(p.g)
    beta = np.ascontiguousarray(p.beta)
    assert q.dtype == k.dtype == v.dtype and g.dtype == beta.dtype
    res = {"dq": np.zeros((rows, p.nk, p.dk)), "dk": np.zeros((rows, p.nk, p.dk)),
           "dv": np.zeros((rows, p.nv, p.dv)), "dg": np.zeros((rows, p.nv)),
           "dbeta": np.zeros((rows, p.nv)), "dh0": np.zeros((p.B, p.nv, p.dk, p.dv))}
    h0 = None if p.h0 is None else np.ascontiguousarray(p.h0)
    cu = None if p.cu_seqlens is None else np.ascontiguousarray(p.cu_seqlens, dtype=np.int32)
    rc = _lib().gdn_oracle_backward(
        _ptr(q), _ptr(k), _ptr(v), ctypes.c_int(_dtype_code(q)),
        _ptr(g), _ptr(beta), ctypes.c_int(_dtype_code(g)),
        _ptr(h0), ctypes.c_int(_dtype_code(h0) if h0 is not None else DT_F32),
        _ptr(dout), _ptr(dst),
        _ptr(res["dq"]), _ptr(res["dk"]), _ptr(res["dv"]), _ptr(res["dg"]), _ptr(res["dbeta"]), _ptr(res["dh0"]),
        ctypes.c_int(p.B), ctypes.c_int(p.T), ctypes.c_int(p.nk), ctypes.c_int(p.nv),
        ctypes.c_int(p.dk), ctypes.c_int(p.dv),
        ctypes.c_int64(q.shape[1]), ctypes.c_int64(k.shape[1]), ctypes.c_int64(v.shape[1]),
        ctypes.c_int64(g.shape[1]), ctypes.c_int64(beta.shape[1]),
        _ptr(cu), ctypes.c_int(threads))
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    return res


L2_EPS = 1e-6


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64; other dtypes are cast."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def l2norm_heads(x: np.ndarray, heads: int, d: int, eps: float = L2_EPS) -> np.ndarray:
    """The fused prologue's q/k normalisation, in fp64.

    x: [rows, >= heads*d] (bf16 bits or float). Every head row x_h = x[:, h*d:(h+1)*d]
    becomes x_h / sqrt(sum(x_h^2) + eps). Returns fp64 [rows, heads*d].

    The GDN prefill op takes q and k from the packed conv layout (ssm_gdn_a3.rs,
    doc comment of `gdn_prefill_fla`: strides of the packed conv tensor); the
    normalisation of each head row is the step between that layout and the
    recurrence. The pages print no formula for it: this is the usual L2 norm
    with eps added to the sum of squares.
    """
    xf = bf16_to_f64(np.ascontiguousarray(x)[:, : heads * d]).reshape(x.shape[0], heads, d)
    n = np.sqrt(np.sum(xf * xf, axis=-1, keepdims=True) + eps)
    return (xf / n).reshape(x.shape[0], heads * d)


def token_loop(p: Problem, heads=None, threads=0, qk_l2norm=False):
    """Oracle evaluation of a ``gdn_synth.Problem`` (see ``token_loop_raw``).

    With ``qk_l2norm`` the q and k head rows first go through ``l2norm_heads``
    and the recurrence runs on fp64 q, k, v.
    """
    q, k, v = p.q, p.k, p.v
    if qk_l2norm:
        q = l2norm_heads(q, p.nk, p.dk)
        k = l2norm_heads(k, p.nk, p.dk)
        v = bf16_to_f64(v)
    return token_loop_raw(q, k, v, p.g, p.beta, p.h0, B=p.B, T=p.T, nk=p.nk, nv=p.nv,
                          dk=p.dk, dv=p.dv, cu_seqlens=p.cu_seqlens, heads=heads,
                          threads=threads)
