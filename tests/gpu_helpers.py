"""Shared helpers for the GPU tests: move a seeded problem onto the device,
run the CUDA path through the C ABI, and compare with the fp64 oracle using
the tolerances the prefill is specified to meet."""
from __future__ import annotations

import numpy as np

# Tolerances for bf16 I/O with an fp32 state: whole-tensor relative L2 of the
# output <= 1e-2 and max |error| <= 5e-2 * rms(oracle output); final state
# relative L2 <= 1e-3. Errors are computed in fp64 from the GPU's bf16/fp32
# values without rounding the oracle.
OUT_REL_L2 = 1e-2
OUT_MAX_OVER_RMS = 5e-2
STATE_REL_L2 = 1e-3


from gdn_synth.device import DeviceProblem, to_torch_bf16  # noqa: F401  (re-exported for the tests)


def compare(out_gpu, st_gpu, out_ref, st_ref, heads=None, rows=None):
    """Returns (out_rel, out_max_over_rms, state_rel) over the selected heads/rows."""
    if heads is not None:
        out_gpu, out_ref = out_gpu[:, heads], out_ref[:, heads]
        st_gpu, st_ref = st_gpu[:, heads], st_ref[:, heads]
    if rows is not None:
        out_gpu, out_ref = out_gpu[rows], out_ref[rows]
    d = out_gpu - out_ref
    n_ref = np.linalg.norm(out_ref)
    rms = np.sqrt(np.mean(out_ref ** 2))
    out_rel = np.linalg.norm(d) / n_ref if n_ref > 0 else np.linalg.norm(d)
    out_max = np.abs(d).max() / rms if rms > 0 else np.abs(d).max()
    sd = st_gpu - st_ref
    s_ref = np.linalg.norm(st_ref)
    st_rel = np.linalg.norm(sd) / s_ref if s_ref > 0 else np.linalg.norm(sd)
    return float(out_rel), float(out_max), float(st_rel)


def assert_parity(out_gpu, st_gpu, out_ref, st_ref, heads=None, rows=None, label=""):
    out_rel, out_max, st_rel = compare(out_gpu, st_gpu, out_ref, st_ref, heads, rows)
    msg = f"{label}: out_rel={out_rel:.3e} out_max/rms={out_max:.3e} state_rel={st_rel:.3e}"
    assert np.isfinite(out_gpu).all() and np.isfinite(st_gpu).all(), msg + " (non-finite values)"
    assert out_rel <= OUT_REL_L2, msg
    assert out_max <= OUT_MAX_OVER_RMS, msg
    assert st_rel <= STATE_REL_L2, msg
    return out_rel, out_max, st_rel
