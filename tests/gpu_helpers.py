"""Shared helpers for the GPU tests: move a seeded problem onto the device,
run the CUDA path through the C ABI, and compare with the fp64 oracle using
the tolerances the prefill is specified to meet."""
from __future__ import annotations

import numpy as np

import gdn_synth

# Tolerances for bf16 I/O with an fp32 state: whole-tensor relative L2 of the
# output <= 1e-2 and max |error| <= 5e-2 * rms(oracle output); final state
# relative L2 <= 1e-3. Errors are computed in fp64 from the GPU's bf16/fp32
# values without rounding the oracle.
OUT_REL_L2 = 1e-2
OUT_MAX_OVER_RMS = 5e-2
STATE_REL_L2 = 1e-3


def to_torch_bf16(bits, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


class DeviceProblem:
    """Device copies of a ``gdn_synth.Problem`` plus output/state buffers."""

    def __init__(self, p: gdn_synth.Problem, device="cuda", state_table=None, out_pad=0, qk_l2norm=None):
        import torch

        self.p = p
        self.device = device
        self.q = to_torch_bf16(p.q, device)
        self.k = to_torch_bf16(p.k, device)
        self.v = to_torch_bf16(p.v, device)
        self.g = torch.from_numpy(p.g).to(device)
        self.beta = torch.from_numpy(p.beta).to(device)
        self.cu = None if p.cu_seqlens is None else torch.from_numpy(p.cu_seqlens).to(device)
        self.table = p.meta.get("state_table", False) if state_table is None else state_table
        self.qk_l2norm = p.meta.get("qk_raw", False) if qk_l2norm is None else qk_l2norm
        self.out = torch.empty((p.rows, p.nv * p.dv + out_pad), dtype=torch.bfloat16, device=device)
        self.reset()

    def reset(self):
        import torch

        p = self.p
        self.out.fill_(float("nan"))
        if self.table:
            self.states = [torch.from_numpy(p.h0[s].copy()).to(self.device) for s in range(p.B)]
            self.state = torch.tensor([t.data_ptr() for t in self.states], dtype=torch.int64, device=self.device)
        else:
            self.states = None
            self.state = torch.from_numpy(p.h0.copy()).to(self.device)

    def run(self, workspace=None, stream=None):
        import gated_delta_rule_17_gb300 as gdn

        p = self.p
        gdn.prefill(self.q, self.k, self.v, self.g, self.beta, self.state, self.out, nk=p.nk, nv=p.nv,
                    B=p.B, T=p.T, cu_seqlens=self.cu, state_is_table=self.table, workspace=workspace,
                    stream=stream, qk_l2norm=self.qk_l2norm)

    def out_np(self):
        import torch

        o = self.out[:, : self.p.nv * self.p.dv].float().cpu().numpy().astype(np.float64)
        return o.reshape(self.p.rows, self.p.nv, self.p.dv)

    def state_np(self):
        import torch

        if self.table:
            return np.stack([t.cpu().numpy() for t in self.states]).astype(np.float64)
        return self.state.cpu().numpy().astype(np.float64)


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
