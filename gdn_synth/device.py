"""Device copies of a seeded ``gdn_synth.Problem`` and the one call that runs the
CUDA path on them (through the binding of the C ABI). Shared by the GPU tests and
the bench; it holds none of the method's arithmetic and is never imported by the
oracle side (``gdn_synth`` itself does not import it)."""
from __future__ import annotations

import numpy as np


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
