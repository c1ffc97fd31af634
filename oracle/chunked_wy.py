"""CPU ORACLE (test infrastructure): chunked WY evaluation in numpy fp64.

Only tests, the smoke check and the benchmark's CPU-baseline leg may use this
module. It is a second, independent evaluation of the gated delta rule: where
``gdn_token_loop.c`` walks tokens one by one, this walks chunks of C tokens
with the three stages of the GDN prefill op (ssm_gdn_a3.rs, doc comment of
`gdn_prefill_fla`), written from their algebra:

1. WY stage, per chunk (tokens i, j in the chunk, gc the inclusive in-chunk
   cumulative sum of the log-gate):
       L_ij = beta_i exp(gc_i - gc_j) (k_i . k_j)   for j < i, else 0
       solve (I + L) U = diag(beta) V
       solve (I + L) W = diag(beta exp(gc)) K
2. State spine, chunks in order, S_c the state entering the chunk:
       u_c = U - W S_c
       S  <- exp(gc_last) S_c + (diag(exp(gc_last - gc)) K)^T u_c
3. Output, per chunk:
       O = [diag(exp(gc)) Q S_c + (tril_incl(exp(gc_i - gc_j)) * (Q K^T)) u_c] / sqrt(dk)

The stage formulas follow from the token recurrence: u_c stacks the delta-rule
corrections of the chunk's tokens, and the output of token i is its read-out
of the state after its own update. With C = 1 the stages reduce to the
recurrence itself. The triangular solve uses numpy's dense solver (a library
primitive); exponentials of gate differences are only taken for j <= i.
"""
from __future__ import annotations

import numpy as np

from gdn_synth import bf16_bits_to_f32


def _as_f64(a):
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def chunked_head(q, k, v, g, beta, S0, C):
    """Chunked evaluation for one (sequence, v-head).

    q, k: [n, dk]; v: [n, dv]; g, beta: [n]; S0: [dk, dv]; all fp64.
    Returns (out [n, dv], S_T [dk, dv], stages) where ``stages`` is a list of
    per-chunk dicts with gc, W, U, S_c and u_c.
    """
    n, dk = k.shape
    S = S0.copy()
    out = np.zeros((n, v.shape[1]))
    stages = []
    scale = 1.0 / np.sqrt(dk)
    for c0 in range(0, n, C):
        c1 = min(c0 + C, n)
        Kc, Vc, Qc = k[c0:c1], v[c0:c1], q[c0:c1]
        bc = beta[c0:c1]
        gc = np.cumsum(g[c0:c1])
        m = c1 - c0
        ii, jj = np.meshgrid(np.arange(m), np.arange(m), indexing="ij")
        lower = jj < ii
        incl = jj <= ii
        diff = np.where(incl, gc[:, None] - gc[None, :], -np.inf)
        decay = np.exp(diff)  # zero above the diagonal
        L = np.where(lower, bc[:, None] * decay * (Kc @ Kc.T), 0.0)
        IL = np.eye(m) + L
        U = np.linalg.solve(IL, bc[:, None] * Vc)
        W = np.linalg.solve(IL, (bc * np.exp(gc))[:, None] * Kc)
        Sc = S
        u = U - W @ Sc
        A = np.where(incl, decay * (Qc @ Kc.T), 0.0)
        out[c0:c1] = (np.exp(gc)[:, None] * (Qc @ Sc) + A @ u) * scale
        glast = gc[-1]
        S = np.exp(glast) * Sc + (np.exp(glast - gc)[:, None] * Kc).T @ u
        stages.append(dict(gc=gc, W=W, U=U, S_c=Sc, u_c=u))
    return out, S, stages


def chunked_prefill(p, C=64, heads=None, keep_stages=False):
    """Chunked evaluation of a whole ``gdn_synth.Problem``.

    Returns (out [rows, nv, dv], hT [B, nv, dk, dv], stages) with stages keyed
    by (sequence, head) when ``keep_stages``.
    """
    nk, nv, dk, dv = p.nk, p.nv, p.dk, p.dv
    group = nv // nk
    heads = range(nv) if heads is None else heads
    out = np.zeros((p.rows, nv, dv))
    hT = np.zeros((p.B, nv, dk, dv))
    stages = {}
    for s, (r0, n) in enumerate(p.seq_bounds()):
        rows = slice(r0, r0 + n)
        for h in heads:
            kh = h // group
            q = _as_f64(p.q[rows, kh * dk:(kh + 1) * dk])
            k = _as_f64(p.k[rows, kh * dk:(kh + 1) * dk])
            v = _as_f64(p.v[rows, h * dv:(h + 1) * dv])
            g = p.g[rows, h].astype(np.float64)
            b = p.beta[rows, h].astype(np.float64)
            o, S, st = chunked_head(q, k, v, g, b, p.h0[s, h].astype(np.float64), C)
            out[rows, h] = o
            hT[s, h] = S
            if keep_stages:
                stages[(s, h)] = st
    return out, hT, stages
