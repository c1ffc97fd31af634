"""The chunked backward's formulas, checked on the CPU against the fp64 oracle (no GPU).

The backward kernels evaluate the gradient of the chunked WY form (ssm_gdn_a3.rs,
`gdn_prefill_fla` doc comment: per chunk, u = T diag(beta)(V - Gamma K S0),
O = Gamma Q S0 / sqrt(dk) + (Q K^T . M) u / sqrt(dk), S_end = gamma S0 +
(gamma / Gamma) K^T u) by the chain rule: a reverse chain for dS and du', then per
chunk dQ, dK, dV, dbeta and the log-decay gradient as sums of products. This file
writes those formulas out once more in plain numpy, in the same split (forward chain,
reverse chain, per-chunk remainder), and checks every gradient against the oracle's
token-by-token backward, which is itself pinned by finite differences. A wrong term
or sign in the chunked derivation fails here whatever the GPU does.
"""
import numpy as np
import pytest

import oracle
from gdn_synth import Problem


def chunked_backward(q, k, v, g, beta, h0, dout, dst, C):
    """One (sequence, head) chain in chunks of C tokens; the tail chunk is padded with
    q = k = v = dO = 0, g = beta = 0. Returns dq, dk, dv, dg, dbeta, dh0."""
    n, dk = k.shape
    scale = 1.0 / np.sqrt(dk)
    nc = (n + C - 1) // C
    pad = nc * C - n

    def padded(a):
        return np.concatenate([a, np.zeros((pad,) + a.shape[1:])]) if pad else a

    q, k, v, g, beta, dout = (padded(a) for a in (q, k, v, g, beta, dout))

    # forward chain: every chunk's entry state S0 and u
    S = h0.copy()
    entry, us, Ts = [], [], []
    for c in range(nc):
        rows = slice(c * C, (c + 1) * C)
        K, V, bc, be = k[rows], v[rows], np.cumsum(g[rows]), beta[rows]
        Gam = np.exp(bc)
        M = np.tril(np.exp(bc[:, None] - bc[None, :]))
        L = np.tril(be[:, None] * M * (K @ K.T), -1)
        T = np.linalg.inv(np.eye(C) + L)
        u = T @ (be[:, None] * (V - Gam[:, None] * (K @ S)))
        entry.append(S.copy())
        us.append(u)
        Ts.append(T)
        S = Gam[-1] * S + (K * (Gam[-1] / Gam)[:, None]).T @ u

    # reverse chain and the per-chunk remainder
    dS = np.zeros_like(h0) if dst is None else dst.copy()
    res = {name: np.zeros_like(a) for name, a in (("dq", q), ("dk", k), ("dv", v))}
    res["dg"] = np.zeros(nc * C)
    res["dbeta"] = np.zeros(nc * C)
    for c in reversed(range(nc)):
        rows = slice(c * C, (c + 1) * C)
        Q, K, V, bc, be, dO = q[rows], k[rows], v[rows], np.cumsum(g[rows]), beta[rows], dout[rows]
        Gam = np.exp(bc)
        gam = Gam[-1]
        M = np.tril(np.exp(bc[:, None] - bc[None, :]))
        S0, u, T = entry[c], us[c], Ts[c]
        dS_end = dS
        du = (((Q @ K.T) * M * scale).T @ dO) + (K * (gam / Gam)[:, None]) @ dS_end
        dup = T.T @ du
        r = be[:, None] * dup
        dS = gam * dS_end + (Q * (Gam * scale)[:, None]).T @ dO - (K * Gam[:, None]).T @ r

        dA = np.tril(dO @ u.T) * M * scale
        F = -np.tril(dup @ u.T, -1) * M
        E = be[:, None] * F
        P = dup @ S0.T
        G = K @ K.T
        dOS = dO @ S0.T
        uD = u @ dS_end.T
        res["dv"][rows] = r
        res["dq"][rows] = (Gam * scale)[:, None] * dOS + dA @ K
        res["dk"][rows] = (E @ K + E.T @ K - (Gam * be)[:, None] * P + dA.T @ Q
                           + (gam / Gam)[:, None] * uD)
        res["dbeta"][rows] = np.sum(dup * V, 1) - Gam * np.sum(K * P, 1) + np.sum(F * G, 1)
        Z = E * G
        Y = dA * (Q @ K.T)
        w = (gam / Gam) * np.sum(K * uD, 1)
        db = (Gam * scale * np.sum(Q * dOS, 1) - Gam * be * np.sum(K * P, 1)
              + Z.sum(1) - Z.sum(0) + Y.sum(1) - Y.sum(0) - w)
        db[-1] += gam * np.sum(dS_end * S0) + w.sum()
        res["dg"][rows] = np.cumsum(db[::-1])[::-1]
    out = {name: a[:n] for name, a in res.items()}
    out["dh0"] = dS
    return out


@pytest.mark.parametrize("seed,n,C,d,weak", [
    (1, 13, 4, 4, False),   # ragged tail chunk
    (2, 16, 4, 4, False),   # whole chunks only
    (3, 37, 8, 4, False),
    (4, 50, 8, 4, True),    # gates near zero: long-range terms dominate
    (5, 1, 4, 4, False),    # one token
    (6, 130, 64, 8, False),  # the kernels' chunk size, three chunks
])
def test_chunked_backward_matches_token_oracle(oracle_lib, seed, n, C, d, weak):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q, v = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    g = -np.logaddexp(0.0, rng.standard_normal(n)) * (0.01 if weak else 1.0)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(n)))
    h0 = 0.3 * rng.standard_normal((d, d))
    dout, dst = rng.standard_normal((n, d)), rng.standard_normal((d, d))
    p = Problem(B=1, T=n, nk=1, nv=1, dk=d, dv=d, q=q, k=k, v=v, g=g[:, None], beta=beta[:, None],
                h0=h0[None, None], cu_seqlens=None)
    ref = oracle.token_loop_backward(p, dout[:, None, :], dst[None, None])
    got = chunked_backward(q, k, v, g, beta, h0, dout, dst, C)
    want = {"dq": ref["dq"][:, 0], "dk": ref["dk"][:, 0], "dv": ref["dv"][:, 0], "dg": ref["dg"][:, 0],
            "dbeta": ref["dbeta"][:, 0], "dh0": ref["dh0"][0, 0]}
    for name, r in want.items():
        err = np.max(np.abs(got[name] - r)) / max(np.max(np.abs(r)), 1e-300)
        assert err < 1e-10, (name, err)
