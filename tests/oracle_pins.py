"""Checks that pin the oracle to facts other than itself.

Each ``pin_*`` function takes ``run(q, k, v, g, beta, h0, B, T, nk, nv, dk, dv,
cu_seqlens) -> (out, hT)`` working on fp64 row arrays and asserts a property
the gated delta rule must have: a closed form, an exact rational expansion,
or an invariant. ``tests/test_oracle.py`` applies them to the C token loop;
``tests/test_oracle_mutants.py`` applies them to deliberately wrong variants
to show that each plausible mistake fails at least one of them.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def rel(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def _rand_inputs(rng, rows, nk, nv, dk, dv, normalise=True):
    q = rng.standard_normal((rows, nk, dk))
    k = rng.standard_normal((rows, nk, dk))
    if normalise:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((rows, nv * dv))
    g = -np.logaddexp(0.0, rng.standard_normal((rows, nv)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((rows, nv))))
    return q.reshape(rows, nk * dk), k.reshape(rows, nk * dk), v, g, beta


def pin_pure_decay(run, seed=1):
    """beta = 0: S_T = e^{sum g} S_0 and o_t = e^{sum_{s<=t} g_s} S_0^T q_t / sqrt(dk)."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 37, 16, 8
    q, k, v, g, beta = _rand_inputs(rng, T, 1, 1, dk, dv)
    beta[:] = 0.0
    h0 = rng.standard_normal((1, 1, dk, dv))
    out, hT = run(q, k, v, g, beta, h0, 1, T, 1, 1, dk, dv, None)
    G = np.cumsum(g[:, 0])
    exp_out = np.exp(G)[:, None] * (q @ h0[0, 0]) / np.sqrt(dk)
    assert rel(out[:, 0], exp_out) < 1e-13
    assert rel(hT[0, 0], np.exp(G[-1]) * h0[0, 0]) < 1e-13
    # zero state stays zero
    out0, hT0 = run(q, k, v, g, beta, np.zeros_like(h0), 1, T, 1, 1, dk, dv, None)
    assert np.abs(out0).max() == 0.0 and np.abs(hT0).max() == 0.0


def _orthonormal_rows(rng, n, d):
    m, _ = np.linalg.qr(rng.standard_normal((d, d)))
    return m[:n]


def pin_exact_overwrite(run, seed=2):
    """g = 0, beta = 1, orthonormal keys: each write replaces the value stored at
    its key, so S_T = (I - sum k k^T) S_0 + sum k v^T and a query equal to an
    earlier (or the current) key reads that key's value / sqrt(dk)."""
    rng = np.random.default_rng(seed)
    dk, dv, T = 32, 12, 20
    keys = _orthonormal_rows(rng, T, dk)
    v = rng.standard_normal((T, dv))
    h0 = rng.standard_normal((1, 1, dk, dv))
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    src = np.array([rng.integers(0, t + 1) for t in range(T)])  # q_t = k_{src[t]}, src[t] <= t
    q = keys[src]
    out, hT = run(q, keys, v, g, beta, h0, 1, T, 1, 1, dk, dv, None)
    assert rel(out[:, 0], v[src] / np.sqrt(dk)) < 1e-12
    P = np.eye(dk) - keys.T @ keys
    assert rel(hT[0, 0], P @ h0[0, 0] + keys.T @ v) < 1e-12
    # a key written twice keeps the later value
    keys2 = keys.copy()
    keys2[7] = keys[3]
    q2 = np.repeat(keys[3][None], T, axis=0)
    out2, _ = run(q2, keys2, v, g, beta, h0, 1, T, 1, 1, dk, dv, None)
    assert rel(out2[7:, 0], np.repeat(v[7][None], T - 7, axis=0) / np.sqrt(dk)) < 1e-12
    assert rel(out2[3:7, 0], np.repeat(v[3][None], 4, axis=0) / np.sqrt(dk)) < 1e-12


def pin_strong_decay(run, seed=3):
    """g = -80 wipes the previous state at every step: S_t = beta_t k_t v_t^T up
    to e^{-80}, so o_t = beta_t (k_t . q_t) v_t / sqrt(dk)."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 29, 16, 16
    q, k, v, g, beta = _rand_inputs(rng, T, 1, 1, dk, dv)
    g[:] = -80.0
    h0 = rng.standard_normal((1, 1, dk, dv))
    out, hT = run(q, k, v, g, beta, h0, 1, T, 1, 1, dk, dv, None)
    expect = beta[:, :1] * np.sum(k * q, axis=1, keepdims=True) * v / np.sqrt(dk)
    assert rel(out[:, 0], expect) < 1e-12
    assert rel(hT[0, 0], beta[-1, 0] * np.outer(k[-1], v[-1])) < 1e-12


def _frac_matrix(a):
    return [[Fraction(float(x)) for x in row] for row in a]


def pin_brute_force_rational(run, seed=4):
    """dk = dv = 4, T <= 8: expand S_T = A_T...A_1 S_0 + sum_t A_T...A_{t+1} beta_t k_t v_t^T
    with A_t = e^{g_t}(I - beta_t k_t k_t^T) in exact rational arithmetic
    (e^{g_t} fixed to its fp64 value; 1/sqrt(4) = 1/2 is exact)."""
    rng = np.random.default_rng(seed)
    d = 4
    for T in (1, 2, 5, 8):
        q, k, v, g, beta = _rand_inputs(rng, T, 1, 1, d, d)
        h0 = rng.standard_normal((1, 1, d, d))
        out, hT = run(q, k, v, g, beta, h0, 1, T, 1, 1, d, d, None)
        a = [Fraction(float(np.exp(x))) for x in g[:, 0]]
        S = _frac_matrix(h0[0, 0])
        for t in range(T):
            kt = [Fraction(float(x)) for x in k[t]]
            vt = [Fraction(float(x)) for x in v[t]]
            qt = [Fraction(float(x)) for x in q[t]]
            b = Fraction(float(beta[t, 0]))
            A = [[a[t] * ((1 if i == j else 0) - b * kt[i] * kt[j]) for j in range(d)] for i in range(d)]
            S = [[sum(A[i][m] * S[m][j] for m in range(d)) + b * kt[i] * vt[j] for j in range(d)]
                 for i in range(d)]
            o = [sum(S[i][j] * qt[i] for i in range(d)) / 2 for j in range(d)]
            assert np.allclose(out[t, 0], [float(x) for x in o], rtol=1e-13, atol=1e-15)
        assert np.allclose(hT[0, 0], [[float(x) for x in row] for row in S], rtol=1e-13, atol=1e-15)


def pin_dense_transition(run, seed=5):
    """d = 128: the transition-matrix expansion in fp64 dense products."""
    rng = np.random.default_rng(seed)
    d, T = 128, 8
    q, k, v, g, beta = _rand_inputs(rng, T, 1, 1, d, d)
    h0 = rng.standard_normal((1, 1, d, d)) * 0.02
    out, hT = run(q, k, v, g, beta, h0, 1, T, 1, 1, d, d, None)
    S = h0[0, 0]
    for t in range(T):
        A = np.exp(g[t, 0]) * (np.eye(d) - beta[t, 0] * np.outer(k[t], k[t]))
        S = A @ S + beta[t, 0] * np.outer(k[t], v[t])
        assert rel(out[t, 0], S.T @ q[t] / np.sqrt(d)) < 1e-12
    assert rel(hT[0, 0], S) < 1e-12


def pin_linearity(run, seed=6):
    """Output and final state are jointly linear in (V, S_0)."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 50, 16, 8
    q, k, v1, g, beta = _rand_inputs(rng, T, 1, 1, dk, dv)
    v2 = rng.standard_normal(v1.shape)
    s1 = rng.standard_normal((1, 1, dk, dv))
    s2 = rng.standard_normal((1, 1, dk, dv))
    al = 0.37
    o1, h1 = run(q, k, v1, g, beta, s1, 1, T, 1, 1, dk, dv, None)
    o2, h2 = run(q, k, v2, g, beta, s2, 1, T, 1, 1, dk, dv, None)
    o3, h3 = run(q, k, al * v1 + v2, g, beta, al * s1 + s2, 1, T, 1, 1, dk, dv, None)
    assert rel(o3, al * o1 + o2) < 1e-12
    assert rel(h3, al * h1 + h2) < 1e-12


def pin_split_sequence(run, seed=7):
    """Running T1 then T2 with the carried state equals running T1+T2 at once."""
    rng = np.random.default_rng(seed)
    T1, T2, dk, dv = 45, 70, 16, 16
    q, k, v, g, beta = _rand_inputs(rng, T1 + T2, 1, 1, dk, dv)
    h0 = rng.standard_normal((1, 1, dk, dv)) * 0.1
    o, h = run(q, k, v, g, beta, h0, 1, T1 + T2, 1, 1, dk, dv, None)
    oa, ha = run(q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], h0, 1, T1, 1, 1, dk, dv, None)
    ob, hb = run(q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], ha, 1, T2, 1, 1, dk, dv, None)
    assert rel(np.concatenate([oa, ob]), o) < 1e-13
    assert rel(hb, h) < 1e-13


def pin_varlen_pack(run, seed=8):
    """A packed ragged batch equals each sequence run on its own."""
    rng = np.random.default_rng(seed)
    lens = [13, 0, 40, 7]
    dk, dv, nk, nv = 16, 8, 2, 4
    rows = sum(lens)
    q, k, v, g, beta = _rand_inputs(rng, rows, nk, nv, dk, dv)
    h0 = rng.standard_normal((len(lens), nv, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, h = run(q, k, v, g, beta, h0, len(lens), rows, nk, nv, dk, dv, cu)
    for s, n in enumerate(lens):
        r = slice(cu[s], cu[s + 1])
        if n == 0:
            assert rel(h[s], h0[s]) == 0.0  # empty sequence: state unchanged
            continue
        os_, hs = run(q[r], k[r], v[r], g[r], beta[r], h0[s:s + 1], 1, n, nk, nv, dk, dv, None)
        assert rel(o[r], os_) < 1e-14
        assert rel(h[s], hs[0]) < 1e-14


def pin_gqa_duplication(run, seed=9):
    """v-head h reads q/k head h // (nv/nk): nk = 2 equals nk = 4 with each q/k
    head duplicated into consecutive slots."""
    rng = np.random.default_rng(seed)
    T, dk, dv, nv = 30, 16, 8, 4
    q, k, v, g, beta = _rand_inputs(rng, T, 2, nv, dk, dv)
    h0 = rng.standard_normal((1, nv, dk, dv))
    o, h = run(q, k, v, g, beta, h0, 1, T, 2, nv, dk, dv, None)
    q4 = np.repeat(q.reshape(T, 2, dk), 2, axis=1).reshape(T, 4 * dk)
    k4 = np.repeat(k.reshape(T, 2, dk), 2, axis=1).reshape(T, 4 * dk)
    o4, h4 = run(q4, k4, v, g, beta, h0, 1, T, 4, nv, dk, dv, None)
    assert rel(o, o4) < 1e-15 and rel(h, h4) < 1e-15
    # and heads in one group really differ when their gates differ
    assert rel(o[:, 0], o[:, 1]) > 1e-3


def pin_head_permutation(run, seed=10):
    """Permuting v-heads (with their v, g, beta and state) permutes the outputs."""
    rng = np.random.default_rng(seed)
    T, dk, dv, nv = 25, 16, 8, 3
    q, k, v, g, beta = _rand_inputs(rng, T, 1, nv, dk, dv)
    h0 = rng.standard_normal((1, nv, dk, dv))
    o, h = run(q, k, v, g, beta, h0, 1, T, 1, nv, dk, dv, None)
    perm = np.array([2, 0, 1])
    vp = v.reshape(T, nv, dv)[:, perm].reshape(T, nv * dv)
    op, hp = run(q, k, vp, g[:, perm], beta[:, perm], h0[:, perm], 1, T, 1, nv, dk, dv, None)
    assert rel(op, o[:, perm]) < 1e-15 and rel(hp, h[:, perm]) < 1e-15


def pin_bounded(run, seed=11):
    """With unit keys and beta in (0,1), I - beta k k^T is a contraction, so
    ||S_t||_F <= ||S_0||_F + sum_s beta_s ||v_s|| for any gate g <= 0."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 300, 16, 16
    q, k, v, g, beta = _rand_inputs(rng, T, 1, 1, dk, dv)
    g[:] = 0.0
    h0 = rng.standard_normal((1, 1, dk, dv))
    _, h = run(q, k, v, g, beta, h0, 1, T, 1, 1, dk, dv, None)
    bound = np.linalg.norm(h0) + np.sum(beta[:, 0] * np.linalg.norm(v, axis=1))
    assert np.linalg.norm(h) <= bound
    # with g = 0 and beta -> 1 on the same key repeated, the state saturates at that key's value
    kk = np.repeat(k[:1], T, axis=0)
    vv = np.repeat(v[:1], T, axis=0)
    bb = np.full_like(beta, 0.5)
    _, h2 = run(q, kk, vv, g, bb, np.zeros_like(h0), 1, T, 1, 1, dk, dv, None)
    assert rel(h2[0, 0].T @ k[0], v[0]) < 1e-12


ALL_PINS = [
    pin_pure_decay,
    pin_exact_overwrite,
    pin_strong_decay,
    pin_brute_force_rational,
    pin_dense_transition,
    pin_linearity,
    pin_split_sequence,
    pin_varlen_pack,
    pin_gqa_duplication,
    pin_head_permutation,
    pin_bounded,
]
