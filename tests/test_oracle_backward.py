"""Pins for the oracle's backward (no GPU): every gradient the backward returns
(q, k, v, g, beta and the initial state) is checked element by element against
central finite differences of the fp64 forward oracle, on problems small enough
to perturb every input: GQA, a carried-in state, a ragged varlen batch with an
empty sequence, and a sequence longer than one 64-token checkpoint block."""
import numpy as np
import pytest

import oracle
from gdn_synth import Problem

EPS = 1e-5


def small_problem(seed, *, B=2, T=7, lengths=None, nk=1, nv=2, d=4):
    rng = np.random.default_rng(seed)
    if lengths is not None:
        cu = np.zeros(len(lengths) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lengths)
        B, rows, T = len(lengths), int(cu[-1]), int(cu[-1])
    else:
        cu, rows = None, B * T
    k = rng.standard_normal((rows, nk, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    return Problem(B=B, T=T, nk=nk, nv=nv, dk=d, dv=d,
                   q=rng.standard_normal((rows, nk * d)), k=k.reshape(rows, nk * d),
                   v=rng.standard_normal((rows, nv * d)),
                   g=-np.logaddexp(0.0, rng.standard_normal((rows, nv))),
                   beta=1.0 / (1.0 + np.exp(-rng.standard_normal((rows, nv)))),
                   h0=0.3 * rng.standard_normal((B, nv, d, d)), cu_seqlens=cu)


def loss(p, dout, dst):
    o, hT = oracle.token_loop(p)
    return float(np.sum(dout * o) + np.sum(dst * hT))


def check_all(p, seed, max_per_input=None):
    rng = np.random.default_rng(seed + 1)
    dout = rng.standard_normal((p.rows, p.nv, p.dv))
    dst = rng.standard_normal((p.B, p.nv, p.dk, p.dv))
    grads = oracle.token_loop_backward(p, dout, dst)
    targets = {"q": grads["dq"].reshape(p.rows, -1), "k": grads["dk"].reshape(p.rows, -1),
               "v": grads["dv"].reshape(p.rows, -1), "g": grads["dg"], "beta": grads["dbeta"],
               "h0": grads["dh0"]}
    worst = {}
    for name, ana in targets.items():
        x = getattr(p, name)
        idx = np.arange(x.size)
        if max_per_input is not None and x.size > max_per_input:
            idx = rng.choice(x.size, max_per_input, replace=False)
        err = 0.0
        for i in idx:
            flat = x.reshape(-1)
            keep = flat[i]
            flat[i] = keep + EPS
            lp = loss(p, dout, dst)
            flat[i] = keep - EPS
            lm = loss(p, dout, dst)
            flat[i] = keep
            fd = (lp - lm) / (2 * EPS)
            a = ana.reshape(-1)[i]
            err = max(err, abs(a - fd) / (1e-6 + abs(fd)))
            assert abs(a - fd) <= 1e-6 * (1.0 + abs(fd)), f"d{name}[{i}]: analytic {a!r} vs finite difference {fd!r}"
        worst[name] = err
    return worst


def test_backward_matches_finite_differences_gqa(oracle_lib):
    check_all(small_problem(11, B=2, T=7, nk=1, nv=2, d=4), 11)


def test_backward_matches_finite_differences_two_key_heads(oracle_lib):
    check_all(small_problem(12, B=1, T=9, nk=2, nv=4, d=3), 12)


def test_backward_varlen_with_empty_sequence(oracle_lib):
    p = small_problem(13, lengths=[5, 0, 3], nk=1, nv=1, d=4)
    check_all(p, 13)


def test_backward_across_checkpoint_blocks(oracle_lib):
    # 150 tokens: three 64-token blocks recomputed from their checkpoints
    check_all(small_problem(14, B=1, T=150, nk=1, nv=1, d=3), 14, max_per_input=60)


def test_zero_cotangent_gives_zero_gradients(oracle_lib):
    p = small_problem(15)
    grads = oracle.token_loop_backward(p, np.zeros((p.rows, p.nv, p.dv)), None)
    assert all(np.all(v == 0.0) for v in grads.values())
