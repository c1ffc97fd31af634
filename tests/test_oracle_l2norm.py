"""Pins for the oracle's fused-prologue normalisation (no GPU).

``oracle.l2norm_heads`` scales every 128-wide q/k head row by
1 / sqrt(sum(x^2) + eps). The pins: with eps = 0 it is numpy's own vector
norm per head row; a zero row stays zero; and the whole normalised recurrence
is invariant (to within eps) under an independent power-of-two scale of each
q and each k head row, which fails for a dropped square root, a norm taken
over the wrong axis (across heads or over the whole row) or a prologue that
skips q or k."""
import numpy as np
import pytest

import gdn_synth
import oracle
from tests.oracle_pins import rel


def test_eps_free_norm_is_numpys_vector_norm():
    p = gdn_synth.make_problem(seed=71, B=1, T=40, nk=3, nv=3, qk_raw=True)
    x = oracle.bf16_to_f64(p.k)[:, : 3 * 128].reshape(40, 3, 128)
    ref = x / np.linalg.norm(x, axis=-1, keepdims=True)
    got = oracle.l2norm_heads(p.k, 3, 128, eps=0.0).reshape(40, 3, 128)
    assert np.abs(got - ref).max() < 1e-15


def test_zero_row_stays_zero():
    x = np.zeros((2, 256), dtype=np.float32)
    x[1, 128:] = 3.0
    y = oracle.l2norm_heads(x, 2, 128)
    assert np.all(y[0] == 0.0) and np.all(y[1, :128] == 0.0)
    assert abs(np.linalg.norm(y[1, 128:]) - 1.0) < 1e-9


def _scale_head_rows(bits, heads, d, exps):
    """Multiply head row (r, h) of bf16 bits by 2^exps[r, h] (exact)."""
    f = gdn_synth.bf16_bits_to_f32(bits).copy()
    rows = f.shape[0]
    f[:, : heads * d] = (f[:, : heads * d].reshape(rows, heads, d)
                         * np.exp2(exps)[:, :, None].astype(np.float32)).reshape(rows, heads * d)
    return gdn_synth.f32_to_bf16_bits(f)


@pytest.mark.parametrize("varlen", [False, True])
def test_normalised_recurrence_is_row_scale_invariant(oracle_lib, varlen):
    kw = dict(lengths=[37, 90]) if varlen else dict(T=70)
    p = gdn_synth.make_problem(seed=72, B=2, nk=2, nv=4, h0_std=0.02, qk_raw=True, **kw)
    o, h = oracle.token_loop(p, qk_l2norm=True)
    rng = np.random.default_rng(5)
    p2 = gdn_synth.make_problem(seed=72, B=2, nk=2, nv=4, h0_std=0.02, qk_raw=True, **kw)
    p2.q = _scale_head_rows(p.q, 2, 128, rng.integers(0, 4, size=(p.rows, 2)))
    p2.k = _scale_head_rows(p.k, 2, 128, rng.integers(0, 4, size=(p.rows, 2)))
    assert not np.array_equal(p2.q, p.q) and not np.array_equal(p2.k, p.k)
    o2, h2 = oracle.token_loop(p2, qk_l2norm=True)
    # eps perturbs a unit row by about eps / (2 |x|^2) <= 3e-7 here (|x| >= ~1.4)
    assert rel(o2, o) < 1e-5 and rel(h2, h) < 1e-5
    # the same scales without the prologue change the result by O(1)
    o3, _ = oracle.token_loop(p2)
    o4, _ = oracle.token_loop(p)
    assert rel(o3, o4) > 0.1


def test_prologue_is_identity_on_unit_rows(oracle_lib):
    # synthetic default rows are unit vectors up to bf16 rounding (|x| = 1 +- 2^-8):
    # the normalised recurrence stays within that rounding of the plain one
    p = gdn_synth.make_problem(seed=73, B=1, T=64, nk=1, nv=2, h0_std=0.02)
    o, h = oracle.token_loop(p)
    o2, h2 = oracle.token_loop(p, qk_l2norm=True)
    assert 0 < rel(o2, o) < 2e-2 and rel(h2, h) < 2e-2
