"""The segment-parallel schedule's recipe, checked with the fp64 oracle on the CPU (no GPU).

The schedule cuts a sequence at chunk boundaries into G segments and uses that the
state map of a segment is affine in its entry state (stage 2 of ssm_gdn_a3.rs
`gdn_prefill_fla`'s doc comment is linear in S): S_end = M S_start + N. It obtains M by
running the segment from S = I with v = 0 and N by running it from S = 0 with the real
v, chains X_{g+1} = M_g X_g + N_g, and runs every segment again from its X_g for the
outputs. Here each step is an oracle call, and the stitched outputs and final state
must equal one serial oracle run of the whole sequence.
"""
import numpy as np
import pytest

import oracle


def run(q, k, v, g, beta, h0):
    d = k.shape[1]
    out, hT = oracle.token_loop_raw(q, k, v, g, beta, h0[None, None], B=1, T=q.shape[0], nk=1, nv=1, dk=d, dv=d)
    return out[:, 0], hT[0, 0]


@pytest.mark.parametrize("n,L,gate_scale", [(200, 64, 1.0), (300, 64, 0.01), (129, 64, 1.0), (97, 32, 0.05)])
def test_segments_stitch_to_the_serial_run(oracle_lib, n, L, gate_scale):
    rng = np.random.default_rng(n + L)
    d = 4
    k = rng.standard_normal((n, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q, v = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    g = (-np.logaddexp(0.0, rng.standard_normal(n)) * gate_scale)[:, None]
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal(n))))[:, None]
    h0 = 0.3 * rng.standard_normal((d, d))
    out_ref, hT_ref = run(q, k, v, g, beta, h0)

    bounds = list(range(0, n, L)) + [n]
    X = h0
    outs = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        seg = (q[a:b], k[a:b])
        _, M = run(*seg, np.zeros_like(v[a:b]), g[a:b], beta[a:b], np.eye(d))
        _, N = run(*seg, v[a:b], g[a:b], beta[a:b], np.zeros((d, d)))
        out_g, end_g = run(*seg, v[a:b], g[a:b], beta[a:b], X)
        X_next = M @ X + N
        assert np.allclose(X_next, end_g, rtol=1e-12, atol=1e-14)  # the affine map is exact
        outs.append(out_g)
        X = X_next
    assert len(bounds) - 1 >= 2
    assert np.allclose(np.concatenate(outs), out_ref, rtol=1e-11, atol=1e-13)
    assert np.allclose(X, hT_ref, rtol=1e-11, atol=1e-13)
