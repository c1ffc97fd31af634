"""Pins for the CPU oracle (no GPU): closed forms, exact expansions, invariants,
and agreement with the independent chunked-WY evaluation."""
import numpy as np
import pytest

import gdn_synth
import oracle
from oracle.chunked_wy import chunked_prefill
from tests import oracle_pins
from tests.oracle_pins import rel


def c_run(q, k, v, g, beta, h0, B, T, nk, nv, dk, dv, cu):
    return oracle.token_loop_raw(np.asarray(q, np.float64), np.asarray(k, np.float64),
                                 np.asarray(v, np.float64), np.asarray(g, np.float64),
                                 np.asarray(beta, np.float64), h0, B=B, T=T, nk=nk, nv=nv,
                                 dk=dk, dv=dv, cu_seqlens=cu)


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_token_loop_pins(oracle_lib, pin):
    pin(c_run)


@pytest.mark.parametrize("C", [1, 16, 64])
def test_token_loop_matches_chunked_wy_config0(oracle_lib, C):
    p = gdn_synth.config_problem(0)
    o, h = oracle.token_loop(p)
    o2, h2, _ = chunked_prefill(p, C=C)
    assert rel(o2, o) < 1e-12 and rel(h2, h) < 1e-12


@pytest.mark.parametrize("C", [1, 16, 64])
def test_token_loop_matches_chunked_wy_gqa_state(oracle_lib, C):
    # GQA (nv = 2 nk), carried-in state, a ragged tail chunk, weak decay.
    p = gdn_synth.make_problem(seed=11, B=2, T=150, nk=2, nv=4, h0_std=0.02,
                               gate_mu=-5.0, gate_sigma=0.5)
    o, h = oracle.token_loop(p)
    o2, h2, _ = chunked_prefill(p, C=C)
    assert rel(o2, o) < 1e-12 and rel(h2, h) < 1e-12


def test_token_loop_matches_chunked_wy_varlen_packed_strides(oracle_lib):
    # ragged lengths incl. 1 and an exact multiple of 64, padded q/k/v rows,
    # g/beta packed at stride 2*nv as in the conv layout.
    p = gdn_synth.make_problem(seed=12, B=4, lengths=[1, 64, 97, 130], nk=1, nv=2,
                               h0_std=0.02, pad_qk=8, pad_v=16, gb_stride=4)
    o, h = oracle.token_loop(p)
    o2, h2, _ = chunked_prefill(p, C=64)
    assert rel(o2, o) < 1e-12 and rel(h2, h) < 1e-12


def test_token_loop_zero_gate(oracle_lib):
    # g = 0: no decay at all, so the cross-chunk state path carries everything.
    p = gdn_synth.make_problem(seed=13, B=1, T=300, nk=1, nv=2, gate_zero=True, h0_std=0.02)
    o, h = oracle.token_loop(p)
    o2, h2, _ = chunked_prefill(p, C=64)
    assert rel(o2, o) < 1e-12 and rel(h2, h) < 1e-12


def test_head_subset_matches_full(oracle_lib):
    p = gdn_synth.make_problem(seed=14, B=2, T=70, nk=2, nv=4, h0_std=0.02)
    o, h = oracle.token_loop(p)
    os_, hs = oracle.token_loop(p, heads=[3, 1])
    for hd in (1, 3):
        assert np.array_equal(os_[:, hd], o[:, hd]) and np.array_equal(hs[:, hd], h[:, hd])
    assert not os_[:, 0].any() and not os_[:, 2].any()


def test_oracle_threads_deterministic(oracle_lib):
    p = gdn_synth.make_problem(seed=15, B=2, T=90, nk=1, nv=3)
    a = oracle.token_loop(p, threads=1)
    b = oracle.token_loop(p, threads=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_oracle_rejects_bad_heads(oracle_lib):
    p = gdn_synth.make_problem(seed=16, B=1, T=8, nk=1, nv=2)
    with pytest.raises(RuntimeError):
        oracle.token_loop_raw(p.q, p.k, p.v, p.g, p.beta, p.h0, B=1, T=8, nk=2, nv=3,
                              dk=128, dv=128)


def test_bf16_rounding_reference_values():
    # round-to-nearest-even at the bf16 boundary, and exact widening
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 1e-40, np.inf], dtype=np.float32)
    b = gdn_synth.f32_to_bf16_bits(x)
    assert list(b[:4]) == [0x3F80, 0x3F80, 0x3F82, 0xC020]
    assert b[5] == 0x7F80
    back = gdn_synth.bf16_bits_to_f32(b)
    assert back[0] == 1.0 and back[3] == -2.5


def test_synth_deterministic_and_independent_streams():
    a = gdn_synth.config_problem(0)
    b = gdn_synth.config_problem(0)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.g, b.g)
    # changing the number of v heads leaves q untouched (own stream)
    c = gdn_synth.make_problem(seed=1000, B=1, T=256, nk=1, nv=2)
    assert np.array_equal(a.q, c.q)
    # q/k rows are unit-norm before bf16 rounding
    qf = gdn_synth.bf16_bits_to_f32(a.q).astype(np.float64)
    assert np.allclose(np.linalg.norm(qf, axis=1), 1.0, atol=5e-3)


def test_config3_lengths():
    lens = gdn_synth.draw_lengths(1003, 8, 100, 16000)
    assert len(lens) == 8 and all(100 <= x <= 16000 and x % 64 for x in lens)
