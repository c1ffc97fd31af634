"""Replays the stored expected values under tests/golden/ (no GPU).

The fixtures are oracle regression records written by tests/golden/make_golden.py
(the pages print no worked example). The token-loop oracle must reproduce them, and
the independent chunked WY evaluation of the forward must agree with the stored
values at every chunk size, including chunks that split the longer sequence."""
import json
import os

import numpy as np
import pytest

from tests.golden import make_golden
from tests.oracle_pins import rel

FIXTURE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", make_golden.NAME)


@pytest.fixture(scope="module")
def fixture():
    with open(FIXTURE) as fh:
        return json.load(fh)


def test_inputs_are_the_seeded_case(fixture):
    case = make_golden.case_inputs()
    for key, val in case.items():
        assert np.array_equal(np.asarray(fixture["inputs"][key]), np.asarray(val)), key


def test_token_loop_reproduces_forward_and_backward(oracle_lib, fixture):
    got = make_golden.oracle_values(fixture["inputs"])
    for key, want in fixture["expected"].items():
        assert rel(np.asarray(got[key]), np.asarray(want)) < 1e-12, key


@pytest.mark.parametrize("C", [1, 2, 4, 64])
def test_chunked_wy_matches_stored_forward(fixture, C):
    from oracle.chunked_wy import chunked_prefill

    p = make_golden.problem(fixture["inputs"])
    out, hT, _ = chunked_prefill(p, C=C)
    assert rel(out, np.asarray(fixture["expected"]["out"])) < 1e-12
    assert rel(hT, np.asarray(fixture["expected"]["hT"])) < 1e-12
