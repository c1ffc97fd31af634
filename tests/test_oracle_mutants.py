"""The oracle's pins are discriminating: each plausible mistake (planted here,
on the CPU, in a small Python copy of the recurrence) fails at least one pin,
while the unmutated copy passes them all."""
import numpy as np
import pytest

from tests import oracle_pins


def make_runner(mutation):
    def run(q, k, v, g, beta, h0, B, T, nk, nv, dk, dv, cu):
        q, k, v, g, beta = (np.asarray(x, np.float64) for x in (q, k, v, g, beta))
        rows = q.shape[0]
        out = np.zeros((rows, nv, dv))
        hT = np.zeros((B, nv, dk, dv))
        group = nv // nk
        bounds = ([(b * T, T) for b in range(B)] if cu is None
                  else [(int(cu[s]), int(cu[s + 1] - cu[s])) for s in range(B)])
        for s, (r0, n) in enumerate(bounds):
            for h in range(nv):
                kh = (h % nk) if mutation == "gqa_modulo" else h // group
                S = np.array(h0[s, h], dtype=np.float64)
                for r in range(r0, r0 + n):
                    qt = q[r, kh * dk:(kh + 1) * dk]
                    kt = k[r, kh * dk:(kh + 1) * dk]
                    vt = v[r, h * dv:(h + 1) * dv]
                    a = np.exp(g[r, h])
                    b = beta[r, h]
                    if mutation == "no_decay":
                        a = 1.0
                    if mutation == "read_before_write":
                        o = S.T @ qt * a
                    if mutation == "decay_after_write":
                        S = a * (S + b * np.outer(kt, vt - S.T @ kt))
                    else:
                        S = a * S
                        p = S.T @ kt
                        if mutation == "sign":
                            S = S + b * np.outer(kt, vt + p)
                        elif mutation == "beta_on_value_only":
                            S = S + np.outer(kt, b * vt - p)
                        else:
                            S = S + b * np.outer(kt, vt - p)
                    if mutation == "transposed_readout":
                        o = S @ qt
                    elif mutation != "read_before_write":
                        o = S.T @ qt
                    if mutation != "no_scale":
                        o = o / np.sqrt(dk)
                    out[r, h] = o
                hT[s, h] = S
        return out, hT

    return run


MUTATIONS = ["no_decay", "read_before_write", "decay_after_write", "sign",
             "beta_on_value_only", "transposed_readout", "no_scale", "gqa_modulo"]


def _fails_some_pin(run):
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(run)
        except (AssertionError, ValueError):
            return pin.__name__
    return None


def test_unmutated_copy_passes_all_pins():
    assert _fails_some_pin(make_runner(None)) is None


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_mutation_is_caught(mutation):
    assert _fails_some_pin(make_runner(mutation)) is not None
