"""Writes the stored expected values under tests/golden/ from the fp64 oracle alone.

The pages print no worked example of the recurrence, so every fixture here is an
oracle regression record: seeded inputs plus what the oracle's token loop (forward)
and its backward return for them. `tests/test_golden.py` replays each fixture, so a
later change to the oracle's arithmetic shows up as a failure there and must be
justified on its own.

    python tests/golden/make_golden.py          # rewrites gdn_varlen_d4.json

Case: two sequences of 3 and 6 tokens in one varlen batch (so the second one spans
more than one 4-token chunk of the chunked cross-check), nk = 1 key head shared by
nv = 2 value heads (GQA), d_k = d_v = 4, a carried-in state, unit-norm keys, gates
log(sigmoid(x)) and sigmoid betas, and random output and final-state cotangents.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

NAME = "gdn_varlen_d4.json"


def case_inputs(seed=20240917):
    rng = np.random.default_rng(seed)
    lengths = [3, 6]
    nk, nv, d = 1, 2, 4
    cu = [0, lengths[0], lengths[0] + lengths[1]]
    rows = cu[-1]
    k = rng.standard_normal((rows, nk, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    return {
        "B": len(lengths), "T": rows, "nk": nk, "nv": nv, "dk": d, "dv": d, "cu_seqlens": cu,
        "q": rng.standard_normal((rows, nk * d)).tolist(),
        "k": k.reshape(rows, nk * d).tolist(),
        "v": rng.standard_normal((rows, nv * d)).tolist(),
        "g": (-np.logaddexp(0.0, rng.standard_normal((rows, nv)))).tolist(),
        "beta": (1.0 / (1.0 + np.exp(-rng.standard_normal((rows, nv))))).tolist(),
        "h0": (0.3 * rng.standard_normal((len(lengths), nv, d, d))).tolist(),
        "dout": rng.standard_normal((rows, nv, d)).tolist(),
        "dst": rng.standard_normal((len(lengths), nv, d, d)).tolist(),
    }


def problem(case):
    from gdn_synth import Problem

    a = {key: np.asarray(case[key], dtype=np.float64) for key in ("q", "k", "v", "g", "beta", "h0")}
    return Problem(B=case["B"], T=case["T"], nk=case["nk"], nv=case["nv"], dk=case["dk"], dv=case["dv"],
                   cu_seqlens=np.asarray(case["cu_seqlens"], dtype=np.int32), **a)


def oracle_values(case):
    import oracle

    oracle.build()
    p = problem(case)
    out, hT = oracle.token_loop(p)
    grads = oracle.token_loop_backward(p, np.asarray(case["dout"]), np.asarray(case["dst"]))
    res = {"out": out.tolist(), "hT": hT.tolist()}
    res.update({key: val.tolist() for key, val in grads.items()})
    return res


def main():
    case = case_inputs()
    fixture = {
        "what": "oracle regression record: token-loop forward and backward on a seeded varlen GQA case",
        "source": "tests/golden/make_golden.py (calls only the oracle)",
        "inputs": case,
        "expected": oracle_values(case),
    }
    with open(os.path.join(HERE, NAME), "w") as fh:
        json.dump(fixture, fh, indent=1)
        fh.write("\n")


if __name__ == "__main__":
    main()
