"""Pin of the oracle's softmax denominator (reading r8) against a hand-derived row.

tests/golden/softmax_denominator.txt works out O and the LSE of one query row
by hand for inputs chosen so that the per-tile P~ codes are not proportional
to the unquantized probabilities (127 * 2^-0.5 is not an integer, and one code
sits on a rounding tie).  The oracle must reproduce those values; the same
oracle with the misreading planted (denominator summed from the dequantized
codes) must not.
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "softmax_denominator.txt")


def _read_golden():
    inputs = {"Q": {}, "K": {}, "V": {}}
    expect = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, _, rest = line.partition(" ")
            if head in inputs:
                row, _, entries = rest.partition(":")
                for e in entries.split():
                    ch, _, val = e.partition("=")
                    inputs[head][(int(row), int(ch))] = float(val)
            else:
                expect[head] = float(rest)
    return inputs, expect


def _tensors(inputs, N=129, d=8):
    import torch
    out = {}
    for name in ("Q", "K", "V"):
        x = torch.zeros(1, 1, N, d)
        for (row, ch), val in inputs[name].items():
            x[0, 0, row, ch] = val
        out[name] = x.to(torch.bfloat16)
    out["dO"] = torch.zeros(1, 1, N, d, dtype=torch.bfloat16)
    return out


def _row0(oracle_mod, l_from_codes):
    inputs, expect = _read_golden()
    x = _tensors(inputs)
    p = oracle_mod.problem(1, 1, 1, 129, 8, False, smooth_k=False, softmax_scale=math.log(2.0) / 128,
                           l_from_codes=l_from_codes)
    o, lse = oracle_mod.fwd(p, x["Q"], x["K"], x["V"])
    return o[0, 0, 0], float(lse[0, 0, 0]), expect


def test_oracle_matches_the_hand_derived_row(oracle_mod):
    o, lse, expect = _row0(oracle_mod, False)
    want = np.array([expect[f"O{c}"] for c in range(8)])
    np.testing.assert_allclose(o, want, rtol=1e-13, atol=1e-15)
    assert lse == pytest.approx(expect["LSE"], rel=1e-13)
    # the closed form of the denominator itself
    assert expect["l"] == pytest.approx(64 + 3 / (2 * math.sqrt(2)), rel=1e-15)


def test_denominator_from_codes_is_caught(oracle_mod):
    o, lse, expect = _row0(oracle_mod, True)
    want = np.array([expect[f"O{c}"] for c in range(4)])
    rel = np.abs(o[:4] - want) / want
    assert rel.min() > 1e-3, rel  # every nonzero output moves by ~0.2 %
    assert abs(lse - expect["LSE"]) > 1e-3
