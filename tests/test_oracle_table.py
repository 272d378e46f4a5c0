"""Pins of the oracle's NF4 code table.

The pages fix: 16 levels derived from the quantiles (CDF) of a standard normal,
each bin holding an equal share of a zero-centred normal, and an exact zero
(inquiringlines.com note, mechanism paragraph; ashishsrivastav.com "QLoRA:
Fine-Tuning a 70B on One GPU", section "NF4 Quantization: Beyond Standard INT4").
The outermost probability delta is a reading (not fixed by the pages): its
value is parity-unpinned and only recorded here.
"""
import math
import os

import numpy as np
import pytest
from scipy import special

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nf4_table.txt")


def test_table_shape_and_invariants(oracle):
    L = oracle.nf4_table()
    assert L.dtype == np.float32 and L.shape == (16,)
    assert np.all(np.diff(L.astype(np.float64)) > 0), "levels must be strictly increasing"
    assert L[0] == -1.0 and L[15] == 1.0 and L[7] == 0.0
    assert np.sum(L < 0) == 7 and np.sum(L > 0) == 8


def test_inverse_cdf_against_library(oracle):
    # Bisection on erfc agrees with scipy's ndtri (a different algorithm).
    for p in np.linspace(0.5, 0.999, 41):
        assert abs(oracle.norm_ppf(p) - special.ndtri(p)) <= 1e-13 * max(1.0, abs(special.ndtri(p)))


def test_equal_share_bins(oracle):
    # Each half is Phi^-1 of equally spaced probabilities between 1/2 and delta,
    # so Phi(L * q) - 1/2 grows in equal steps (8 on the positive side, 7 on the
    # negative side). Checked with scipy's ndtr / ndtri, not with the oracle's own
    # bisection; the tolerance covers the fp32 rounding of the levels.
    L = oracle.nf4_table().astype(np.float64)
    q = special.ndtri(oracle.nf4_delta())
    top = special.ndtr(q) - 0.5
    for j in range(1, 9):
        share = (special.ndtr(L[7 + j] * q) - 0.5) / top
        assert abs(share - j / 8) < 2e-7, (j, share)
    for j in range(1, 8):
        share = (0.5 - special.ndtr(L[7 - j] * q)) / top
        assert abs(share - j / 7) < 2e-7, (j, share)


def test_delta_reading_recorded(oracle):
    # Reading (parity-unpinned by the pages): the average of the centres of the
    # outermost bins of a 16-bin and a 15-bin equal-mass split.
    d = oracle.nf4_delta()
    assert 1 - 1 / 30 < d < 1 - 1 / 32
    assert d == pytest.approx(0.5 * (31 / 32 + 29 / 30), abs=0)


def test_table_matches_golden(oracle):
    vals = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            i, hx, _ = line.split()
            vals.append(float.fromhex(hx))
    assert len(vals) == 16
    L = oracle.nf4_table()
    assert [float(v) for v in L] == vals


def test_table_normal_quantile_sanity(oracle):
    # The first positive level is Phi^-1 of the smallest step over Phi^-1(delta):
    # an independent closed form through math.erf-based bisection is not needed;
    # this checks the order of magnitude against the textbook median-absolute
    # value of a standard normal (0.6745 at p = 3/4).
    q = special.ndtri(oracle.nf4_delta())
    # the level whose probability is nearest 3/4 lies near 0.6745 / q
    L = oracle.nf4_table().astype(np.float64)
    probs = special.ndtr(L * q)
    j = int(np.argmin(np.abs(probs - 0.75)))
    assert abs(L[j] * q - 0.6745) < 0.1
    assert math.isclose(float(L[15] * q), float(q))
