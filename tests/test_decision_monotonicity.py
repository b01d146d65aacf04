"""The quantiser's decisions are monotone in the rotated values they read
(CPU, on the oracle's quantiser).

The tensor-core append kernels take each decision at y - e and at y + e and
accept it when the two agree, re-forming y exactly only where they differ.
That is sound because every decision is a monotone function of its inputs:
for a fixed (s, z) the code is non-decreasing in y; the stored zero z =
rnd(r·min) is non-decreasing in the group minimum, and the stored scale
s = rnd((r·max - r·min)/3) is non-decreasing in the maximum and non-increasing
in the minimum (rnd the fp16 or E4M3 rounding, r the clip ratio).  Between
two inputs that agree at both ends of an interval, so does every input inside
it.  These checks run the oracle's quantiser on groups built to vary one input
at a time.
"""

import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("fmt", ["f16", "e4m3"])
def test_codes_non_decreasing_in_y_for_a_fixed_pair(fmt):
    rng = np.random.default_rng(31)
    G = 64
    for _ in range(50):
        lo, hi = np.sort(rng.standard_normal(2) * 4).astype(np.float32)
        inner = np.sort(rng.uniform(lo, hi, G - 2).astype(np.float32))
        Y = np.concatenate([[lo, hi], inner]).astype(np.float32)[None, :]
        c, s, z = oracle.quantize_rows(Y, G, 0.9, fmt)
        assert np.all(np.diff(c[0, 2:].astype(np.int64)) >= 0)


@pytest.mark.parametrize("fmt", ["f16", "e4m3"])
def test_pair_monotone_in_the_group_extremes(fmt):
    rng = np.random.default_rng(32)
    G = 32
    base = rng.uniform(-1.0, 1.0, G).astype(np.float32)
    # the maximum grows (channel 0), everything else fixed: s does not fall, z stays
    maxes = np.sort(rng.uniform(1.0, 8.0, 400)).astype(np.float32)
    rows = np.repeat(base[None, :], len(maxes), axis=0)
    rows[:, 0] = maxes
    rows[:, 1] = -1.5
    _, s, z = oracle.quantize_rows(rows, G, 0.9, fmt)
    assert np.all(np.diff(s[:, 0].astype(np.float64)) >= 0)
    assert np.all(z[:, 0] == z[0, 0])
    # the minimum grows (channel 1) below the fixed maximum: z does not fall, s does not grow
    mins = np.sort(rng.uniform(-8.0, -1.0, 400)).astype(np.float32)
    rows = np.repeat(base[None, :], len(mins), axis=0)
    rows[:, 0] = 1.5
    rows[:, 1] = mins
    _, s, z = oracle.quantize_rows(rows, G, 0.9, fmt)
    assert np.all(np.diff(z[:, 0].astype(np.float64)) >= 0)
    assert np.all(np.diff(s[:, 0].astype(np.float64)) <= 0)
