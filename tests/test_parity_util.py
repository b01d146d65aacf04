"""Host checks of the parity helpers' rounding-tie bands (no GPU)."""

import numpy as np

from parity_util import REL_TIE, fp16_near_tie, fp32_rotation_bound


def test_fp32_rotation_bound_holds_for_an_fp32_product():
    rng = np.random.default_rng(7)
    for d in (64, 128, 256):
        x = rng.standard_normal((64, d)) * np.where(rng.random(d) < 0.03, 20.0, 1.0)
        R, _ = np.linalg.qr(rng.standard_normal((d, d)))
        x32, R32 = x.astype(np.float32), R.astype(np.float32)
        exact = x32.astype(np.float64) @ R32.astype(np.float64)
        # a sequential fp32 inner product rounds once per addition: d - 1 roundings
        y = np.zeros((64, d), np.float32)
        for k in range(d):
            y = (y + x32[:, k:k + 1] * R32[k:k + 1, :]).astype(np.float32)
        err = np.abs(y.astype(np.float64) - exact)
        # each product also rounds once: d products + d - 1 additions
        bound = fp32_rotation_bound(x32, R32, 2 * d)
        assert (err <= bound).all()
        # and the bound is not vacuous: the typical error is far below it
        assert np.median(err / bound) < 0.05


def test_fp16_near_tie_bands():
    # 1 + 2^-11 is the midpoint between fp16 1.0 and its successor
    mid = np.float32(1.0 + 2.0 ** -11)
    assert fp16_near_tie(mid)
    off = np.float32(mid + 4 * REL_TIE)            # outside the relative band
    assert not fp16_near_tie(off)
    assert fp16_near_tie(off, band=5 * REL_TIE)     # inside an absolute band that covers it
    far = np.float32(1.0 + 2.0 ** -12)              # a quarter step from either neighbour
    assert not fp16_near_tie(far, band=1e-5)
