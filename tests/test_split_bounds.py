"""Facts about splitting fp32 into bf16 parts that the tensor-core append
kernels' error bounds rest on, checked exhaustively over one binade of fp32
significands (the relative residual depends on the significand only, for
normal numbers).

- hi + mid + lo (three parts, each the bf16 rounding of what the earlier parts
  left) reproduces every normal fp32 value exactly, so the head_dim <= 128
  kernel's products with R are exact and its bound is the accumulation alone.
- hi + lo (two parts, the head_dim 256 kernel) leaves |R - hi - lo| up to
  about 2^-17·|R|: above 2^-18, so no elementwise constant of 2^-18 bounds the
  residual term, and the kernel takes the column norm of the residual from R
  itself.
"""
import numpy as np


def _bf16(x):
    """Round fp32 to bf16 (round to nearest, ties to even), returned as fp32."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _parts(x):
    hi = _bf16(x)
    r1 = (x - hi).astype(np.float32)
    mid = _bf16(r1)
    r2 = (r1 - mid).astype(np.float32)
    lo = _bf16(r2)
    return hi, mid, lo, r1, r2


def _binade(exp):
    m = np.arange(0, 1 << 23, dtype=np.uint32)
    return ((np.uint32(exp) << 23) | m).view(np.float32)


def test_bf16_rounding_helper():
    # values with a known bf16 rounding: 1 + 2^-8 is a tie (rounds to even, 1),
    # 1 + 3·2^-8 rounds up to 1 + 2^-6 ... checked against the definition
    one = np.float32(1.0)
    assert _bf16(np.float32(1.0 + 2.0 ** -8)) == one
    assert _bf16(np.float32(1.0 + 3 * 2.0 ** -8)) == np.float32(1.0 + 2.0 ** -6)
    assert _bf16(np.float32(1.0 + 2.0 ** -8 + 2.0 ** -20)) == np.float32(1.0 + 2.0 ** -7)
    assert _bf16(np.float32(-1.5)) == np.float32(-1.5)


def test_three_parts_are_exact():
    for exp in (127, 122, 96):                 # [1, 2), [2^-5, 2^-4), [2^-31, 2^-30)
        x = _binade(exp)
        hi, mid, lo, r1, r2 = _parts(x)
        # each residual is exact in fp32 (Sterbenz-like), so the sum is exact
        # when the last residual is itself a bf16 value
        assert np.array_equal((r2 - lo).astype(np.float32), np.zeros_like(x))
        s = hi.astype(np.float64) + mid.astype(np.float64) + lo.astype(np.float64)
        assert np.array_equal(s, x.astype(np.float64))


def test_two_part_residual_reaches_2_to_minus_17():
    x = _binade(127)
    hi, mid, _, _, r2 = _parts(x)
    # r2 = x - hi - mid exactly (fp64 check of the fp32 residual)
    assert np.array_equal(r2.astype(np.float64),
                          x.astype(np.float64) - hi.astype(np.float64) - mid.astype(np.float64))
    rel = np.abs(r2.astype(np.float64)) / x.astype(np.float64)
    assert rel.max() <= 2.0 ** -17
    assert rel.max() > 2.0 ** -18              # 2^-18·|R| is not an elementwise bound
    # scale invariance over binades (normal numbers)
    y = _binade(110)
    _, _, _, _, r2y = _parts(y)
    assert np.allclose(np.abs(r2y.astype(np.float64)) / y.astype(np.float64), rel, rtol=0, atol=0)
