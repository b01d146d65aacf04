"""Clipped group-wise asymmetric INT2 quantiser, 2-bit packing, record bytes.

Test infrastructure only (see the package docstring).

[OSCAR news] "サービングシステム：混合精度キャッシュレイアウト": history tokens are
stored in INT2 after the OSCAR rotation and clipping.  [Escha log] part 2,
settings table: one scale per group of 64 channels ("--kv-cache-quant-group-size
64"); fix 1: INT2 codes take 0.25 byte per element.

Readings where the pages are silent:
* every K/V vector is first rounded to bf16 (round to nearest even), the
  storage type of the unquantised windows; the quantiser reads that bf16
  vector, so a token's codes do not depend on whether it reached the history
  directly or by leaving the recent window;
* y = x · R is the exact product with the stored fp32 R, rounded to fp32
  (the precision the kernel carries y in);
* clipping scales the group's extremes toward zero: lo = r·min(y_g),
  hi = r·max(y_g) with the clip ratio r;
* scale s = fp16((hi - lo) / 3) and zero z = fp16(lo), a real-valued fp16
  offset (not an integer zero point);
* the fp8 variant ([OSCAR news] quotes 2.28 bits per KV element, which
  group 64 reaches with one byte each for s and z): s and z are rounded to
  float8 E4M3 instead (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
  no infinities, largest finite value 448), to nearest with ties to even,
  and values beyond ±448 saturate to ±448;
* the code is decided in fp32 from the rounded s and z:
  c = clamp(rint((y - z) / s), 0, 3), rint rounding half to even, each fp32
  operation correctly rounded; a group whose s rounds to 0 gets codes 0;
* dequantisation is ŷ = s·c + z;
* packing: channel j sits at bits 2·(j mod 4) of byte j // 4 (low bits first).
"""

import numpy as np


def bf16_round(x):
    """Round to bfloat16 (nearest, ties to even); returns float32 values."""
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = x32.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return rounded.astype(np.uint32).view(np.float32).reshape(x32.shape)


def bf16_bits(x):
    """bfloat16 bit patterns (uint16) of values that are already bf16-exact."""
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return (x32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_from_bits(b):
    """float32 values of bfloat16 bit patterns."""
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def e4m3_round(x):
    """Round to float8 E4M3 (nearest, ties to even), saturating at ±448.

    Normal numbers 2^e·(1 + m/8) for -6 <= e <= 8, subnormals m·2^-9; the
    spacing of the grid around |x| is 2^(max(e, -6) - 3) with e = floor(log2|x|).
    Returns float32 values (every E4M3 value is exact in fp16 and fp32).
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))          # a = f·2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)                          # floor(log2 a), clamped to the subnormal range
    ulp = np.ldexp(1.0, e - 3)
    r = np.rint(a / ulp) * ulp                          # exact: a/ulp and the product are scalings by 2^k
    r = np.minimum(r, 448.0)
    return np.copysign(r, x).astype(np.float32)


def e4m3_bits(v):
    """E4M3 bit patterns (uint8) of values that are already E4M3-exact."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    sign = np.signbit(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = ex - 1
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, e + 7, 0)
    man = np.where(normal, a / np.ldexp(1.0, e) - 1.0, a / 2.0 ** -9) * np.where(normal, 8.0, 1.0)
    man = np.where(a == 0, 0.0, man)
    bits = (sign.astype(np.int64) << 7) | (exp_field.astype(np.int64) << 3) | np.rint(man).astype(np.int64)
    return bits.astype(np.uint8)


def e4m3_from_bits(b):
    """Values (float32) of E4M3 bit patterns (0x7F / 0xFF, the NaNs, excluded)."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    sign = np.where(b >> 7, -1.0, 1.0)
    ef = (b >> 3) & 15
    m = b & 7
    val = np.where(ef == 0, m * 2.0 ** -9, np.ldexp(1.0 + m / 8.0, ef - 7))
    return (sign * val).astype(np.float32)


SCALE_FORMATS = ("f16", "e4m3")


def _round_scale(x, scale_fmt):
    if scale_fmt == "f16":
        return np.asarray(x, np.float32).astype(np.float16)
    if scale_fmt == "e4m3":
        return e4m3_round(x).astype(np.float16)
    raise ValueError("scale_fmt must be 'f16' or 'e4m3'")


def rotate_rows(X, R):
    """y = x · R for every row, computed in fp64 and rounded to fp32."""
    X64 = np.asarray(X, dtype=np.float64)
    R64 = np.asarray(R, dtype=np.float64)
    return (X64 @ R64).astype(np.float32)


def quantize_rows(Y, group_size, clip_ratio, scale_fmt="f16"):
    """Quantise fp32 rows Y (n×d) group-wise to INT2.

    Returns (codes uint8 n×d in {0..3}, scale float16 n×(d/G), zero float16
    n×(d/G)).  Steps, per group of G consecutive channels: min and max of the
    group, clipped by r; s = rnd((hi - lo)/3), z = rnd(lo) with rnd the fp16
    rounding (scale_fmt "f16") or the E4M3 rounding ("e4m3"; the values are
    returned in float16, which holds every E4M3 value exactly);
    c = clamp(rint((y - z)/s), 0, 3) in fp32; s == 0 gives c = 0.
    """
    Y = np.asarray(Y, dtype=np.float32)
    n, d = Y.shape
    G = int(group_size)
    if d % G != 0:
        raise ValueError("group size must divide d")
    ng = d // G
    Yg = Y.reshape(n, ng, G)
    r = np.float32(clip_ratio)
    mn = Yg.min(axis=2)
    mx = Yg.max(axis=2)
    lo = (r * mn).astype(np.float32)
    hi = (r * mx).astype(np.float32)
    s32 = ((hi - lo).astype(np.float32) / np.float32(3.0)).astype(np.float32)
    s16 = _round_scale(s32, scale_fmt)
    z16 = _round_scale(lo, scale_fmt)
    s_f = s16.astype(np.float32)[:, :, None]
    z_f = z16.astype(np.float32)[:, :, None]
    num = (Yg - z_f).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        u = (num / s_f).astype(np.float32)
    c = np.clip(np.rint(u), 0.0, 3.0)
    c = np.where(s_f == 0.0, 0.0, c)
    codes = c.astype(np.uint8).reshape(n, d)
    return codes, s16, z16


def dequantize_rows(codes, scale, zero):
    """ŷ = s·c + z per group, in fp64."""
    codes = np.asarray(codes)
    n, d = codes.shape
    ng = scale.shape[1]
    G = d // ng
    s = np.asarray(scale, dtype=np.float64)[:, :, None]
    z = np.asarray(zero, dtype=np.float64)[:, :, None]
    c = codes.reshape(n, ng, G).astype(np.float64)
    return (s * c + z).reshape(n, d)


def pack_codes(codes):
    """Pack 2-bit codes (…×d) into bytes (…×d/4): channel j -> bits 2(j%4) of byte j//4."""
    codes = np.asarray(codes, dtype=np.uint8)
    d = codes.shape[-1]
    c = codes.reshape(codes.shape[:-1] + (d // 4, 4)).astype(np.uint16)
    b = c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)
    return b.astype(np.uint8)


def unpack_codes(packed):
    """Inverse of pack_codes."""
    packed = np.asarray(packed, dtype=np.uint8)
    parts = [(packed >> (2 * k)) & 3 for k in range(4)]
    out = np.stack(parts, axis=-1)
    return out.reshape(packed.shape[:-1] + (packed.shape[-1] * 4,)).astype(np.uint8)


def record_layout(d, group_size, scale_fmt="f16"):
    """Byte offsets inside one (slot, KV head) record.

    [K codes d/4][V codes d/4][K (s, z) pairs × d/G][V (s, z) × d/G]: fp16
    pairs (4 bytes) padded to a multiple of 16 bytes, or E4M3 pairs (2 bytes)
    padded to a multiple of 8 bytes.
    """
    ng = d // group_size
    pb = 4 if scale_fmt == "f16" else 2
    off_kc = 0
    off_vc = d // 4
    off_ks = d // 2
    off_vs = d // 2 + pb * ng
    raw = d // 2 + 2 * pb * ng
    al = 16 if scale_fmt == "f16" else 8
    rec = (raw + al - 1) // al * al
    return dict(k_codes=off_kc, v_codes=off_vc, k_sz=off_ks, v_sz=off_vs,
                bytes=rec, groups=ng, pair_bytes=pb)


def slot_bytes(d, group_size, num_kv_heads, scale_fmt="f16"):
    """Bytes of one pool slot: the records of all KV heads back to back
    (head h at h·record bytes), padded to a multiple of 16 bytes."""
    raw = num_kv_heads * record_layout(d, group_size, scale_fmt)["bytes"]
    return (raw + 15) // 16 * 16


def pack_slots(recs, slot_size):
    """(…, Hkv, rec) per-head records -> (…, slot_size) slot bytes (zero padded)."""
    recs = np.asarray(recs, dtype=np.uint8)
    flat = recs.reshape(recs.shape[:-2] + (recs.shape[-2] * recs.shape[-1],))
    out = np.zeros(recs.shape[:-2] + (slot_size,), np.uint8)
    out[..., :flat.shape[-1]] = flat
    return out


def head_records(slots, num_kv_heads, rec_size):
    """(…, slot_size) slot bytes -> (…, Hkv, rec) per-head records (a copy)."""
    slots = np.asarray(slots, dtype=np.uint8)
    n = num_kv_heads * rec_size
    return np.ascontiguousarray(slots[..., :n]).reshape(slots.shape[:-1] + (num_kv_heads, rec_size))


def pack_record(kc, ks, kz, vc, vs, vz, d, group_size, scale_fmt="f16"):
    """Serialise one or many (slot, head) records to bytes (…×rec_bytes)."""
    lay = record_layout(d, group_size, scale_fmt)
    lead = np.asarray(kc).shape[:-1]
    out = np.zeros(lead + (lay["bytes"],), dtype=np.uint8)
    out[..., lay["k_codes"]:lay["k_codes"] + d // 4] = pack_codes(kc)
    out[..., lay["v_codes"]:lay["v_codes"] + d // 4] = pack_codes(vc)
    ng = lay["groups"]

    pb = lay["pair_bytes"]

    def sz_bytes(s, z):
        if scale_fmt == "f16":
            pair = np.stack([np.asarray(s, np.float16), np.asarray(z, np.float16)], axis=-1)
            return np.ascontiguousarray(pair).view(np.uint8).reshape(lead + (4 * ng,))
        pair = np.stack([e4m3_bits(s), e4m3_bits(z)], axis=-1)
        return np.ascontiguousarray(pair).reshape(lead + (2 * ng,))

    out[..., lay["k_sz"]:lay["k_sz"] + pb * ng] = sz_bytes(ks, kz)
    out[..., lay["v_sz"]:lay["v_sz"] + pb * ng] = sz_bytes(vs, vz)
    return out


def unpack_record(rec, d, group_size, scale_fmt="f16"):
    """Inverse of pack_record: returns (kc, ks, kz, vc, vs, vz)."""
    lay = record_layout(d, group_size, scale_fmt)
    rec = np.asarray(rec, dtype=np.uint8)
    lead = rec.shape[:-1]
    ng = lay["groups"]
    kc = unpack_codes(rec[..., lay["k_codes"]:lay["k_codes"] + d // 4])
    vc = unpack_codes(rec[..., lay["v_codes"]:lay["v_codes"] + d // 4])

    def sz(off):
        if scale_fmt == "f16":
            raw = np.ascontiguousarray(rec[..., off:off + 4 * ng])
            pair = raw.view(np.float16).reshape(lead + (ng, 2))
            return pair[..., 0].copy(), pair[..., 1].copy()
        raw = np.ascontiguousarray(rec[..., off:off + 2 * ng]).reshape(lead + (ng, 2))
        return (e4m3_from_bits(raw[..., 0]).astype(np.float16),
                e4m3_from_bits(raw[..., 1]).astype(np.float16))

    ks, kz = sz(lay["k_sz"])
    vs, vz = sz(lay["v_sz"])
    return kc, ks, kz, vc, vs, vz
