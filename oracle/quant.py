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
* the code is decided in fp32 from the fp16-rounded s and z:
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


def rotate_rows(X, R):
    """y = x · R for every row, computed in fp64 and rounded to fp32."""
    X64 = np.asarray(X, dtype=np.float64)
    R64 = np.asarray(R, dtype=np.float64)
    return (X64 @ R64).astype(np.float32)


def quantize_rows(Y, group_size, clip_ratio):
    """Quantise fp32 rows Y (n×d) group-wise to INT2.

    Returns (codes uint8 n×d in {0..3}, scale float16 n×(d/G), zero float16
    n×(d/G)).  Steps, per group of G consecutive channels: min and max of the
    group, clipped by r; s = fp16((hi - lo)/3), z = fp16(lo);
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
    s16 = s32.astype(np.float16)
    z16 = lo.astype(np.float16)
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


def record_layout(d, group_size):
    """Byte offsets inside one (slot, KV head) record.

    [K codes d/4][V codes d/4][K (s, z) fp16 pairs × d/G][V (s, z) × d/G],
    padded to a multiple of 16 bytes.
    """
    ng = d // group_size
    off_kc = 0
    off_vc = d // 4
    off_ks = d // 2
    off_vs = d // 2 + 4 * ng
    raw = d // 2 + 8 * ng
    rec = (raw + 15) // 16 * 16
    return dict(k_codes=off_kc, v_codes=off_vc, k_sz=off_ks, v_sz=off_vs,
                bytes=rec, groups=ng)


def pack_record(kc, ks, kz, vc, vs, vz, d, group_size):
    """Serialise one or many (slot, head) records to bytes (…×rec_bytes)."""
    lay = record_layout(d, group_size)
    lead = np.asarray(kc).shape[:-1]
    out = np.zeros(lead + (lay["bytes"],), dtype=np.uint8)
    out[..., lay["k_codes"]:lay["k_codes"] + d // 4] = pack_codes(kc)
    out[..., lay["v_codes"]:lay["v_codes"] + d // 4] = pack_codes(vc)
    ng = lay["groups"]

    def sz_bytes(s, z):
        pair = np.stack([np.asarray(s, np.float16), np.asarray(z, np.float16)], axis=-1)
        return np.ascontiguousarray(pair).view(np.uint8).reshape(lead + (4 * ng,))

    out[..., lay["k_sz"]:lay["k_sz"] + 4 * ng] = sz_bytes(ks, kz)
    out[..., lay["v_sz"]:lay["v_sz"] + 4 * ng] = sz_bytes(vs, vz)
    return out


def unpack_record(rec, d, group_size):
    """Inverse of pack_record: returns (kc, ks, kz, vc, vs, vz)."""
    lay = record_layout(d, group_size)
    rec = np.asarray(rec, dtype=np.uint8)
    lead = rec.shape[:-1]
    ng = lay["groups"]
    kc = unpack_codes(rec[..., lay["k_codes"]:lay["k_codes"] + d // 4])
    vc = unpack_codes(rec[..., lay["v_codes"]:lay["v_codes"] + d // 4])

    def sz(off):
        raw = np.ascontiguousarray(rec[..., off:off + 4 * ng])
        pair = raw.view(np.float16).reshape(lead + (ng, 2))
        return pair[..., 0].copy(), pair[..., 1].copy()

    ks, kz = sz(lay["k_sz"])
    vs, vz = sz(lay["v_sz"])
    return kc, ks, kz, vc, vs, vz
