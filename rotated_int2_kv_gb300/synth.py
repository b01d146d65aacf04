"""Seeded synthetic inputs shaped like the workloads of the OSCAR pages.

This module only draws random numbers: it contains none of the method's
arithmetic (no rotation, quantisation, covariance or attention).  Tests feed
its outputs to both the CUDA library and the fp64 oracle; the bench feeds
them to the library and, on a small sample, to the oracle.

Recipe:
* K, V ~ N(0, 1) per element, with outlier channels: "fixed4" scales four
  seeded channels (the same in every KV head) by 20 in K and by 4 in V;
  "per_head" draws, per KV head, 2-8 K channels scaled by 10-30 (V keeps the
  fixed four channels scaled by 4).
* q ~ N(0, 1).
* calibration samples: 4096 rows x = z · diag(sqrt(λ)) · Qᵀ with
  λ_i ∝ i^-1.5 and Q a seeded random orthogonal matrix (a separate Q for the
  key side and the value side).
* page tables: a seeded permutation of a global token pool (page_size 1).
Token values are a pure function of (seed, request, position): they are
drawn in blocks of 1024 positions, each block from its own generator, so any
chunking of the appends sees the same values.
"""

import numpy as np
import torch

BLOCK = 1024
_MIX = 0x9E3779B97F4A7C15


def _sub_seed(*parts):
    h = 0x243F6A8885A308D3
    for p in parts:
        h = ((h ^ (int(p) & 0xFFFFFFFFFFFFFFFF)) * _MIX) & 0xFFFFFFFFFFFFFFFF
        h ^= h >> 29
    return h & 0x7FFFFFFFFFFFFFFF


def _gen(device, *parts):
    g = torch.Generator(device=device)
    g.manual_seed(_sub_seed(*parts))
    return g


def outlier_scales(seed, num_kv_heads, head_dim, mode="fixed4"):
    """Per-(KV head, channel) multipliers for K and V: two (Hkv, d) fp32 tensors."""
    rng = np.random.default_rng(_sub_seed(seed, 1))
    ks = np.ones((num_kv_heads, head_dim), np.float32)
    vs = np.ones((num_kv_heads, head_dim), np.float32)
    fixed = rng.choice(head_dim, size=4, replace=False)
    vs[:, fixed] = 4.0
    if mode == "fixed4":
        ks[:, fixed] = 20.0
    elif mode == "per_head":
        for h in range(num_kv_heads):
            n = int(rng.integers(2, 9))
            ch = rng.choice(head_dim, size=n, replace=False)
            ks[h, ch] = rng.uniform(10.0, 30.0, size=n).astype(np.float32)
    elif mode != "none":
        raise ValueError(mode)
    return torch.from_numpy(ks), torch.from_numpy(vs)


def kv_tokens(seed, req, p0, n, num_kv_heads, head_dim, scales, device="cpu",
              dtype=torch.bfloat16, shared=0.0):
    """K and V rows for positions [p0, p0+n) of request `req`: (n, Hkv, d) each.
    shared > 0 adds shared·base_h to every row of KV head h (base_h ~ N(0, 1),
    one per head, K and V, the same for every request and position), before the
    channel multipliers: rows that share one strong direction."""
    ks, vs = scales
    ks = ks.to(device)
    vs = vs.to(device)
    base = None
    if shared:
        base = torch.randn((2, num_kv_heads, head_dim), generator=_gen(device, seed, 5),
                           device=device, dtype=torch.float32) * float(shared)
    out_k = torch.empty((n, num_kv_heads, head_dim), dtype=dtype, device=device)
    out_v = torch.empty_like(out_k)
    if n == 0:
        return out_k, out_v
    b0 = p0 // BLOCK
    b1 = (p0 + n - 1) // BLOCK
    for blk in range(b0, b1 + 1):
        g = _gen(device, seed, 2, req, blk)
        raw = torch.randn((2, BLOCK, num_kv_heads, head_dim), generator=g,
                          device=device, dtype=torch.float32)
        lo = max(p0, blk * BLOCK)
        hi = min(p0 + n, (blk + 1) * BLOCK)
        sl = slice(lo - blk * BLOCK, hi - blk * BLOCK)
        rk, rv = raw[0, sl], raw[1, sl]
        if base is not None:
            rk = rk + base[0]
            rv = rv + base[1]
        out_k[lo - p0:hi - p0] = (rk * ks).to(dtype)
        out_v[lo - p0:hi - p0] = (rv * vs).to(dtype)
    return out_k, out_v


def queries(seed, step, batch, num_q_heads, head_dim, device="cpu",
            dtype=torch.bfloat16):
    """q ~ N(0, 1): (batch, Hq, d)."""
    g = _gen(device, seed, 3, step)
    q = torch.randn((batch, num_q_heads, head_dim), generator=g, device=device,
                    dtype=torch.float32)
    return q.to(dtype)


def calib_samples(seed, side, head_dim, n=4096, alpha=1.5):
    """Calibration rows (n, d) fp64 with power-law spectrum λ_i ∝ i^-alpha."""
    rng = np.random.default_rng(_sub_seed(seed, 4, side))
    A = rng.standard_normal((head_dim, head_dim))
    Q, Rr = np.linalg.qr(A)
    Q = Q * np.sign(np.diag(Rr))[None, :]
    lam = np.arange(1, head_dim + 1, dtype=np.float64) ** (-alpha)
    Z = rng.standard_normal((n, head_dim))
    return (Z * np.sqrt(lam)[None, :]) @ Q.T


def page_table(seed, batch, max_len, num_slots, shuffled=True):
    """(batch, max_len) int32 slot ids: a seeded permutation of the pool, or identity."""
    if batch * max_len > num_slots:
        raise ValueError("pool too small")
    if shuffled:
        g = torch.Generator()
        g.manual_seed(_sub_seed(seed, 5))
        perm = torch.randperm(num_slots, generator=g)[: batch * max_len]
    else:
        perm = torch.arange(batch * max_len)
    return perm.to(torch.int32).reshape(batch, max_len)


def ragged_lengths(seed, batch, lo, hi):
    """Sequence lengths uniform in [lo, hi]."""
    rng = np.random.default_rng(_sub_seed(seed, 6))
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)
