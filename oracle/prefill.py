"""Chunked-prefill attention over the mixed-precision cache, exact softmax, fp64.

Test infrastructure only (see the package docstring).

[Prefix log] "KVプールが上限だった — hybrid GDN の長文キャッシュ…": when a long
prompt is prefilled in chunks, each chunk's queries attend over the prefix
already cached in INT2; the integration described there first expands that
prefix to fp16 in a workspace that grows with the sequence
(dequantize_prefix_kv), then runs ordinary attention.  The quantity computed
is the same without the workspace:

* for query i of the chunk (position p = L0 + i of a request that held L0
  tokens before the chunk), the keys are the cached prefix as stored -- sink
  and recent windows in BF16 (unrotated), history in INT2 in the rotated
  domain (logit against q·R_K, value sum mapped back with R_Vᵀ), exactly as
  in decode attention at length L0 -- followed by the chunk's own keys at
  positions L0 .. p (causal);
* the chunk's own keys and values enter at bf16 (the storage type of the
  windows) and unrotated;
* one softmax over all of them, scale 1/sqrt(d); query head h reads KV head
  h // (Hq / Hkv).

Reading: the chunk attends over the cache as it stands before the chunk is
appended (the page's dequantised workspace holds the prefix; the chunk's own
K/V come fresh from the projection), so none of the chunk's tokens is
quantised for its own attention.
"""

import numpy as np

from .attention import _request_parts
from .quant import bf16_round


def prefill_attention(cache, q, k, v, page_table, L0, rq, b=0, heads=None):
    """Attention of one request's prefill chunk.

    q: (C, Hq, d) queries of positions L0 .. L0+C-1; k, v: (C, Hkv, d) the
    chunk's keys and values (rounded to bf16 here); page_table row b holds the
    slots of the cached prefix; rq: window row.  heads: optional query heads to
    evaluate (others NaN).  Returns (C, Hq, d) fp64.
    """
    cfg = cache.cfg
    d = cfg.head_dim
    g = cfg.gqa
    q = np.asarray(q, dtype=np.float64)
    C, Hq, _ = q.shape
    kc = bf16_round(np.asarray(k, dtype=np.float32)).astype(np.float64)
    vc = bf16_round(np.asarray(v, dtype=np.float32)).astype(np.float64)
    out = np.full((C, Hq, d), np.nan)
    scale = 1.0 / np.sqrt(d)
    causal = np.tril(np.ones((C, C), dtype=bool))
    for h in (range(Hq) if heads is None else heads):
        kvh = h // g
        Kp, Vp, Kh, Vh = _request_parts(cache, b, L0, rq, page_table, kvh) if L0 > 0 else (
            np.zeros((0, d)), np.zeros((0, d)), np.zeros((0, d)), np.zeros((0, d)))
        Q = q[:, h, :]
        lp = (Q @ Kp.T) * scale                          # (C, n_bf16)
        lh = (Q @ cache.rot_k @ Kh.T) * scale            # (C, n_hist)
        lc = np.where(causal, (Q @ kc[:, kvh, :].T) * scale, -np.inf)
        m = np.maximum(np.maximum(lp.max(axis=1, initial=-np.inf), lh.max(axis=1, initial=-np.inf)),
                       lc.max(axis=1))
        ep = np.exp(lp - m[:, None])
        eh = np.exp(lh - m[:, None])
        ec = np.exp(lc - m[:, None])
        den = ep.sum(axis=1) + eh.sum(axis=1) + ec.sum(axis=1)
        num = ep @ Vp + ec @ vc[:, kvh, :] + (eh @ Vh) @ cache.rot_v.T
        out[:, h, :] = num / den[:, None]
    return out
