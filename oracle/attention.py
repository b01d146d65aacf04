"""Decode attention over the mixed-precision cache, exact softmax, fp64.

Test infrastructure only (see the package docstring).

For a request holding L tokens and query q (one vector per query head):
* sink and recent tokens are BF16 and unrotated: logit = q·k / sqrt(d);
* history tokens are INT2 in the rotated domain: k̂ = s·c + z, and since R_K
  is orthogonal, q·k ≈ (q R_K)·k̂ ([OSCAR news] "OSCARの違い": the rotation is
  applied before quantisation, so the logit is taken against the rotated key);
* one softmax over all L logits;
* output = Σ_bf16 p·v + (Σ_hist p·v̂) · R_Vᵀ (the value rotation is undone once,
  after the weighted sum).
Query head h reads KV head h // (Hq / Hkv): [Escha log] fix 4 describes the
silent bug when a block of query heads straddles two KV heads; the mapping
below is the one that bug violated.
Readings: softmax scale 1/sqrt(d); positional encoding is the caller's job.
"""

import numpy as np

from .cache import regions


def _request_parts(cache, b, L, rq, page_table, kvh):
    cfg = cache.cfg
    S, W = cfg.sink, cfg.recent
    sink_end, hist_lo, hist_hi, rec_lo, rec_hi = regions(L, S, W)
    Kp = [cache.sink[rq, :sink_end, kvh, 0, :].astype(np.float64)]
    Vp = [cache.sink[rq, :sink_end, kvh, 1, :].astype(np.float64)]
    pos = np.arange(rec_lo, rec_hi)
    Kp.append(cache.ring[rq, pos % W, kvh, 0, :].astype(np.float64))
    Vp.append(cache.ring[rq, pos % W, kvh, 1, :].astype(np.float64))
    Kp = np.concatenate(Kp, axis=0)
    Vp = np.concatenate(Vp, axis=0)
    slots = np.asarray(page_table[b][hist_lo:hist_hi], dtype=np.int64)
    Kh = cache.dequant_k(slots, kvh)
    Vh = cache.dequant_v(slots, kvh)
    return Kp, Vp, Kh, Vh


def decode_attention(cache, q, page_table, seq_lens, req_idx, pairs=None):
    """Exact decode attention.  q: (B, Hq, d).  Returns (B, Hq, d) fp64.

    pairs: optional list of (b, query head) to evaluate; other outputs are NaN.
    """
    cfg = cache.cfg
    d = cfg.head_dim
    g = cfg.gqa
    q = np.asarray(q, dtype=np.float64)
    B, Hq, _ = q.shape
    out = np.full((B, Hq, d), np.nan)
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(Hq)]
    by_kv = {}
    for b, h in pairs:
        by_kv.setdefault((b, h // g), []).append(h)
    scale = 1.0 / np.sqrt(d)
    for (b, kvh), heads in by_kv.items():
        L = int(seq_lens[b])
        rq = int(req_idx[b])
        Kp, Vp, Kh, Vh = _request_parts(cache, b, L, rq, page_table, kvh)
        for h in heads:
            qv = q[b, h]
            qr = qv @ cache.rot_k
            lp = (Kp @ qv) * scale
            lh = (Kh @ qr) * scale
            m = max(lp.max(initial=-np.inf), lh.max(initial=-np.inf))
            ep = np.exp(lp - m)
            eh = np.exp(lh - m)
            den = ep.sum() + eh.sum()
            num = ep @ Vp + (eh @ Vh) @ cache.rot_v.T
            out[b, h] = num / den
    return out


def decode_attention_split(cache, q, page_table, seq_lens, req_idx, chunk):
    """Same result via split-K: per-chunk (m, l, o) partials merged by log-sum-exp.

    The history is cut into chunks of `chunk` tokens; the BF16 tokens form one
    more partial.  Merge: M = max_s m_s; o = Σ_s e^{m_s-M} o_s / Σ_s e^{m_s-M} l_s,
    with the rotated-domain partials summed before R_Vᵀ is applied once.
    """
    cfg = cache.cfg
    d = cfg.head_dim
    g = cfg.gqa
    q = np.asarray(q, dtype=np.float64)
    B, Hq, _ = q.shape
    out = np.zeros((B, Hq, d))
    scale = 1.0 / np.sqrt(d)
    for b in range(B):
        L = int(seq_lens[b])
        rq = int(req_idx[b])
        for h in range(Hq):
            kvh = h // g
            Kp, Vp, Kh, Vh = _request_parts(cache, b, L, rq, page_table, kvh)
            qv = q[b, h]
            qr = qv @ cache.rot_k
            parts = []  # (m, l, o, rotated?)
            if len(Kp):
                lp = (Kp @ qv) * scale
                m = lp.max()
                e = np.exp(lp - m)
                parts.append((m, e.sum(), e @ Vp, False))
            for c0 in range(0, len(Kh), chunk):
                lh = (Kh[c0:c0 + chunk] @ qr) * scale
                m = lh.max()
                e = np.exp(lh - m)
                parts.append((m, e.sum(), e @ Vh[c0:c0 + chunk], True))
            M = max(p[0] for p in parts)
            den = sum(np.exp(p[0] - M) * p[1] for p in parts)
            o_plain = sum((np.exp(p[0] - M) * p[2] for p in parts if not p[3]),
                          np.zeros(d))
            o_rot = sum((np.exp(p[0] - M) * p[2] for p in parts if p[3]),
                        np.zeros(d))
            out[b, h] = (o_plain + o_rot @ cache.rot_v.T) / den
    return out
