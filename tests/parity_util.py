"""Helpers for the GPU parity tests: moving an oracle cache to the device,
and classifying INT2 record mismatches against the acceptance rule

    codes are bit-exact except where the oracle's pre-rounding value
    u = (y - z)/s lies within 1e-6·max(1, |u|) of a rounding boundary, and
    (s, z) are exact except where the fp32 value rounded to fp16 (or to E4M3
    for one-byte scales) lies within 1e-6 relative of a rounding tie of that
    format (all codes of such a group excused).

Both kinds of boundary case are counted; `record_boundary_cases` keeps the
counts of a test so that the session summary reports them.
"""

import numpy as np
import torch

import oracle
from oracle import quant as oq

REL_TIE = 1e-6


def fp16_near_tie(x, band=0.0):
    """True where fp32 x is within REL_TIE (relative), or within the absolute
    `band`, of a midpoint between fp16 neighbours."""
    x = np.asarray(x, np.float32)
    h = x.astype(np.float16)
    up = np.nextafter(h, np.float16(np.inf)).astype(np.float32)
    dn = np.nextafter(h, np.float16(-np.inf)).astype(np.float32)
    hf = h.astype(np.float32)
    mid = np.where(x >= hf, (hf + up) / 2, (hf + dn) / 2)
    return np.abs(x.astype(np.float64) - mid) <= np.maximum(REL_TIE * np.maximum(np.abs(x), 1e-30), band)


_E4M3_GRID = None


def e4m3_near_tie(x, band=0.0):
    """True where fp32 x is within REL_TIE (relative), or within the absolute
    `band`, of a midpoint between E4M3 neighbours.  Beyond ±448 every value
    saturates to ±448, so there is no tie there."""
    global _E4M3_GRID
    if _E4M3_GRID is None:
        b = np.array([i for i in range(256) if (i & 0x7F) != 0x7F], np.uint8)
        _E4M3_GRID = np.unique(oq.e4m3_from_bits(b).astype(np.float64))
    g = _E4M3_GRID
    x = np.atleast_1d(np.asarray(x, np.float32)).astype(np.float64)
    i = np.clip(np.searchsorted(g, x), 1, len(g) - 1)
    mid = (g[i - 1] + g[i]) / 2
    inside = (x >= g[0]) & (x <= g[-1])
    return inside & (np.abs(x - mid) <= np.maximum(REL_TIE * np.maximum(np.abs(x), 1e-30), band))


def classify_records(gpu_rec, ora_cache, slots, ora_y=None):
    """Compare GPU records with the oracle's for the given slots (all heads).

    Returns dict(exact, code_ties, sz_ties, bad) counted over
    (slot, head, K|V, group).
    `ora_y` (optional): dict slot -> (ky (Hkv, d), vy (Hkv, d)) fp32 rotated rows of the oracle.
    """
    cfg = ora_cache.cfg
    d, G, H = cfg.head_dim, cfg.group_size, cfg.num_kv_heads
    fmt = cfg.scale_fmt
    near_tie = e4m3_near_tie if fmt == "e4m3" else fp16_near_tie
    ng = d // G
    r = np.float32(cfg.clip_ratio)
    slots = np.asarray(slots, dtype=np.int64)
    want = ora_cache.records()[slots]
    got = np.asarray(gpu_rec)[slots]
    if got.ndim == 2:                      # slot layout (E4M3): per-head records
        got = oq.head_records(got, H, ora_cache.record_bytes())
    stats = dict(exact=0, code_ties=0, sz_ties=0, bad=0, bad_examples=[])
    diff = (want != got).any(axis=-1)               # (n, H)
    stats["exact"] = int((~diff).sum()) * 2 * ng
    for i, h in zip(*np.nonzero(diff)):
        s = int(slots[i])
        gk = oq.unpack_record(got[i, h], d, G, fmt)
        wk = oq.unpack_record(want[i, h], d, G, fmt)
        for mat in (0, 1):
            gc, gs, gz = gk[3 * mat: 3 * mat + 3]
            wc, ws, wz = wk[3 * mat: 3 * mat + 3]
            y = None
            if ora_y is not None:
                y = ora_y[s][mat][h]
            elif s in (ora_cache.ky if mat == 0 else ora_cache.vy):
                y = (ora_cache.ky if mat == 0 else ora_cache.vy)[s][h]
            for gi in range(ng):
                sl = slice(gi * G, (gi + 1) * G)
                same_sz = gs[gi] == ws[gi] and gz[gi] == wz[gi]
                if same_sz and np.array_equal(gc[sl], wc[sl]):
                    stats["exact"] += 1
                    continue
                if y is None:
                    stats["bad"] += 1
                    continue
                yg = y[sl].astype(np.float32)
                lo = np.float32(r * yg.min())
                hi = np.float32(r * yg.max())
                s32 = np.float32(np.float32(hi - lo) / np.float32(3.0))
                if not same_sz:
                    if near_tie(s32) or near_tie(lo):
                        stats["sz_ties"] += 1
                        continue
                    stats["bad"] += 1
                    stats["bad_examples"].append(("sz", s, int(h), mat, gi))
                    continue
                sf = np.float32(ws[gi])
                zf = np.float32(wz[gi])
                u = (np.float32(yg - zf) / sf).astype(np.float32)
                bad_here = False
                for j in np.nonzero(gc[sl] != wc[sl])[0]:
                    uj = float(u[j])
                    near = min(abs(uj - (k + 0.5)) for k in range(3))
                    if near > REL_TIE * max(1.0, abs(uj)):
                        bad_here = True
                if bad_here:
                    stats["bad"] += 1
                    stats["bad_examples"].append(("code", s, int(h), mat, gi))
                else:
                    stats["code_ties"] += 1
    return stats


def device_cache_from_oracle(ops, ocache, cfg, device="cuda"):
    """A LayerCache holding exactly the oracle cache's records and windows."""
    dc = ops.LayerCache(cfg, ocache.num_slots, ocache.max_reqs, ocache.rot_k.astype(np.float32),
                        ocache.rot_v.astype(np.float32), device=device)
    rec = ocache.records() if dc.records.dim() == 3 else ocache.slot_records()
    dc.records.copy_(torch.from_numpy(rec))
    sink_bits, ring_bits = ocache.window_bits()
    if cfg.sink > 0:
        dc.sink.copy_(torch.from_numpy(sink_bits.view(np.int16)).view(torch.bfloat16))
    dc.recent.copy_(torch.from_numpy(ring_bits.view(np.int16)).view(torch.bfloat16))
    return dc


def attn_errors(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    err = float(np.abs(got - want).max())
    rel = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))
    return err, rel


ATOL = 2e-3      # max-abs bound on attention outputs
RTOL_L2 = 1e-3   # relative-L2 bound on attention outputs


# Boundary-case counts of the tests in this session: (test, code ties, (s, z) ties, records compared).
BOUNDARY_CASES = []


def record_boundary_cases(name, stats, n_records):
    """Keeps the tie counts of one comparison for the session summary."""
    BOUNDARY_CASES.append((name, int(stats.get("code_ties", 0)), int(stats.get("sz_ties", 0)), int(n_records)))
