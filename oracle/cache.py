"""The three-region mixed-precision KV cache and its append semantics (fp64 model).

Test infrastructure only (see the package docstring).

[OSCAR news] "サービングシステム：混合精度キャッシュレイアウト": per request, the
first 64 tokens (sink) and the last 256 tokens before the current position
(recent) are kept in BF16; every token in between (history) is stored in
INT2 after the OSCAR rotation and clipping.  [Scheduler log]: the page table
is token-granular (page_size 1), so every position p of a request owns one
slot page_table[b][p] of a global token pool.

Region boundaries for a request holding L tokens (S = sink, W = recent):
  sink    [0, min(S, L))
  history [S, max(S, L - W))
  recent  [max(S, L - W), L)
(the current token is inside the recent window; L <= S + W means no history).

Append of tokens [L0, L1) (reading of the pages, which describe the layout
but not the update):
  1. every position in [hist_hi(L0), hist_hi(L1)) enters the history: those
     below L0 leave the recent window and are read from the BF16 ring, those
     at or above L0 come from the new input; each is rotated, clipped,
     quantised and written to its slot;
  2. then new positions below S are written to the sink, and new positions at
     or above hist_hi(L1) to the recent ring at index p mod W.
"""

from dataclasses import dataclass

import numpy as np

from .quant import (bf16_round, bf16_bits, rotate_rows, quantize_rows,
                    dequantize_rows, pack_record, record_layout, slot_bytes, pack_slots)


@dataclass
class OracleConfig:
    head_dim: int
    num_q_heads: int
    num_kv_heads: int
    group_size: int
    sink: int = 64
    recent: int = 256
    clip_ratio: float = 0.9
    scale_fmt: str = "f16"          # "f16" or "e4m3" (s, z) storage

    @property
    def gqa(self):
        return self.num_q_heads // self.num_kv_heads

    @property
    def groups(self):
        return self.head_dim // self.group_size


def regions(L, S, W):
    """(sink_end, hist_lo, hist_hi, recent_lo, recent_hi) for a request of L tokens."""
    hist_hi = max(S, L - W)
    return min(S, L), S, hist_hi, hist_hi, L


class OracleCache:
    """Cache state: INT2 records per (slot, KV head) and BF16 windows per request."""

    def __init__(self, cfg, num_slots, max_reqs, rot_k, rot_v):
        self.cfg = cfg
        d, H, ng = cfg.head_dim, cfg.num_kv_heads, cfg.groups
        self.num_slots = num_slots
        self.max_reqs = max_reqs
        self.rot_k = np.asarray(rot_k, dtype=np.float64)
        self.rot_v = np.asarray(rot_v, dtype=np.float64)
        self.kc = np.zeros((num_slots, H, d), np.uint8)
        self.vc = np.zeros((num_slots, H, d), np.uint8)
        self.ks = np.zeros((num_slots, H, ng), np.float16)
        self.kz = np.zeros((num_slots, H, ng), np.float16)
        self.vs = np.zeros((num_slots, H, ng), np.float16)
        self.vz = np.zeros((num_slots, H, ng), np.float16)
        # unrotated (pre-quantisation) fp32 rotated rows, kept for diagnostics
        self.ky = {}
        self.vy = {}
        self.sink = np.zeros((max_reqs, cfg.sink, H, 2, d), np.float32)
        self.ring = np.zeros((max_reqs, cfg.recent, H, 2, d), np.float32)

    # -- append -----------------------------------------------------------
    def _quantize_into(self, slots, Xk, Xv, keep_y=False):
        cfg = self.cfg
        n = len(slots)
        if n == 0:
            return
        d, H = cfg.head_dim, cfg.num_kv_heads
        Yk = rotate_rows(Xk.reshape(n * H, d), self.rot_k)
        Yv = rotate_rows(Xv.reshape(n * H, d), self.rot_v)
        kc, ks, kz = quantize_rows(Yk, cfg.group_size, cfg.clip_ratio, cfg.scale_fmt)
        vc, vs, vz = quantize_rows(Yv, cfg.group_size, cfg.clip_ratio, cfg.scale_fmt)
        ng = cfg.groups
        self.kc[slots] = kc.reshape(n, H, d)
        self.vc[slots] = vc.reshape(n, H, d)
        self.ks[slots] = ks.reshape(n, H, ng)
        self.kz[slots] = kz.reshape(n, H, ng)
        self.vs[slots] = vs.reshape(n, H, ng)
        self.vz[slots] = vz.reshape(n, H, ng)
        if keep_y:
            Yk = Yk.reshape(n, H, d)
            Yv = Yv.reshape(n, H, d)
            for i, s in enumerate(slots):
                self.ky[int(s)] = Yk[i]
                self.vy[int(s)] = Yv[i]

    def append(self, k, v, cu_new, start_pos, req_idx, page_table, keep_y=False):
        """Append new tokens for a batch of requests.

        k, v: (T_total, Hkv, d) float arrays (fp32 or bf16-exact values);
        cu_new: (B+1,) prefix offsets of each request's new rows;
        start_pos: (B,) tokens already cached (L0); req_idx: (B,) window row;
        page_table: (B, >= L1) slot of every position.
        """
        cfg = self.cfg
        S, W = cfg.sink, cfg.recent
        k = np.asarray(k)
        v = np.asarray(v)
        B = len(start_pos)
        for b in range(B):
            c0, c1 = int(cu_new[b]), int(cu_new[b + 1])
            L0 = int(start_pos[b])
            L1 = L0 + (c1 - c0)
            rq = int(req_idx[b])
            xk = bf16_round(k[c0:c1])
            xv = bf16_round(v[c0:c1])
            lo = max(S, L0 - W)
            hi = max(S, L1 - W)
            pos = np.arange(lo, hi)
            if len(pos):
                Xk = np.empty((len(pos),) + xk.shape[1:], np.float32)
                Xv = np.empty_like(Xk)
                old = pos < L0
                if old.any():
                    Xk[old] = self.ring[rq, pos[old] % W, :, 0, :]
                    Xv[old] = self.ring[rq, pos[old] % W, :, 1, :]
                new = ~old
                if new.any():
                    Xk[new] = xk[pos[new] - L0]
                    Xv[new] = xv[pos[new] - L0]
                slots = np.asarray(page_table[b][pos], dtype=np.int64)
                self._quantize_into(slots, Xk, Xv, keep_y)
            for p in range(L0, L1):
                if p < S:
                    self.sink[rq, p, :, 0, :] = xk[p - L0]
                    self.sink[rq, p, :, 1, :] = xv[p - L0]
                elif p >= hi:
                    self.ring[rq, p % W, :, 0, :] = xk[p - L0]
                    self.ring[rq, p % W, :, 1, :] = xv[p - L0]

    # -- views --------------------------------------------------------------
    def dequant_k(self, slots, h):
        return dequantize_rows(self.kc[slots, h], self.ks[slots, h], self.kz[slots, h])

    def dequant_v(self, slots, h):
        return dequantize_rows(self.vc[slots, h], self.vs[slots, h], self.vz[slots, h])

    def records(self):
        """Per-head records of the INT2 pool: (num_slots, Hkv, rec_bytes) uint8."""
        cfg = self.cfg
        return pack_record(self.kc, self.ks, self.kz, self.vc, self.vs, self.vz,
                           cfg.head_dim, cfg.group_size, cfg.scale_fmt)

    def slot_records(self):
        """Device byte layout of the INT2 pool: (num_slots, slot_bytes) uint8,
        the records of all KV heads of a slot back to back, padded to 16 bytes."""
        cfg = self.cfg
        return pack_slots(self.records(), self.slot_bytes())

    def slot_bytes(self):
        cfg = self.cfg
        return slot_bytes(cfg.head_dim, cfg.group_size, cfg.num_kv_heads, cfg.scale_fmt)

    def window_bits(self):
        """Device layout of the BF16 windows: (sink bits, recent bits), uint16."""
        return bf16_bits(self.sink), bf16_bits(self.ring)

    def record_bytes(self):
        return record_layout(self.cfg.head_dim, self.cfg.group_size, self.cfg.scale_fmt)["bytes"]
