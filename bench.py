"""Benchmark of the OSCAR-style rotated INT2 KV hot path on GB300.

Workload (one GPU): Qwen3-8B-shaped layer, 32 query / 8 KV heads, head_dim
128, group 64, clip 0.9, batch 32, every sequence at 100,000 tokens (64 BF16
sink + 99,680 INT2 history + 256 BF16 recent) with a token-granular page
table shuffled over a pool of 32 × 100,100+ slots.  A step is one decode step
of the hot path: oscar_quantize_append of one new token per request (the
token leaving the recent window spills into INT2) followed by
oscar_decode_attention.  Steps cycle through the 100-step decode sequence
(L = 100,001 … 100,100).  Inputs are seeded synthetic data (no model weights).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own batch
of 32 requests on its own GPU (requests are independent: weak scaling, no
collective on the data path); `value` aggregates over ranks.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV tokens/s & HBM GB/s (% of ~8 TB/s) at 100K ctx; append GB/s"
UNIT = "KV tokens/s"
SEED = 1234

B, HQ, HKV, D, G = 32, 32, 8, 128, 64
L_BASE = 100_000          # tokens cached before the first decode step
LB = np.full(B, L_BASE, dtype=np.int64)   # per-request cached tokens; uniform unless a workload sets it
OUTLIERS = "fixed4"       # K/V outlier-channel recipe of the synthetic inputs
SCALE_FMT = "f16"         # storage of each group's (s, z): fp16 or E4M3 pairs
CYCLE = 100               # decode steps of the sequence
S_SINK, W_RECENT = 64, 256


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-kernel", choices=["auto", "simt"], default="auto")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-append", action="store_true")
    ap.add_argument("--no-shapes", dest="shapes", action="store_false",
                    help="skip the ragged GQA-8 / wide GQA-6 decode shapes and the prefill chunks of the default line")
    ap.add_argument("--workload", choices=["qwen8b-100k", "qwen8b-100k-e4m3", "mid", "small", "b1-32k",
                                           "qwen32b-ragged", "gqa6-wide"],
                    default="qwen8b-100k",
                    help="qwen8b-100k-e4m3: the default shape with one-byte (E4M3) scale and zero; "
                         "small: batch 4 at 65,536 tokens (168 MB of INT2 records, > L2), for ncu captures; "
                         "mid: batch 8 at 100,000 tokens (0.51 GB); b1-32k: one request at 32,768 tokens "
                         "(launch-bound); qwen32b-ragged: 64 q / 8 KV heads, batch 8, lengths uniform in "
                         "[65,536, 131,072], per-head K outliers, 50-step cycle; gqa6-wide: 24 q / 4 KV heads, "
                         "d 256, group 128, batch 5 at 112,000 tokens")
    ap.add_argument("--prefill-only", choices=["qwen8b", "gqa6-wide"], default=None,
                    help="time only the prefill attention of one request (shape qwen8b: 32 q / 8 KV heads, d 128; "
                         "gqa6-wide: 24 q / 4 KV heads, d 256) and print its measurement; --steps is the number "
                         "of timed calls")
    ap.add_argument("--calibration-only", action="store_true",
                    help="time only the calibration statistics on the device (C_Q and C_S) and print them")
    ap.add_argument("--prefill-prefix", type=int, default=32768, help="cached prefix of --prefill-only, tokens")
    ap.add_argument("--prefill-chunk", type=int, default=8192, help="queries of --prefill-only's chunk")
    return ap.parse_args()


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------
REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 4:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                bits = int(parts[3], 16)
            except ValueError:
                continue
            for bit, name in REASON_BITS.items():
                if bits & bit:
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# distributed plumbing (one process per GPU; barrier + max over ranks only)
# --------------------------------------------------------------------------
def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_throughput(units, ms, ws):
    """Whole-job rate: the units all ranks processed over the slowest rank's time.

    Returns (units per second, max-over-ranks milliseconds)."""
    ms_max = max_over_ranks(ms, ws)
    return sum_over_ranks(units, ws) / (ms_max / 1e3), ms_max


# --------------------------------------------------------------------------
# workload
# --------------------------------------------------------------------------
def rotations(d):
    from rotated_int2_kv_gb300 import ops, synth
    Ck = ops.covariance(synth.calib_samples(SEED, 0, d))
    Cv = ops.covariance(synth.calib_samples(SEED, 1, d))
    Rk, _, _ = ops.build_rotation(Ck, d)
    Rv, _, _ = ops.build_rotation(Cv, d)
    return Rk, Rv


def build_decode_workload(rank, steps_total):
    import torch
    from rotated_int2_kv_gb300 import ops, synth
    dev = torch.device("cuda")
    seed = SEED + 7919 * rank
    cfg = ops.Config(D, HQ, HKV, G, S_SINK, W_RECENT, 0.9, scale_fmt=SCALE_FMT)
    Rk, Rv = rotations(D)
    max_len = int(LB.max()) + CYCLE
    pool = B * max_len
    pt = synth.page_table(seed, B, max_len, pool).to(dev)
    cache = ops.LayerCache(cfg, pool, B, Rk, Rv, device=dev)
    scales = synth.outlier_scales(seed, HKV, D, OUTLIERS)
    # fill request b to LB[b] tokens with chunked appends (rounds of up to 8,192
    # tokens per request; a request that is full takes no tokens)
    chunk = 8192
    pos = 0
    while pos < int(LB.max()):
        n = np.clip(LB - pos, 0, chunk)
        kk, vv = [], []
        for b in range(B):
            k, v = synth.kv_tokens(seed, b, pos, int(n[b]), HKV, D, scales, device=dev)
            kk.append(k)
            vv.append(v)
        k = torch.cat(kk)
        v = torch.cat(vv)
        cu = torch.from_numpy(np.concatenate([[0], np.cumsum(n)]).astype(np.int32)).to(dev)
        start = torch.from_numpy(np.minimum(LB, pos).astype(np.int32)).to(dev)
        ops.quantize_append(cache, k, v, cu, start, pt)
        pos += chunk
        del k, v, kk, vv
    torch.cuda.synchronize()
    # per-step inputs of the decode cycle (device-resident)
    newk, newv, qs = [], [], []
    for s in range(CYCLE):
        kk, vv = zip(*[synth.kv_tokens(seed, b, int(LB[b]) + s, 1, HKV, D, scales, device=dev) for b in range(B)])
        newk.append(torch.cat(kk))
        newv.append(torch.cat(vv))
        qs.append(synth.queries(seed, s, B, HQ, D, device=dev))
    starts = [torch.from_numpy((LB + s).astype(np.int32)).to(dev) for s in range(CYCLE)]
    lens = [torch.from_numpy((LB + s + 1).astype(np.int32)).to(dev) for s in range(CYCLE)]
    cu1 = torch.arange(0, B + 1, dtype=torch.int32, device=dev)
    ws = ops.alloc_workspace(cfg, B, max_len, device=dev)
    out = torch.empty((B, HQ, D), dtype=torch.float32, device=dev)
    return dict(cfg=cfg, cache=cache, pt=pt, newk=newk, newv=newv, qs=qs, starts=starts, lens=lens, cu1=cu1,
                ws=ws, out=out, max_len=max_len, Rk=Rk, Rv=Rv, seed=seed, scales=scales)


def decode_step(w, i, kernel):
    """One decode step: the fused call (oscar_decode_step) for the default
    kernels; the append and decode calls for the CUDA-core history path."""
    from rotated_int2_kv_gb300 import ops
    s = i % CYCLE
    if kernel == "auto":
        ops.decode_step(w["cache"], w["newk"][s], w["newv"][s], w["qs"][s], w["pt"], w["lens"][s], w["max_len"],
                        w["ws"], out=w["out"])
        return
    ops.quantize_append(w["cache"], w["newk"][s], w["newv"][s], w["cu1"], w["starts"][s], w["pt"])
    ops.decode_attention(w["cache"], w["qs"][s], w["pt"], w["lens"][s], w["max_len"], w["ws"], out=w["out"],
                         impl=kernel)


def launches_per_step(kernel="auto"):
    # fused step: (append + query preparation + window tiles), history, combine;
    # the two-call path: the append (one launch when the step appends at most W
    # tokens, else quantise + window copy), then window + history + combine
    if kernel == "auto":
        return 3
    return (1 if B <= W_RECENT else 2) + 3


def bits_per_element():
    """Stored bits per KV element of the workload's requests (mean): 16 in the
    BF16 windows, 2 + 2·(scale bits)/G in the INT2 history."""
    sb = 16.0 if SCALE_FMT == "f16" else 8.0
    return float(np.mean((16.0 * 320 + (2 + 2 * sb / G) * (LB - 320)) / LB))


def algorithmic_history_bytes(rec_bytes_per_token, L):
    hist = max(S_SINK, L - W_RECENT) - S_SINK      # history [S, max(S, L - W))
    return hist * (rec_bytes_per_token + 4)   # records + page-table entry


# --------------------------------------------------------------------------
# the oracle as CPU baseline / reference arm
# --------------------------------------------------------------------------
def oracle_sample(seed, L=None):
    """Builds (untimed) an oracle cache of one request at L tokens; returns a closure timing one decode."""
    import torch
    import oracle
    from rotated_int2_kv_gb300 import synth
    L = int(LB.max()) + 1 if L is None else L
    Ck = oracle.covariance(synth.calib_samples(SEED, 0, D))
    Cv = oracle.covariance(synth.calib_samples(SEED, 1, D))
    Rk = oracle.build_rotation(Ck, D)[0].astype(np.float32)
    Rv = oracle.build_rotation(Cv, D)[0].astype(np.float32)
    oc = oracle.OracleCache(oracle.OracleConfig(D, HQ, HKV, G, S_SINK, W_RECENT, 0.9, SCALE_FMT), L, 1, Rk, Rv)
    scales = synth.outlier_scales(seed, HKV, D, OUTLIERS)
    k, v = synth.kv_tokens(seed, 0, 0, L, HKV, D, scales)
    pt = np.arange(L, dtype=np.int64)[None, :]
    oc.append(k.float().numpy(), v.float().numpy(), [0, L], [0], [0], pt)
    q = synth.queries(seed, 0, 1, HQ, D).float().numpy()

    def run():
        t0 = time.perf_counter()
        oracle.decode_attention(oc, q, pt, [L], [0])
        return time.perf_counter() - t0
    return run, L


def boundary_cases(w, n_hist=8192):
    """INT2 records of request 0's first n_hist history tokens (written by the
    chunked fill) against the oracle's: exact, rounding ties (codes within 1e-6
    of a boundary, (s, z) at an fp16 tie) and other mismatches, counted over
    (token, KV head, K|V, group)."""
    import torch
    import oracle
    from rotated_int2_kv_gb300 import synth
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from parity_util import classify_records
    L = S_SINK + n_hist + W_RECENT
    k, v = synth.kv_tokens(w["seed"], 0, 0, L, HKV, D, w["scales"], device="cuda")
    oc = oracle.OracleCache(oracle.OracleConfig(D, HQ, HKV, G, S_SINK, W_RECENT, 0.9, SCALE_FMT), L, 1,
                            w["Rk"], w["Rv"])
    oc.append(k.float().cpu().numpy(), v.float().cpu().numpy(), [0, L], [0], [0],
              np.arange(L, dtype=np.int64)[None, :], keep_y=True)
    hist = np.arange(S_SINK, S_SINK + n_hist)
    hr = w["cache"].head_records()
    got = np.zeros((L, HKV, hr.shape[-1]), np.uint8)
    got[hist] = hr[w["pt"][0, S_SINK:S_SINK + n_hist].long()].cpu().numpy()
    st = classify_records(got, oc, hist)
    return {"sample": "request 0, history tokens %d..%d (chunked-fill path), all KV heads, K and V"
                      % (S_SINK, S_SINK + n_hist - 1),
            "group_records": int(n_hist * HKV * 2 * (D // G)), "exact": st["exact"], "code_ties": st["code_ties"],
            "sz_ties": st["sz_ties"], "other_mismatches": st["bad"],
            "rule": "codes bit-exact except (y-z)/s within 1e-6*max(1,|u|) of a rounding boundary; (s, z) exact "
                    "except the fp32 value within 1e-6 relative of a rounding tie of the storage format (%s)"
                    % ("fp16" if SCALE_FMT == "f16" else "E4M3")}


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, rank, ws):
    if rank != 0:
        return
    run, L = oracle_sample(SEED)
    for _ in range(args.warmup):
        run()
    t = sum(run() for _ in range(args.steps))
    val = args.steps * L / t
    sample = "oracle fp64 decode of 1 request x 32 q heads at L=%d (cache built untimed)" % L
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(rec_tok=640):
    hist_gb = float(np.maximum(LB - S_SINK - W_RECENT, 0).sum()) * rec_tok / 1e9
    uniform = bool((LB == LB[0]).all())
    ctx = ("context %d (64 sink + %d INT2 + 256 recent)" % (int(LB[0]), int(LB[0]) - 320) if uniform else
           "contexts %d..%d (ragged)" % (int(LB.min()), int(LB.max())))
    shape = ("Qwen3-8B-shaped" if (HQ, HKV, D) == (32, 8, 128) else
             "Qwen3-32B-shaped" if (HQ, HKV, D) == (64, 8, 128) else "GQA-%d wide-head" % (HQ // HKV))
    sz = "" if SCALE_FMT == "f16" else ", E4M3 scale and zero"
    return {"workload": "%s decode step (append 1 token + attention), batch %d, %s, %d q / %d KV heads, "
                        "d %d, group %d%s, clip 0.9, shuffled page table, page_size 1"
                        % (shape, B, ctx, HQ, HKV, D, G, sz),
            "batch": B, "context": int(LB.max()), "q_heads": HQ, "kv_heads": HKV, "head_dim": D, "group_size": G,
            "l2": ("inputs larger than L2 (%.2f GB INT2 history per step)" % hist_gb if hist_gb * 1e9 > 129e6 else
                   "inputs smaller than L2 (%.3f GB INT2 history, not flushed): a latency figure, not a "
                   "bandwidth one" % hist_gb),
            "parallelism": "replicas (independent requests per GPU)"}


def set_workload(name):
    """Sets the module's workload shape (the globals the builders read)."""
    global B, HQ, HKV, D, G, L_BASE, LB, OUTLIERS, CYCLE, SCALE_FMT
    B, HQ, HKV, D, G, L_BASE, OUTLIERS, CYCLE = 32, 32, 8, 128, 64, 100_000, "fixed4", 100
    SCALE_FMT = "f16"
    if name == "qwen8b-100k-e4m3":
        SCALE_FMT = "e4m3"
    elif name == "small":
        B, L_BASE = 4, 65536
    elif name == "mid":
        B, L_BASE = 8, 100_000
    elif name == "b1-32k":
        B, L_BASE = 1, 32_767
    elif name == "qwen32b-ragged":
        from rotated_int2_kv_gb300 import synth
        B, HQ, HKV, D, G = 8, 64, 8, 128, 64
        OUTLIERS, CYCLE = "per_head", 50
        LB = synth.ragged_lengths(SEED, B, 65_536, 131_072).astype(np.int64) - 1
    elif name == "gqa6-wide":
        B, HQ, HKV, D, G, L_BASE = 5, 24, 4, 256, 128, 112_000
    if name != "qwen32b-ragged":
        LB = np.full(B, L_BASE, dtype=np.int64)


def shape_measure(name, steps, warmup, hbm_peak):
    """Decode steps of another workload shape (history kernel time, roofline,
    clocks), for the extra keys of the default bench line."""
    import torch
    from rotated_int2_kv_gb300 import ops
    saved = (B, HQ, HKV, D, G, L_BASE, LB, OUTLIERS, CYCLE, SCALE_FMT)
    try:
        set_workload(name)
        w = build_decode_workload(0, steps + warmup)
        for i in range(warmup):
            decode_step(w, i, "auto")
        torch.cuda.synchronize()
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
        time.sleep(0.3)
        ops.profile_enable([ops.PROF_HISTORY])
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            decode_step(w, warmup + i, "auto")
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        hms, hn = ops.profile_read(ops.PROF_HISTORY)
        ops.profile_enable(None)
        clk = clocks.stop()
        assert ops.device_status() == 0
        rec_tok, _ = ops.cache_bytes_per_token(w["cfg"])
        tokens, hist_bytes = 0, 0
        for i in range(steps):
            Ls = LB + (warmup + i) % CYCLE + 1
            tokens += int(Ls.sum())
            hist_bytes += sum(algorithmic_history_bytes(rec_tok, int(L)) for L in Ls)
        achieved = (hist_bytes / hn) / (hms / hn / 1e3) / 1e9
        out = {"workload": workload_config(rec_tok)["workload"], "value": tokens / (ms / 1e3), "unit": UNIT,
               "ms_per_step": ms / steps, "steps": steps,
               "history_ms_per_step": hms / hn, "bits_per_kv_element": bits_per_element(),
               "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                            "frac": achieved / hbm_peak, "kernel": "history kernel (INT2 split-K)",
                            "peak_source": "measured hbm_gbs"},
               "clocks": clk}
        del w
        return out
    finally:
        globals().update(dict(zip(("B", "HQ", "HKV", "D", "G", "L_BASE", "LB", "OUTLIERS", "CYCLE", "SCALE_FMT"),
                                  saved)))
        torch.cuda.empty_cache()


def prefill_measure(name, L0, C, reps, bf16_peak):
    """One request's prefill chunk of C queries over an L0-token prefix
    (oscar_prefill_attention): time per call, chunk tokens/s and the
    attention's algorithmic tensor rate (4·d flops per (query, head, key))."""
    import torch
    from rotated_int2_kv_gb300 import ops, synth
    dev = torch.device("cuda")
    hq, hkv, d, g_ = (32, 8, 128, 64) if name == "qwen8b" else (24, 4, 256, 128)
    cfg = ops.Config(d, hq, hkv, g_, S_SINK, W_RECENT, 0.9)
    Rk, Rv = rotations(d)
    L = L0 + C
    pt = synth.page_table(SEED, 1, L, L).to(dev)
    cache = ops.LayerCache(cfg, L, 1, Rk, Rv, device=dev)
    scales = synth.outlier_scales(SEED, hkv, d, "fixed4")
    for p0 in range(0, L0, 8192):
        n = min(8192, L0 - p0)
        k, v = synth.kv_tokens(SEED, 0, p0, n, hkv, d, scales, device=dev)
        ops.quantize_append(cache, k, v, torch.tensor([0, n], dtype=torch.int32, device=dev),
                            torch.tensor([p0], dtype=torch.int32, device=dev), pt)
    k, v = synth.kv_tokens(SEED, 0, L0, C, hkv, d, scales, device=dev)
    q = synth.queries(SEED, 5, C, hq, d, device=dev)
    cu = torch.tensor([0, C], dtype=torch.int32, device=dev)
    st = torch.tensor([L0], dtype=torch.int32, device=dev)
    ws = torch.empty(ops.prefill_workspace_bytes(cfg, 1, C), dtype=torch.uint8, device=dev)
    out = torch.empty((C, hq, d), dtype=torch.float32, device=dev)
    for _ in range(2):
        ops.prefill_attention(cache, q, k, v, cu, st, pt, C, out=out, workspace=ws)
    torch.cuda.synchronize()
    ops.profile_enable([ops.PROF_PREFILL])
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ops.prefill_attention(cache, q, k, v, cu, st, pt, C, out=out, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    call_ms = e0.elapsed_time(e1) / reps
    kms, kn = ops.profile_read(ops.PROF_PREFILL)
    ops.profile_enable(None)
    assert ops.device_status() == 0
    keys = C * L0 + C * (C + 1) / 2                      # (query, key) pairs per head
    flops = 4.0 * d * hq * keys
    kern_ms = kms / max(kn, 1)
    tf = flops / (kern_ms / 1e3) / 1e12
    del cache, ws, out
    torch.cuda.empty_cache()
    return {"workload": "%s prefill chunk: %d queries over a %d-token prefix (%d INT2 history), %d q / %d KV heads, "
                        "d %d, group %d, batch 1" % ("Qwen3-8B-shaped" if name == "qwen8b" else "GQA-6 wide-head",
                                                     C, L0, max(0, L0 - 320), hq, hkv, d, g_),
            "ms_per_call": call_ms, "attention_kernel_ms": kern_ms, "chunk_tokens_per_s": C / (call_ms / 1e3),
            "roofline": {"bound": "tensor", "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": tf / bf16_peak, "kernel": "prefill_attn_kernel (mma.sync f16, INT2 in place)",
                         "peak_source": "measured bf16_tflops (f16 runs at the bf16 rate)",
                         "flops": "4*d per (query head, key) pair, causal within the chunk"}}


# GB300 fp64 on the CUDA cores: 1.25 TFLOP/s nominal (2 fp64 FMA per SM and
# cycle x 152 SMs x 2.07 GHz x 2 flops = 1.26 TFLOP/s); no measured fp64 peak.
FP64_PEAK_TFLOPS = 1.25


def calibration_measure(reps):
    """The calibration statistics on the device: C_Q over 65,536 key rows and
    C_S over one 4,096-token sequence's scores, d 128, bf16 activations.
    Time per call (CUDA events) and the fp64 rate of the algorithmic flops:
    n·d(d+1) for C_Q (one triangle of XᵀX), 2·n_q·n_k·d + n_q·d(d+1) for C_S."""
    import numpy as np
    import torch
    from rotated_int2_kv_gb300 import ops, synth
    dev = torch.device("cuda")
    d, n, nq = 128, 65536, 4096
    x = torch.from_numpy(synth.calib_samples(SEED, 0, d, n=n).astype(np.float32)).to(torch.bfloat16).to(dev)
    v = torch.from_numpy(synth.calib_samples(SEED, 1, d, n=nq).astype(np.float32)).to(torch.bfloat16).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(SEED)
    scores = torch.softmax(torch.randn((nq, nq), generator=g, device=dev), dim=1)   # rows of attention weights

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    cq_ms = timed(lambda: ops.covariance_device(x))
    cs_ms = timed(lambda: ops.value_covariance_device(scores, v))
    assert ops.device_status() == 0
    cq_tf = n * d * (d + 1) / (cq_ms / 1e3) / 1e12
    cs_tf = (2.0 * nq * nq * d + nq * d * (d + 1)) / (cs_ms / 1e3) / 1e12
    del x, v, scores
    torch.cuda.empty_cache()
    return {"workload": "C_Q of 65,536 bf16 rows and C_S of a 4,096 x 4,096 score matrix over 4,096 bf16 value rows, "
                        "d 128, fp64 accumulation",
            "covariance_ms": cq_ms, "value_covariance_ms": cs_ms, "covariance_fp64_tflops": cq_tf,
            "roofline": {"bound": "alu", "achieved": cs_tf, "peak": FP64_PEAK_TFLOPS, "unit": "TFLOP/s",
                         "frac": cs_tf / FP64_PEAK_TFLOPS, "kernel": "value covariance (Y = S V, then YᵀY; fp64 FMA)",
                         "peak_source": "nominal fp64 rate (152 SMs x 2 FMA/cycle x 2.07 GHz)"}}


# --------------------------------------------------------------------------
def main():
    args = parse()
    rank, ws, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, ws)
        return
    set_workload(args.workload)
    import torch
    from rotated_int2_kv_gb300 import ops
    if not os.path.exists(ops._LIB_PATH):
        from rotated_int2_kv_gb300 import build
        build.build()
    ops.lib()
    if args.calibration_only:
        if rank == 0:
            print(json.dumps(calibration_measure(max(args.steps, 1))), flush=True)
        return
    if args.prefill_only:
        peaks = {}
        try:
            peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        except (OSError, ValueError):
            pass
        if rank == 0:
            print(json.dumps(prefill_measure(args.prefill_only, args.prefill_prefix, args.prefill_chunk,
                                             max(args.steps, 1), float(peaks.get("bf16_tflops", 1900.0)))),
                  flush=True)
        return
    steps_total = args.steps + args.warmup
    w = build_decode_workload(rank, steps_total)
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        decode_step(w, i, args.decode_kernel)
    torch.cuda.synchronize()
    assert ops.device_status() == 0

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    ops.profile_enable([ops.PROF_HISTORY])
    barrier(ws)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        decode_step(w, args.warmup + i, args.decode_kernel)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    ms = e0.elapsed_time(e1)
    hist_ms, hist_n = ops.profile_read(ops.PROF_HISTORY)
    ops.profile_enable(None)
    # the same steps again without the event pair around the history kernel
    # (it separates that kernel from its neighbours' dependent launches, which
    # shows at launch-bound sizes): the step time a caller sees
    barrier(ws)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        decode_step(w, args.warmup + i, args.decode_kernel)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    ms_plain = max_over_ranks(e0.elapsed_time(e1), ws)
    clk = clocks.stop()
    # per-kernel breakdown from a separate pass (every launch between event pairs,
    # which costs the step some time, so it is not the timed region)
    nb = min(args.steps, 200)
    kinds = ((ops.PROF_HISTORY, "history"), (ops.PROF_STEP_PRE, "append + query prep + window (one launch)"),
             (ops.PROF_QUANTIZE, "append (quantise + window rows)"),
             (ops.PROF_WINDOW_COPY, "window_copy"), (ops.PROF_WINDOW, "window + query prep"),
             (ops.PROF_COMBINE, "combine"))
    ops.profile_enable([k for k, _ in kinds])
    for i in range(nb):
        decode_step(w, args.warmup + i, args.decode_kernel)
    torch.cuda.synchronize()
    kernel_ms = {}
    for kind, name in kinds:
        kms, kn = ops.profile_read(kind)
        if kn:                                   # kinds that launched in this step
            kernel_ms[name] = kms / nb
    ops.profile_enable(None)

    rec_tok, _ = ops.cache_bytes_per_token(w["cfg"])
    tokens = 0
    hist_bytes = 0
    for i in range(args.steps):
        Ls = LB + (args.warmup + i) % CYCLE + 1
        tokens += int(Ls.sum())
        hist_bytes += sum(algorithmic_history_bytes(rec_tok, int(L)) for L in Ls)
    value, ms = job_throughput(tokens, ms, ws)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    achieved = (hist_bytes / hist_n) / (hist_ms / hist_n / 1e3) / 1e9 if hist_n else None
    traffic = None
    try:
        prof = json.load(open(os.path.join(ROOT, "profiles", "history_traffic.json")))
        import hashlib
        src = os.path.join(ROOT, "rotated_int2_kv_gb300", "csrc", "oscar_decode_mma.cu")
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        # counters taken on another version of the kernel do not describe this one
        if (prof.get("kernel") == "history_mma_kernel" and prof.get("kernel_source_sha256") == sha
                and args.decode_kernel == "auto" and args.workload == "qwen8b-100k"):
            traffic = prof.get("bytes_per_launch_full")
    except (OSError, ValueError):
        pass
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if args.decode_kernel == "simt" else "f16 mma / f32 accumulate",
            "data": "synthetic", "config": workload_config(rec_tok),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": (achieved / hbm_peak) if achieved else None, "traffic": traffic,
                         "kernel": "history kernel (INT2 split-K)", "peak_source": "measured hbm_gbs",
                         "history_ms_per_step": hist_ms / max(hist_n, 1),
                         "pct_of_8TBs": (achieved / 8000.0) if achieved else None},
            "kernel_ms_per_step": kernel_ms,
            "ms_per_step_without_kernel_events": ms_plain / args.steps,
            "gpu_launches": launches_per_step(args.decode_kernel) * args.steps,
            "bits_per_kv_element": bits_per_element(),
            "clocks": clk}
    # ---- end to end through the C ABI with host buffers ----------------------
    if not args.no_e2e:
        line["e2e"] = e2e_measure(w, args, ws)
    if not args.no_append:
        line["append"] = append_measure()
        if args.shapes and ws == 1:
            line["append_d256"] = append_measure_d256()
    if args.shapes and args.workload == "qwen8b-100k" and ws == 1:
        line["shapes"] = {name: shape_measure(name, 400, 5, hbm_peak)
                          for name in ("qwen32b-ragged", "gqa6-wide", "qwen8b-100k-e4m3")}
        line["prefill"] = {name: prefill_measure(name, 32768, 8192, 3, float(peaks.get("bf16_tflops", 1900.0)))
                           for name in ("qwen8b", "gqa6-wide")}
        line["calibration"] = calibration_measure(5)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        run, L = oracle_sample(w["seed"])
        run()
        t = 0.0
        n = 0
        while t < 10.0 and n < 8:
            t += run()
            n += 1
        line["cpu_baseline"] = {"value": n * L / t, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                                "sample": "%d x oracle fp64 decode of 1 request x %d q heads at L=%d "
                                          "(cache built untimed)" % (n, HQ, L)}
        line["boundary_cases"] = boundary_cases(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def e2e_measure(w, args, ws):
    """Same metric with per-step inputs in pinned host memory and the output read back."""
    import torch
    from rotated_int2_kv_gb300 import ops
    dev = torch.device("cuda")
    n = max(10, min(args.steps, 500))
    hk = [t.cpu().pin_memory() for t in w["newk"]]
    hv = [t.cpu().pin_memory() for t in w["newv"]]
    hq = [t.cpu().pin_memory() for t in w["qs"]]
    hout = torch.empty((B, HQ, D), dtype=torch.float32).pin_memory()
    dk = torch.empty_like(w["newk"][0])
    dv = torch.empty_like(w["newv"][0])
    dq = torch.empty_like(w["qs"][0])
    stream = torch.cuda.current_stream()
    barrier(ws)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    tokens = 0
    for i in range(n):
        s = i % CYCLE
        dk.copy_(hk[s], non_blocking=True)
        dv.copy_(hv[s], non_blocking=True)
        dq.copy_(hq[s], non_blocking=True)
        if args.decode_kernel == "auto":
            ops.decode_step(w["cache"], dk, dv, dq, w["pt"], w["lens"][s], w["max_len"], w["ws"], out=w["out"])
        else:
            ops.quantize_append(w["cache"], dk, dv, w["cu1"], w["starts"][s], w["pt"])
            ops.decode_attention(w["cache"], dq, w["pt"], w["lens"][s], w["max_len"], w["ws"], out=w["out"],
                                 impl=args.decode_kernel)
        hout.copy_(w["out"], non_blocking=True)
        tokens += int((LB + s + 1).sum())
    e1.record(stream)
    torch.cuda.synchronize()
    value, _ = job_throughput(tokens, e0.elapsed_time(e1), ws)
    h2d = dk.numel() * 2 + dv.numel() * 2 + dq.numel() * 2
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": hout.numel() * 4, "steps": n}


def append_measure():
    """Chunked-prefill append of a 32,768-token Qwen3-8B-shaped request (32,448 INT2 + 320 BF16)."""
    import torch
    from rotated_int2_kv_gb300 import ops, synth
    dev = torch.device("cuda")
    L = 32768
    cfg = ops.Config(D, HQ, HKV, G, S_SINK, W_RECENT, 0.9, scale_fmt=SCALE_FMT)
    Rk, Rv = rotations(D)
    pt = synth.page_table(SEED, 1, L, L).to(dev)
    cache = ops.LayerCache(cfg, L, 1, Rk, Rv, device=dev)
    scales = synth.outlier_scales(SEED, HKV, D, "fixed4")
    k, v = synth.kv_tokens(SEED, 0, 0, L, HKV, D, scales, device=dev)
    cu = torch.tensor([0, L], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(3):
        ops.quantize_append(cache, k, v, cu, st, pt)
    torch.cuda.synchronize()
    ops.profile_enable([ops.PROF_QUANTIZE, ops.PROF_WINDOW_COPY])
    reps = 20
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    h0 = time.perf_counter()
    for _ in range(reps):
        ops.quantize_append(cache, k, v, cu, st, pt)
    host_ms = (time.perf_counter() - h0) * 1e3 / reps     # host time to issue one call
    e1.record()
    torch.cuda.synchronize()
    qms, qn = ops.profile_read(1)
    wms, wn = ops.profile_read(2)
    ops.profile_enable(None)
    call_ms = e0.elapsed_time(e1) / reps
    hist = L - S_SINK - W_RECENT
    rec_tok, _ = ops.cache_bytes_per_token(cfg)
    alg_bytes = hist * (HKV * D * 2 * 2 + rec_tok + 4)   # bf16 K,V in + records out + page table
    kern_ms = qms / max(qn, 1)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    bf16_peak = float(peaks.get("bf16_tflops", 1900.0))
    # the rotation runs as three bf16 passes (hi, mid, lo parts of R) on the tensor cores
    mma_flops = 3 * hist * HKV * 2 * 2 * D * D
    achieved = alg_bytes / (kern_ms / 1e3) / 1e9
    return {"workload": "one 32,768-token request appended at once (32,448 INT2 + 320 BF16), "
                        "Qwen3-8B-shaped layer", "value": alg_bytes / (call_ms / 1e3) / 1e9, "unit": "GB/s",
            "ms_per_call": call_ms, "quantize_kernel_ms": kern_ms,
            "window_copy_kernel_ms": wms / max(wn, 1), "host_ms_per_call": host_ms,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "kernel": "quantize_tc_kernel (tcgen05 rotation + INT2)",
                         "peak_source": "measured hbm_gbs",
                         "tensor_tflops": mma_flops / (kern_ms / 1e3) / 1e12,
                         "tensor_frac_of_bf16_burst": mma_flops / (kern_ms / 1e3) / 1e12 / bf16_peak}}

def append_measure_d256():
    """Chunked-prefill append at head_dim 256: one 8,192-token chunk (L0 = 16,384) of a
    GQA-6 wide-head layer (24 q / 4 KV heads, group 128): the fp32 FMA tiles."""
    import torch
    from rotated_int2_kv_gb300 import ops, synth
    dev = torch.device("cuda")
    d, hq, hkv, g_ = 256, 24, 4, 128
    C, L0 = 8192, 16384
    L = L0 + C
    cfg = ops.Config(d, hq, hkv, g_, S_SINK, W_RECENT, 0.9)
    Rk, Rv = rotations(d)
    pt = synth.page_table(SEED, 1, L, L).to(dev)
    cache = ops.LayerCache(cfg, L, 1, Rk, Rv, device=dev)
    scales = synth.outlier_scales(SEED, hkv, d, "fixed4")
    one = torch.zeros(1, dtype=torch.int32, device=dev)
    for p0 in range(0, L0, C):
        k, v = synth.kv_tokens(SEED, 0, p0, C, hkv, d, scales, device=dev)
        ops.quantize_append(cache, k, v, torch.tensor([0, C], dtype=torch.int32, device=dev), one + p0, pt)
    k, v = synth.kv_tokens(SEED, 0, L0, C, hkv, d, scales, device=dev)
    cu = torch.tensor([0, C], dtype=torch.int32, device=dev)
    st = one + L0
    ops.quantize_append(cache, k, v, cu, st, pt)
    torch.cuda.synchronize()
    ops.profile_enable([ops.PROF_QUANTIZE, ops.PROF_WINDOW_COPY])
    reps = 20
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ops.quantize_append(cache, k, v, cu, st, pt)
    e1.record()
    torch.cuda.synchronize()
    qms, qn = ops.profile_read(ops.PROF_QUANTIZE)
    wms, wn = ops.profile_read(ops.PROF_WINDOW_COPY)
    ops.profile_enable(None)
    assert ops.device_status() == 0
    call_ms = e0.elapsed_time(e1) / reps
    kern_ms = qms / max(qn, 1)
    n_hist = C                                           # positions entering the history per call
    rec_tok, _ = ops.cache_bytes_per_token(cfg)
    alg_bytes = n_hist * (hkv * d * 2 * 2 + rec_tok + 4)
    flops = 2.0 * n_hist * hkv * 2 * d * d               # y = x·R for every K and V head vector
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    bf16_peak = float(peaks.get("bf16_tflops", 1900.0))
    tf = flops / (kern_ms / 1e3) / 1e12
    return {"workload": "one 8,192-token chunk appended at L0 = 16,384 (8,192 enter the history), GQA-6 wide-head "
                        "layer: 24 q / 4 KV heads, d 256, group 128",
            "value": alg_bytes / (call_ms / 1e3) / 1e9, "unit": "GB/s", "ms_per_call": call_ms,
            "quantize_kernel_ms": kern_ms, "window_copy_kernel_ms": wms / max(wn, 1),
            "roofline": {"bound": "tensor", "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s", "frac": tf / bf16_peak,
                         "kernel": "quantize_tc256_kernel (tcgen05, R's half in two bf16 parts per CTA, exact INT2 "
                                   "decisions)",
                         "peak_source": "measured bf16_tflops",
                         "flops": "2*d*d per K or V head vector (the rotation; the tensor cores run it as two bf16 parts)",
                         "hbm_gbs": alg_bytes / (kern_ms / 1e3) / 1e9}}


if __name__ == "__main__":
    main()
