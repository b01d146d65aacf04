"""GPU parity of oscar_quantize_append against the fp64 oracle.

INT2 records: bit-exact except counted rounding-boundary cases (see
parity_util).  BF16 windows: bit-exact.  Slots outside the history: untouched.
"""

import numpy as np
import pytest
import torch

import oracle
from rotated_int2_kv_gb300 import synth
from parity_util import classify_records, record_boundary_cases

pytestmark = pytest.mark.gpu

SEED = 1234


def _rotations(d, seed=SEED):
    Rk, _ = oracle.build_rotation(oracle.covariance(synth.calib_samples(seed, 0, d)), d)
    Rv, _ = oracle.build_rotation(oracle.covariance(synth.calib_samples(seed, 1, d)), d)
    return Rk.astype(np.float32), Rv.astype(np.float32)


def _misaligned(t):
    """A copy of t whose data pointer is one element past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
    out = buf[1:1 + t.numel()].view(t.shape)
    out.copy_(t)
    assert out.data_ptr() % 16 != 0
    return out


def run_append_scenario(d, Hq, Hkv, G, S, W, kv_dtype, calls, clip=0.9, mode="fixed4", pool_extra=37,
                        seed=SEED, unaligned=False, rotations=None, keep=None, scale_fmt="f16", shared=0.0):
    from rotated_int2_kv_gb300 import ops
    B = len(calls[0])
    Lfin = [sum(c[b] for c in calls) for b in range(B)]
    maxL = max(max(Lfin), 1)
    pool = B * maxL + pool_extra
    cfg = ops.Config(d, Hq, Hkv, G, S, W, clip, kv_dtype=kv_dtype, scale_fmt=scale_fmt)
    Rk, Rv = _rotations(d, seed) if rotations is None else rotations
    pt = synth.page_table(seed, B, maxL, pool, shuffled=True)
    req = torch.tensor(list(reversed(range(B))), dtype=torch.int32)   # window rows permuted
    max_reqs = B + 2
    dev = torch.device("cuda")
    dc = ops.LayerCache(cfg, pool, max_reqs, Rk, Rv, device=dev)
    oc = oracle.OracleCache(oracle.OracleConfig(d, Hq, Hkv, G, S, W, clip, scale_fmt), pool, max_reqs, Rk, Rv)
    scales = synth.outlier_scales(seed, Hkv, d, mode)
    pos = [0] * B
    for call in calls:
        ks, vs = [], []
        for b in range(B):
            k, v = synth.kv_tokens(seed, b, pos[b], call[b], Hkv, d, scales, dtype=kv_dtype, shared=shared)
            ks.append(k)
            vs.append(v)
        k = torch.cat(ks)
        v = torch.cat(vs)
        cu = np.concatenate([[0], np.cumsum(call)]).astype(np.int32)
        kd, vd = k.to(dev), v.to(dev)
        if unaligned:
            kd, vd = _misaligned(kd), _misaligned(vd)
        ops.quantize_append(dc, kd, vd, torch.from_numpy(cu).to(dev),
                            torch.tensor(pos, dtype=torch.int32, device=dev), pt.to(dev), req_idx=req.to(dev))
        oc.append(k.float().numpy(), v.float().numpy(), cu, pos, req.numpy(), pt.numpy(), keep_y=True)
        pos = [pos[b] + call[b] for b in range(B)]
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    gpu_rec = dc.records.cpu().numpy()
    hist_slots = []
    for b in range(B):
        _, lo, hi, rlo, rhi = oracle.regions(Lfin[b], S, W)
        hist_slots += list(pt[b, lo:hi].numpy())
    hist_slots = np.array(sorted(hist_slots), dtype=np.int64)
    stats = classify_records(gpu_rec, oc, hist_slots)
    assert stats["bad"] == 0, stats
    record_boundary_cases("append d%d G%d Hkv%d %s" % (d, G, Hkv, scale_fmt), stats,
                          len(hist_slots) * Hkv * 2 * (d // G))
    others = np.setdiff1d(np.arange(pool), hist_slots)
    assert not gpu_rec[others].any(), "records outside the history were written"
    # windows: bit-exact bf16
    sink_bits, ring_bits = oc.window_bits()
    gs = dc.sink.view(torch.int16).cpu().numpy().view(np.uint16)
    gr = dc.recent.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(B):
        rq = int(req[b])
        se, lo, hi, rlo, rhi = oracle.regions(Lfin[b], S, W)
        if S > 0:
            assert np.array_equal(gs[rq, :se], sink_bits[rq, :se])
        idx = np.arange(rlo, rhi) % W
        assert np.array_equal(gr[rq, idx], ring_bits[rq, idx])
    if keep is not None:
        keep.update(cfg=cfg, dc=dc, oc=oc, pt=pt, req=req, lens=Lfin)
    return stats


def test_tiny_config_single_fill_fp32():
    # 1 layer, 4 q / 1 KV head, d 128, 64 + 704 + 256 tokens, fp32 K/V, group 64
    st = run_append_scenario(128, 4, 1, 64, 64, 256, torch.float32, [[1024]], pool_extra=0)
    assert st["exact"] > 0


def test_spill_heavy_small_windows_ragged():
    calls = [[5, 0, 17], [1, 1, 1], [20, 3, 0], [1, 30, 2], [9, 9, 9], [0, 0, 1], [40, 1, 64]]
    run_append_scenario(64, 12, 2, 32, 4, 8, torch.bfloat16, calls)


def test_wide_head_gqa6_chunks_then_decode_steps():
    calls = [[700, 400], [1, 1], [300, 0], [1, 1], [0, 513], [1, 1]]
    run_append_scenario(256, 24, 4, 128, 64, 256, torch.bfloat16, calls, mode="fixed4")


def test_gqa8_per_head_outliers():
    calls = [[2000, 333, 1], [1, 1, 1], [1, 1, 1], [257, 1, 300]]
    run_append_scenario(128, 64, 8, 64, 64, 256, torch.bfloat16, calls, mode="per_head")


@pytest.mark.parametrize("d,G", [(256, 256), (256, 32), (128, 128), (64, 64), (128, 32)])
def test_group_sizes(d, G):
    run_append_scenario(d, 2, 1, G, 16, 32, torch.bfloat16, [[300], [1], [77]])


@pytest.mark.parametrize("d,G,dtype,unaligned", [
    (128, 64, torch.bfloat16, False), (128, 32, torch.bfloat16, False), (128, 128, torch.float32, False),
    (64, 64, torch.bfloat16, False), (64, 32, torch.float32, False), (128, 64, torch.bfloat16, True),
    (256, 128, torch.bfloat16, False), (256, 64, torch.bfloat16, False), (256, 32, torch.float32, False),
    (256, 128, torch.bfloat16, True), (256, 256, torch.bfloat16, False)])
def test_large_appends_tiled_path(d, G, dtype, unaligned):
    # the second call moves 12,600+ vectors into the history (the tiled kernels:
    # tensor cores, at d = 256 one half of the channels per CTA with R in two
    # bf16 parts; fp32 FMA tiles for group 256): the ring's spilled tokens and
    # new ones, a ragged last tile
    calls = [[300, 290, 13], [2600, 2700, 1001]]
    st = run_append_scenario(d, 8, 2, G, 64, 256, dtype, calls, unaligned=unaligned)
    assert st["exact"] > 0


@pytest.mark.parametrize("d,G", [(256, 128), (256, 32), (128, 64), (128, 32)])
def test_tiled_exact_paths_under_load(d, G):
    # every row shares one strong direction per head, so the extremes of most
    # vectors fall on the same few channels of y: at d 256 more exact products
    # queue for one channel than a batch holds, and with group 32 more vectors
    # of a tile have an uncertain (s, z) than the row stash holds, so the
    # overflow paths (products over global memory) run next to the on-chip ones
    calls = [[300, 290, 13], [2600, 2700, 1001]]
    st = run_append_scenario(d, 8, 2, G, 64, 256, torch.bfloat16, calls, shared=8.0)
    assert st["exact"] > 0


@pytest.mark.parametrize("d,Hq,Hkv,G,S,W,calls", [
    # tensor-core tiles (a 5,000-token fill), decode steps with ring spills
    (128, 32, 8, 64, 64, 256, [[5000, 333, 1], [1, 1, 1], [1, 1, 1], [257, 1, 300]]),
    # d 256 fp32 tiles and decode steps (the wide GQA-6 layer, group 128)
    (256, 24, 4, 128, 64, 256, [[700, 2600], [1, 1], [300, 0], [1, 1]]),
    # small ragged calls through the warp-per-vector kernels; group 32
    (64, 12, 2, 32, 4, 8, [[5, 0, 17], [1, 1, 1], [20, 3, 0], [40, 1, 64]]),
    # one group per head (group = head_dim): 68-byte records padded to 72, odd KV head count
    (128, 6, 3, 128, 16, 32, [[1300, 20, 700], [1, 1, 1], [77, 0, 5]]),
])
def test_e4m3_scale_zero(d, Hq, Hkv, G, S, W, calls):
    # one-byte (E4M3) scale and zero: packed records, slot layout, the same
    # exact-decision rule with E4M3 rounding ties
    from rotated_int2_kv_gb300 import ops
    keep = {}
    st = run_append_scenario(d, Hq, Hkv, G, S, W, torch.bfloat16, calls, scale_fmt="e4m3", keep=keep)
    assert st["exact"] > 0
    dc = keep["dc"]
    assert dc.records.numel() == dc.num_slots * ops.slot_bytes(keep["cfg"])
    assert ops.record_bytes(keep["cfg"]) == (d // 2 + 4 * (d // G) + 7) // 8 * 8


def test_many_kv_heads():
    # 32 KV heads: a large call through the tiled kernel, then decode steps
    run_append_scenario(128, 32, 32, 64, 64, 256, torch.bfloat16, [[300, 290], [1500, 1300], [1, 1], [1, 1]])


def test_large_windows():
    # sink 128 and a 1,024-token recent ring: spills start only past 1,152 tokens
    run_append_scenario(64, 4, 1, 64, 128, 1024, torch.bfloat16, [[1500], [1], [700], [1]])


def test_no_sink_tokens():
    run_append_scenario(128, 8, 2, 64, 0, 256, torch.bfloat16, [[600, 100], [1, 1], [300, 0], [1, 1]])


def test_decode_step_appends_spill_every_step():
    calls = [[330, 330, 400, 64]] + [[1, 1, 1, 1]] * 12
    run_append_scenario(128, 32, 8, 64, 64, 256, torch.bfloat16, calls)


def test_sink_only_and_no_history():
    # lengths that never reach the history: everything stays in the windows
    st = run_append_scenario(128, 8, 2, 64, 64, 256, torch.bfloat16, [[10, 64, 320], [5, 0, 0]])
    assert st["exact"] == 0 and st["bad"] == 0


def test_clip_ratio_one_and_empty_calls():
    from rotated_int2_kv_gb300 import ops
    run_append_scenario(128, 4, 2, 64, 8, 16, torch.bfloat16, [[0, 0], [100, 50], [0, 0], [3, 0]], clip=1.0)
    # an empty batch and an all-empty call are no-ops
    cfg = ops.Config(128, 4, 2, 64, 8, 16)
    Rk, Rv = _rotations(128)
    dc = ops.LayerCache(cfg, 64, 2, Rk, Rv)
    z = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    ops.quantize_append(dc, z, z, torch.zeros(1, dtype=torch.int32, device="cuda"),
                        torch.zeros(0, dtype=torch.int32, device="cuda"),
                        torch.zeros((0, 16), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert not dc.records.any()


def test_device_checks_flag_bad_slots_without_faulting():
    from rotated_int2_kv_gb300 import ops
    cfg = ops.Config(64, 2, 1, 32, 4, 8)
    Rk, Rv = _rotations(64)
    dc = ops.LayerCache(cfg, 32, 1, Rk, Rv)
    ops.device_status(clear=True)
    k = torch.randn((40, 1, 64), device="cuda").to(torch.bfloat16)
    pt = torch.arange(40, dtype=torch.int32, device="cuda").reshape(1, 40)
    pt[0, 20] = 10 ** 6            # slot outside the pool: skipped and flagged
    ops.quantize_append(dc, k, k, torch.tensor([0, 40], dtype=torch.int32, device="cuda"),
                        torch.zeros(1, dtype=torch.int32, device="cuda"), pt)
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) & ops.DEV_BAD_SLOT
    assert ops.device_status(clear=True) == 0


@pytest.mark.parametrize("block", [None, 16])
def test_library_built_rotation_end_to_end(block):
    # R_K, R_V from the library's own builder (oscar_build_rotation, and with a
    # block-diagonal Hadamard factor), not the oracle's: append parity, then
    # decode against the oracle on the same R
    from rotated_int2_kv_gb300 import ops
    from parity_util import ATOL, RTOL_L2, attn_errors, device_cache_from_oracle
    d = 128
    Rk, _, _ = ops.build_rotation(ops.covariance(synth.calib_samples(SEED, 0, d)), d, hadamard_block=block)
    Rv, _, _ = ops.build_rotation(ops.covariance(synth.calib_samples(SEED, 1, d)), d, hadamard_block=block)
    keep = {}
    calls = [[1500, 700], [1, 1], [1, 1], [1, 1]]
    run_append_scenario(d, 32, 8, 64, 64, 256, torch.bfloat16, calls, rotations=(Rk, Rv), keep=keep)
    cfg, dc, oc, pt, req, lens = keep["cfg"], keep["dc"], keep["oc"], keep["pt"], keep["req"], keep["lens"]
    dev = torch.device("cuda")
    B = len(lens)
    q = synth.queries(SEED, 9, B, cfg.num_q_heads, d)
    want = oracle.decode_attention(oc, q.float().numpy(), pt.numpy(), lens, req.numpy())
    ws = ops.alloc_workspace(cfg, B, pt.shape[1])
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    same = device_cache_from_oracle(ops, oc, cfg)
    out = ops.decode_attention(same, q.to(dev), pt.to(dev), lens_d, pt.shape[1], ws, req_idx=req.to(dev))
    err, rel = attn_errors(out.cpu().numpy(), want)
    assert err <= ATOL and rel <= RTOL_L2, ("identical cache", err, rel)
    out = ops.decode_attention(dc, q.to(dev), pt.to(dev), lens_d, pt.shape[1], ws, req_idx=req.to(dev))
    err, rel = attn_errors(out.cpu().numpy(), want)
    assert rel <= RTOL_L2, ("gpu-built cache", err, rel)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
