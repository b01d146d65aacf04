"""GPU checks of the fused decode step (oscar_decode_step).

Its output and every byte it writes to the cache must equal those of
oscar_quantize_append (one token per request) followed by
oscar_decode_attention on the same stream: both paths run over two caches
filled identically, step after step, and are compared bit for bit.  The
two-call path itself is checked against the oracle by the append and decode
parity tests; one oracle comparison here closes the loop on the fused path.
"""

import numpy as np
import pytest
import torch

import oracle
from rotated_int2_kv_gb300 import synth
from parity_util import ATOL, RTOL_L2, attn_errors, classify_records

pytestmark = pytest.mark.gpu

SEED = 4321


def _rotations(d, seed=SEED):
    Rk, _ = oracle.build_rotation(oracle.covariance(synth.calib_samples(seed, 0, d)), d)
    Rv, _ = oracle.build_rotation(oracle.covariance(synth.calib_samples(seed, 1, d)), d)
    return Rk.astype(np.float32), Rv.astype(np.float32)


def _run(d, Hq, Hkv, G, S, W, prefix, steps, kv_dtype=torch.bfloat16, q_dtype=torch.bfloat16,
         scale_fmt="f16", mode="fixed4", oracle_check=True):
    from rotated_int2_kv_gb300 import ops
    dev = torch.device("cuda")
    B = len(prefix)
    maxL = max(prefix) + steps + 1
    pool = B * maxL + 7
    Rk, Rv = _rotations(d)
    cfg = ops.Config(d, Hq, Hkv, G, S, W, 0.9, kv_dtype=kv_dtype, q_dtype=q_dtype, scale_fmt=scale_fmt)
    pt = synth.page_table(SEED, B, maxL, pool).to(dev)
    req = torch.tensor(list(reversed(range(B))), dtype=torch.int32, device=dev)
    two = ops.LayerCache(cfg, pool, B + 1, Rk, Rv, device=dev)      # append + decode calls
    one = ops.LayerCache(cfg, pool, B + 1, Rk, Rv, device=dev)      # fused step
    scales = synth.outlier_scales(SEED, Hkv, d, mode)
    # the prefixes (chunked append, identical in both caches)
    # every input is drawn on the host (the generator's stream depends on the device) and copied
    kk, vv = zip(*[synth.kv_tokens(SEED, b, 0, prefix[b], Hkv, d, scales, dtype=kv_dtype) for b in range(B)])
    cu = torch.tensor(np.concatenate([[0], np.cumsum(prefix)]).astype(np.int32), device=dev)
    zero = torch.zeros(B, dtype=torch.int32, device=dev)
    for c in (two, one):
        ops.quantize_append(c, torch.cat(kk).to(dev), torch.cat(vv).to(dev), cu, zero, pt, req_idx=req)
    ws_a = ops.alloc_workspace(cfg, B, maxL)
    ws_b = ops.alloc_workspace(cfg, B, maxL)
    cu1 = torch.arange(B + 1, dtype=torch.int32, device=dev)
    pos = np.array(prefix)
    for s in range(steps):
        kk, vv = zip(*[synth.kv_tokens(SEED, b, int(pos[b]), 1, Hkv, d, scales, dtype=kv_dtype) for b in range(B)])
        k = torch.cat(kk).to(dev)
        v = torch.cat(vv).to(dev)
        q = synth.queries(SEED, s, B, Hq, d, dtype=q_dtype).to(dev)
        start = torch.tensor(pos, dtype=torch.int32, device=dev)
        lens = start + 1
        ops.quantize_append(two, k, v, cu1, start, pt, req_idx=req)
        out_a = ops.decode_attention(two, q, pt, lens, maxL, ws_a, req_idx=req)
        out_b = ops.decode_step(one, k, v, q, pt, lens, maxL, ws_b, req_idx=req)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b), ("step", s, float((out_a - out_b).abs().max()))
        assert torch.equal(two.records, one.records), ("records", s)
        assert torch.equal(two.sink.view(torch.int16), one.sink.view(torch.int16)), ("sink", s)
        assert torch.equal(two.recent.view(torch.int16), one.recent.view(torch.int16)), ("recent", s)
        pos = pos + 1
    assert ops.device_status() == 0
    if oracle_check:
        # the fused path's records and attention against the oracle
        oc = oracle.OracleCache(oracle.OracleConfig(d, Hq, Hkv, G, S, W, 0.9, scale_fmt), pool, B + 1, Rk, Rv)
        ptn = pt.cpu().numpy()
        reqn = req.cpu().numpy()
        ks, vs = zip(*[synth.kv_tokens(SEED, b, 0, int(pos[b]), Hkv, d, scales, dtype=kv_dtype) for b in range(B)])
        L = pos.astype(np.int64)
        oc.append(torch.cat(ks).float().numpy(), torch.cat(vs).float().numpy(),
                  np.concatenate([[0], np.cumsum(L)]).astype(np.int32), [0] * B, reqn, ptn, keep_y=True)
        hist = np.concatenate([ptn[b, S:max(S, int(L[b]) - W)] for b in range(B)])
        st = classify_records(one.records.cpu().numpy(), oc, hist)
        assert st["bad"] == 0, st
        want = oracle.decode_attention(oc, q.float().cpu().numpy(), ptn, L, reqn)
        err, rel = attn_errors(out_b.cpu().numpy(), want)
        if st["code_ties"] + st["sz_ties"] == 0:
            assert err <= ATOL and rel <= RTOL_L2, (err, rel)
        else:
            assert rel <= RTOL_L2, (err, rel)


def test_qwen8b_heads_ragged_with_short_requests():
    # 32 q / 8 KV heads: the tensor-core window and history; requests that stay
    # in the sink (1, 40), fill the windows exactly (320) and spill every step
    _run(128, 32, 8, 64, 64, 256, [1, 40, 319, 320, 1500, 700], steps=6)


def test_gqa8_e4m3():
    _run(128, 64, 8, 64, 64, 256, [1300, 333, 2000], steps=4, scale_fmt="e4m3", mode="per_head")


def test_gqa6_wide_heads_d256():
    # CUDA-core window tiles, and the append of a 256-channel vector by a 128-thread block
    _run(256, 24, 4, 128, 64, 256, [900, 400], steps=4)


def test_gqa16_fp32_inputs_small_windows():
    _run(128, 32, 2, 64, 4, 16, [100, 7, 33], steps=20, kv_dtype=torch.float32, q_dtype=torch.float32)


def test_d64_no_sink_group32():
    _run(64, 12, 2, 32, 0, 8, [50, 9], steps=12)


def test_invalid_length_flags_and_appends_nothing():
    from rotated_int2_kv_gb300 import ops
    d, Hq, Hkv = 128, 8, 2
    cfg = ops.Config(d, Hq, Hkv, 64, 8, 16)
    Rk, Rv = _rotations(d)
    dev = torch.device("cuda")
    c = ops.LayerCache(cfg, 64, 1, Rk, Rv, device=dev)
    pt = torch.arange(64, dtype=torch.int32, device=dev).reshape(1, 64)
    k = torch.ones((1, Hkv, d), dtype=torch.bfloat16, device=dev)
    q = torch.ones((1, Hq, d), dtype=torch.bfloat16, device=dev)
    ws = ops.alloc_workspace(cfg, 1, 64)
    ops.device_status(clear=True)
    out = ops.decode_step(c, k, k, q, pt, torch.tensor([65], dtype=torch.int32, device=dev), 64, ws)
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) & ops.DEV_BAD_LEN
    assert not out.any()
    assert not c.records.any() and not c.recent.view(torch.int16).any() and not c.sink.view(torch.int16).any()
