"""GPU parity of oscar_prefill_attention against the oracle's chunked-prefill
attention (oracle.prefill_attention), on the same cache contents: the oracle
builds the cache and the test copies it to the device.  Bound: max-abs 2e-3 and
relative-L2 1e-3 on the fp32 outputs."""

import numpy as np
import pytest
import torch

import oracle
from rotated_int2_kv_gb300 import synth
from parity_util import ATOL, RTOL_L2, attn_errors, device_cache_from_oracle

pytestmark = pytest.mark.gpu

SEED = 1234


def _rotations(d, seed=SEED):
    Rk, _ = oracle.build_rotation(oracle.covariance(synth.calib_samples(seed, 0, d)), d)
    Rv, _ = oracle.build_rotation(oracle.covariance(synth.calib_samples(seed, 1, d)), d)
    return Rk.astype(np.float32), Rv.astype(np.float32)


def _run(d, Hq, Hkv, G, S, W, prefixes, chunks, heads=None, mode="fixed4", q_dtype=torch.bfloat16,
         kv_dtype=torch.bfloat16, scale_fmt="f16"):
    from rotated_int2_kv_gb300 import ops
    B = len(prefixes)
    maxL = max(p + c for p, c in zip(prefixes, chunks)) + 1
    pool = B * maxL + 11
    Rk, Rv = _rotations(d)
    cfg = ops.Config(d, Hq, Hkv, G, S, W, 0.9, kv_dtype=kv_dtype, q_dtype=q_dtype, scale_fmt=scale_fmt)
    ocfg = oracle.OracleConfig(d, Hq, Hkv, G, S, W, 0.9, scale_fmt)
    pt = synth.page_table(SEED, B, maxL, pool)
    req = np.arange(B, dtype=np.int32)[::-1].copy()          # window rows permuted
    oc = oracle.OracleCache(ocfg, pool, B, Rk, Rv)
    scales = synth.outlier_scales(SEED, Hkv, d, mode)
    # the prefixes, appended in two calls (a chunk and a few decode-like tokens)
    for b in range(B):
        if prefixes[b]:
            k, v = synth.kv_tokens(SEED, b, 0, prefixes[b], Hkv, d, scales)
            oc.append(k.float().numpy(), v.float().numpy(), [0, prefixes[b]], [0], [int(req[b])], pt.numpy()[b:b + 1])
    dc = device_cache_from_oracle(ops, oc, cfg)
    # the chunks
    ks, vs = zip(*[synth.kv_tokens(SEED, b, prefixes[b], chunks[b], Hkv, d, scales, dtype=kv_dtype) for b in range(B)])
    k = torch.cat(ks)
    v = torch.cat(vs)
    T = k.shape[0]
    q = synth.queries(SEED, 7, T, Hq, d, dtype=q_dtype)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    dev = torch.device("cuda")
    out = ops.prefill_attention(dc, q.to(dev), k.to(dev), v.to(dev), torch.from_numpy(cu).to(dev),
                                torch.tensor(prefixes, dtype=torch.int32, device=dev), pt.to(dev), max(chunks),
                                req_idx=torch.from_numpy(req).to(dev))
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    for b in range(B):
        want = oracle.prefill_attention(oc, q[cu[b]:cu[b + 1]].float().numpy(), k[cu[b]:cu[b + 1]].float().numpy(),
                                        v[cu[b]:cu[b + 1]].float().numpy(), pt.numpy(), prefixes[b], int(req[b]), b=b,
                                        heads=heads)
        hs = range(Hq) if heads is None else heads
        for h in hs:
            err, rel = attn_errors(got[cu[b]:cu[b + 1], h], want[:, h])
            assert err <= ATOL and rel <= RTOL_L2, (b, h, err, rel)


def test_prefill_small_ragged_batch():
    # prefixes with and without history, ragged chunks (one query, a partial tile, several tiles)
    _run(128, 32, 8, 64, 64, 256, prefixes=[0, 100, 2000, 777], chunks=[40, 1, 97, 64], heads=(0, 3, 13, 31))


def test_prefill_gqa6_wide_heads():
    _run(256, 24, 4, 128, 64, 256, prefixes=[3000, 500], chunks=[70, 33], heads=(0, 5, 6, 17, 23))


def test_prefill_gqa8_and_group32_fp32_inputs():
    _run(128, 16, 2, 32, 16, 64, prefixes=[900, 0], chunks=[50, 20], q_dtype=torch.float32, kv_dtype=torch.float32)


@pytest.mark.parametrize("d,Hq,Hkv,G", [(128, 32, 8, 64), (256, 24, 4, 128), (128, 6, 3, 128)])
def test_prefill_e4m3_scale_zero(d, Hq, Hkv, G):
    _run(d, Hq, Hkv, G, 64, 256, prefixes=[2100, 700], chunks=[77, 16], heads=(0, 1, Hq - 1), scale_fmt="e4m3")


def test_prefill_d64_no_sink():
    _run(64, 8, 2, 64, 0, 128, prefixes=[600, 129], chunks=[45, 16])


def test_prefill_one_query_equals_decode_after_append():
    # a one-token chunk against the prefix, and oscar_decode_attention of the
    # same token after its append, agree when no token leaves the recent
    # window (the prefix still fits S + W - 1)
    from rotated_int2_kv_gb300 import ops
    d, Hq, Hkv, G, S, W = 128, 32, 8, 64, 64, 256
    L0 = 200
    Rk, Rv = _rotations(d)
    cfg = ops.Config(d, Hq, Hkv, G, S, W)
    dev = torch.device("cuda")
    pt = synth.page_table(SEED, 1, L0 + 1, L0 + 1).to(dev)
    dc = ops.LayerCache(cfg, L0 + 1, 1, Rk, Rv, device=dev)
    scales = synth.outlier_scales(SEED, Hkv, d)
    k, v = synth.kv_tokens(SEED, 0, 0, L0 + 1, Hkv, d, scales, device=dev)
    one = torch.zeros(1, dtype=torch.int32, device=dev)
    ops.quantize_append(dc, k[:L0].contiguous(), v[:L0].contiguous(), torch.tensor([0, L0], dtype=torch.int32, device=dev), one, pt)
    q = synth.queries(SEED, 3, 1, Hq, d, device=dev)
    pre = ops.prefill_attention(dc, q, k[L0:].contiguous(), v[L0:].contiguous(),
                                torch.tensor([0, 1], dtype=torch.int32, device=dev),
                                torch.tensor([L0], dtype=torch.int32, device=dev), pt, 1)
    ops.quantize_append(dc, k[L0:].contiguous(), v[L0:].contiguous(), torch.tensor([0, 1], dtype=torch.int32, device=dev),
                        torch.tensor([L0], dtype=torch.int32, device=dev), pt)
    ws = ops.alloc_workspace(cfg, 1, L0 + 1)
    dec = ops.decode_attention(dc, q, pt, torch.tensor([L0 + 1], dtype=torch.int32, device=dev), L0 + 1, ws)
    torch.cuda.synchronize()
    err, rel = attn_errors(pre.cpu().numpy(), dec.cpu().numpy())
    assert err <= ATOL and rel <= RTOL_L2, (err, rel)
