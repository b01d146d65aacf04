"""CUDA-graph capture of a decode step (append one token per request + decode).

Every call of the library is capturable: no host synchronisation, no device
allocation, kernels launched on the caller's stream.  A step captured into a
CUDA graph and replayed gives the same cache contents and the same output, bit
for bit, as the same step run eagerly; replays with new inputs copied into the
captured buffers match eager steps too.
"""

import numpy as np
import pytest
import torch

import oracle
from rotated_int2_kv_gb300 import synth

pytestmark = pytest.mark.gpu


def _setup(B=3, L0=1500, d=128, Hq=16, Hkv=4, G=64, S=64, W=256, seed=77):
    from rotated_int2_kv_gb300 import ops
    Rk, _ = oracle.build_rotation(oracle.covariance(synth.calib_samples(seed, 0, d)), d)
    Rv, _ = oracle.build_rotation(oracle.covariance(synth.calib_samples(seed, 1, d)), d)
    cfg = ops.Config(d, Hq, Hkv, G, S, W, 0.9)
    max_len = L0 + 8
    pool = B * max_len
    dev = torch.device("cuda")
    dc = ops.LayerCache(cfg, pool, B, Rk.astype(np.float32), Rv.astype(np.float32), device=dev)
    pt = synth.page_table(seed, B, max_len, pool).to(dev)
    scales = synth.outlier_scales(seed, Hkv, d, "fixed4")
    k, v = zip(*[synth.kv_tokens(seed, b, 0, L0, Hkv, d, scales, device=dev) for b in range(B)])
    cu = torch.arange(0, (B + 1) * L0, L0, dtype=torch.int32, device=dev)
    ops.quantize_append(dc, torch.cat(k), torch.cat(v), cu, torch.zeros(B, dtype=torch.int32, device=dev), pt)
    torch.cuda.synchronize()
    return cfg, dc, pt, scales, max_len, seed


def _step_inputs(seed, B, Hkv, Hq, d, L, scales, s):
    k, v = zip(*[synth.kv_tokens(seed, b, L, 1, Hkv, d, scales, device="cuda") for b in range(B)])
    q = synth.queries(seed, 100 + s, B, Hq, d, device="cuda")
    return torch.cat(k), torch.cat(v), q


def _snapshot(dc):
    return [t.clone() for t in (dc.records, dc.sink, dc.recent)]


def _restore(dc, snap):
    for t, s in zip((dc.records, dc.sink, dc.recent), snap):
        t.copy_(s)


def test_captured_step_matches_eager():
    from rotated_int2_kv_gb300 import ops
    cfg, dc, pt, scales, max_len, seed = _setup()
    B, L0 = pt.shape[0], 1500
    d, Hq, Hkv = cfg.head_dim, cfg.num_q_heads, cfg.num_kv_heads
    dev = torch.device("cuda")
    ws = ops.alloc_workspace(cfg, B, max_len)
    cu1 = torch.arange(0, B + 1, dtype=torch.int32, device=dev)
    start = torch.full((B,), L0, dtype=torch.int32, device=dev)
    lens = start + 1
    # static buffers of the captured step
    sk, sv, sq = _step_inputs(seed, B, Hkv, Hq, d, L0, scales, 0)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
    snap = _snapshot(dc)

    def step():
        ops.quantize_append(dc, sk, sv, cu1, start, pt)
        ops.decode_attention(dc, sq, pt, lens, max_len, ws, out=out)

    # eager reference of two different steps (inputs of step 0 and step 1)
    eager = []
    for s in range(2):
        _restore(dc, snap)
        k, v, q = _step_inputs(seed, B, Hkv, Hq, d, L0, scales, s)
        sk.copy_(k); sv.copy_(v); sq.copy_(q)
        step()
        torch.cuda.synchronize()
        eager.append((out.clone(), [t.clone() for t in (dc.records, dc.sink, dc.recent)]))
    assert ops.device_status() == 0

    # capture once (after the eager warm-up), then replay with each step's inputs
    _restore(dc, snap)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    for s in range(2):
        _restore(dc, snap)
        k, v, q = _step_inputs(seed, B, Hkv, Hq, d, L0, scales, s)
        sk.copy_(k); sv.copy_(v); sq.copy_(q)
        g.replay()
        torch.cuda.synchronize()
        want_out, want_cache = eager[s]
        assert torch.equal(out, want_out), s
        for got, want in zip((dc.records, dc.sink, dc.recent), want_cache):
            assert torch.equal(got, want), s
    assert ops.device_status() == 0
