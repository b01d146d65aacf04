"""The allocation-free decode entry point (oscar_decode_attention_noalloc).

It exists for callers that cannot allocate device memory -- runtimes that
reserve the GPU for their own pool, or code paths where cudaMalloc is not
allowed -- and uses a fixed scratch array built into the library.  Its output
must match oscar_decode_attention (caller workspace) within the attention
tolerance, on two calls in a row through the C ABI (the second call runs on
scratch left over from the first).  Collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

SEED = 4321


def _case(ops, B, L, step):
    from rotated_int2_kv_gb300 import synth
    import oracle
    d, Hq, Hkv, G = 128, 32, 8, 64
    cfg = ops.Config(d, Hq, Hkv, G)
    Rk, _ = oracle.build_rotation(oracle.covariance(synth.calib_samples(SEED, 0, d)), d)
    Rv, _ = oracle.build_rotation(oracle.covariance(synth.calib_samples(SEED, 1, d)), d)
    dev = torch.device("cuda")
    pool = B * L
    pt = synth.page_table(SEED, B, L, pool).to(dev)
    cache = ops.LayerCache(cfg, pool, B, Rk.astype(np.float32), Rv.astype(np.float32), device=dev)
    scales = synth.outlier_scales(SEED, Hkv, d)
    kk, vv = zip(*[synth.kv_tokens(SEED, b, 0, L, Hkv, d, scales, device=dev) for b in range(B)])
    cu = torch.arange(0, (B + 1) * L, L, dtype=torch.int32, device=dev)
    ops.quantize_append(cache, torch.cat(kk), torch.cat(vv), cu, torch.zeros(B, dtype=torch.int32, device=dev), pt)
    q = synth.queries(SEED, step, B, Hq, d, device=dev)
    lens = torch.tensor([L - 7 * b for b in range(B)], dtype=torch.int32, device=dev)
    return cfg, cache, pt, q, lens


def test_noalloc_matches_workspace_entry_point_twice():
    from rotated_int2_kv_gb300 import ops
    from parity_util import ATOL, RTOL_L2, attn_errors
    L = 6000
    for step, B in enumerate((3, 5)):              # two calls in a row, different shapes
        cfg, cache, pt, q, lens = _case(ops, B, L, step)
        ws = ops.alloc_workspace(cfg, B, L)
        ref = ops.decode_attention(cache, q, pt, lens, L, ws)
        out = torch.full_like(ref, float("nan"))
        rc = ops.lib().oscar_decode_attention_noalloc(
            ctypes.byref(cfg.c()), ctypes.byref(cache.c()), q.data_ptr(), pt.data_ptr(), pt.shape[1],
            lens.data_ptr(), None, B, L, out.data_ptr(),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, ops.last_error()
        torch.cuda.synchronize()
        err, rel = attn_errors(out.cpu().numpy(), ref.cpu().numpy())
        assert err <= ATOL and rel <= RTOL_L2, (step, err, rel)
        # the Python binding of the same entry point, into a caller-given output
        out2 = torch.full_like(ref, float("nan"))
        ops.decode_attention_noalloc(cache, q, pt, lens, L, out=out2)
        torch.cuda.synchronize()
        err, rel = attn_errors(out2.cpu().numpy(), ref.cpu().numpy())
        assert err <= ATOL and rel <= RTOL_L2, ("binding", step, err, rel)
    assert ops.device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from rotated_int2_kv_gb300 import ops
    cfg = ops.Config(128, 32, 8, 64)
    need = ops.decode_workspace_bytes(cfg, 4096, 200000)
    assert need > 16 << 20
    cache = ops.CLayerCache(16, 16, 16, 16, 16, 10, 1)
    rc = ops.lib().oscar_decode_attention_noalloc(ctypes.byref(cfg.c()), ctypes.byref(cache), 16, 16, 200000,
                                                  16, None, 4096, 200000, 16, None)
    assert rc == -3 and "16777216" in ops.last_error()
