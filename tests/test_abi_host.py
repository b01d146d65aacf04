"""Host-side tests of liboscar.so: it loads, exports every symbol include/oscar.h
declares, validates arguments before touching the GPU, and its host rotation
builder agrees with the fp64 oracle.  No GPU needed."""

import ctypes
import math
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "oscar.h")


@pytest.fixture(scope="module")
def ops():
    from rotated_int2_kv_gb300 import ops as _ops
    from rotated_int2_kv_gb300 import build as _build
    if not os.path.exists(_ops._LIB_PATH):
        _build.build()
    _ops.lib()
    return _ops


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oscar_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(ops):
    syms = declared_symbols()
    assert "oscar_quantize_append" in syms and "oscar_decode_attention" in syms
    assert "oscar_build_rotation" in syms
    for s in syms:
        assert hasattr(ops.lib(), s), s
    assert "sm_103a" in ops.version()


def _cfg(ops, **kw):
    base = dict(head_dim=128, num_q_heads=32, num_kv_heads=8, group_size=64)
    base.update(kw)
    return ops.Config(**base)


def test_record_and_token_bytes_match_oracle(ops):
    for d, G in ((128, 64), (256, 128), (128, 32), (64, 64), (256, 32)):
        cfg = _cfg(ops, head_dim=d, group_size=G, num_q_heads=8, num_kv_heads=4)
        assert ops.record_bytes(cfg) == oracle.record_bytes(d, G)
        int2, bf16 = ops.cache_bytes_per_token(cfg)
        assert int2 == 4 * oracle.record_bytes(d, G)
        assert bf16 == 4 * 2 * d * 2
    # 640 B/token for the 8-KV-head d=128 layer
    assert ops.cache_bytes_per_token(_cfg(ops))[0] == 640
    assert ops.slot_bytes(_cfg(ops)) == 640


def test_e4m3_record_and_slot_bytes_match_oracle(ops):
    from oracle import quant as oq
    for d, G, H in ((128, 64, 8), (256, 128, 4), (128, 32, 2), (64, 64, 1), (128, 128, 3), (256, 256, 5)):
        cfg = _cfg(ops, head_dim=d, group_size=G, num_q_heads=2 * H, num_kv_heads=H, scale_fmt="e4m3")
        assert ops.record_bytes(cfg) == oracle.record_bytes(d, G, scale_bits=8) == oq.record_layout(d, G, "e4m3")["bytes"]
        assert ops.slot_bytes(cfg) == oq.slot_bytes(d, G, H, "e4m3")
        assert ops.cache_bytes_per_token(cfg)[0] == ops.slot_bytes(cfg)
    # 576 B/token for the 8-KV-head d=128 layer with one-byte scale and zero
    assert ops.cache_bytes_per_token(_cfg(ops, scale_fmt="e4m3"))[0] == 576


def test_unknown_scale_format_rejected(ops):
    c = _cfg(ops).c()
    c.scale_dtype = 2
    out = ctypes.c_int64()
    assert ops.lib().oscar_record_bytes(ctypes.byref(c), ctypes.byref(out)) == -1
    assert "scale_dtype" in ops.last_error()
    with pytest.raises(ValueError):
        _cfg(ops, scale_fmt="bf16").c()


@pytest.mark.parametrize("field,value", [
    ("head_dim", 96), ("head_dim", 512), ("group_size", 48), ("group_size", 16),
    ("num_q_heads", 30), ("num_q_heads", 8 * 17), ("sink", -1), ("recent", 0),
    ("clip_ratio", 0.0), ("clip_ratio", 1.5), ("num_kv_heads", 0)])
def test_invalid_config_rejected_before_launch(ops, field, value):
    cfg = _cfg(ops, **{field: value})
    with pytest.raises(ops.OscarError) as ei:
        ops.record_bytes(cfg)
    assert ei.value.code == -1
    assert ops.last_error()
    # the append entry validates the same way, with no device touched
    cache = ops.CLayerCache(16, 16, 16, 16, 16, 10, 1)
    rc = ops.lib().oscar_quantize_append(ctypes.byref(cfg.c()), ctypes.byref(cache), 16, 16, 1,
                                         16, 16, None, 16, 10, 1, None)
    assert rc == -1


def test_null_and_shape_errors(ops):
    L = ops.lib()
    assert L.oscar_record_bytes(None, None) == -2
    cfg = _cfg(ops)
    good = ops.CLayerCache(16, 16, 16, 16, 16, 10, 1)
    # NULL records
    bad = ops.CLayerCache(0, 16, 16, 16, 16, 10, 1)
    assert L.oscar_quantize_append(ctypes.byref(cfg.c()), ctypes.byref(bad), 16, 16, 1, 16, 16, None,
                                   16, 10, 1, None) == -2
    # misaligned records
    mis = ops.CLayerCache(8, 16, 16, 16, 16, 10, 1)
    assert L.oscar_quantize_append(ctypes.byref(cfg.c()), ctypes.byref(mis), 16, 16, 1, 16, 16, None,
                                   16, 10, 1, None) == -1
    # missing page table / negative batch
    assert L.oscar_quantize_append(ctypes.byref(cfg.c()), ctypes.byref(good), 16, 16, 1, 16, 16, None,
                                   None, 10, 1, None) == -2
    assert L.oscar_quantize_append(ctypes.byref(cfg.c()), ctypes.byref(good), 16, 16, 1, 16, 16, None,
                                   16, 10, -1, None) == -1
    # empty batch is a no-op success
    assert L.oscar_quantize_append(ctypes.byref(cfg.c()), ctypes.byref(good), None, None, 0, None, None,
                                   None, None, 1, 0, None) == 0
    # decode: pt_stride smaller than max_seq_len
    assert L.oscar_decode_attention(ctypes.byref(cfg.c()), ctypes.byref(good), 16, 16, 5, 16, None, 1,
                                    10, 16, 256, 1 << 20, None) == -1
    assert L.oscar_decode_attention(ctypes.byref(cfg.c()), ctypes.byref(good), 16, 16, 10, 16, None, 9999,
                                    10, 16, 256, 1 << 20, None) == -1


def test_covariances_match_oracle(ops):
    rng = np.random.default_rng(21)
    X = rng.standard_normal((333, 24))
    assert np.abs(ops.covariance(X) - oracle.covariance(X)).max() <= 1e-13
    S = rng.uniform(size=(17, 40))
    V = rng.standard_normal((40, 24))
    assert np.abs(ops.value_covariance(S, V) - oracle.value_covariance(S, V)).max() <= 1e-12


def test_rotation_without_covariance_is_exact_hadamard(ops):
    for d in (2, 64, 128, 256):
        R32, R64, w = ops.build_rotation(None, d, use_bitrev=False)
        H = oracle.hadamard(d) / math.sqrt(d)
        assert np.array_equal(R64, H)
        assert np.array_equal(R32, H.astype(np.float32))
    R32, _, _ = ops.build_rotation(None, 256, use_bitrev=False)
    assert np.abs(R32 @ R32.T - np.eye(256, dtype=np.float32)).max() == 0.0
    Rb32, Rb64, _ = ops.build_rotation(None, 128, use_bitrev=True)
    Ro, _ = oracle.build_rotation(None, 128, use_bitrev=True)
    assert np.array_equal(Rb64, Ro)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_rotation_from_covariance_matches_oracle(ops, d):
    from rotated_int2_kv_gb300 import synth
    X = synth.calib_samples(1234, 0, d)
    C = oracle.covariance(X)
    R32, R64, w = ops.build_rotation(C, d)
    Ro, wo = oracle.build_rotation(C, d)
    assert np.abs(w - wo).max() <= 1e-12 * abs(wo[0])
    assert np.abs(R64 - Ro).max() <= 1e-9
    assert np.abs(R64 @ R64.T - np.eye(d)).max() <= 1e-12
    assert np.abs(R32.astype(np.float64) - Ro).max() <= 1e-7


def test_rotation_argument_errors(ops):
    L = ops.lib()
    buf = np.zeros((96, 96), np.float32)
    assert L.oscar_build_rotation(None, 96, 1, buf.ctypes.data, None, None) == -1
    assert L.oscar_build_rotation(None, 64, 1, None, None, None) == -2
    bad = np.full((4, 4), np.nan)
    out = np.zeros((4, 4), np.float32)
    assert L.oscar_build_rotation(bad.ctypes.data, 4, 1, out.ctypes.data, None, None) == -1


@pytest.mark.parametrize("d,B", [(128, 16), (64, 8), (256, 64), (128, 1)])
def test_block_hadamard_rotation_matches_oracle(ops, d, B):
    import oracle
    rng = np.random.default_rng(d + B)
    X = rng.standard_normal((2048, d)) * (np.arange(1, d + 1) ** -0.75)
    C = oracle.covariance(X)
    R32, R64, w = ops.build_rotation(C, d, hadamard_block=B)
    Ro, wo = oracle.build_rotation(C, d, hadamard_block=B)
    assert np.abs(R64 - Ro).max() <= 1e-9
    assert np.abs(R32 - Ro.astype(np.float32)).max() <= 1e-7
    assert np.abs(R64 @ R64.T - np.eye(d)).max() <= 1e-12
    with pytest.raises(ops.OscarError):
        ops.build_rotation(C, d, hadamard_block=3)


def test_calibration_arguments_rejected_before_launch(ops):
    # the device calibration entry points check their arguments on the host
    # before any CUDA call (so these run without a GPU): -1 argument, -2 NULL
    L = ops.lib()
    nb = ctypes.c_size_t()
    assert L.oscar_covariance_workspace_bytes(0, 8, ctypes.byref(nb)) == -1
    assert L.oscar_covariance_workspace_bytes(10, 0, ctypes.byref(nb)) == -1
    assert L.oscar_covariance_workspace_bytes(10, 4097, ctypes.byref(nb)) == -1
    assert L.oscar_covariance_workspace_bytes(10, 8, None) == -2
    assert L.oscar_covariance_device(None, 0, 10, 8, 16, 16, 1 << 20, None) == -2
    assert L.oscar_covariance_device(16, 0, 10, 8, None, 16, 1 << 20, None) == -2
    assert L.oscar_covariance_device(16, 7, 10, 8, 16, 16, 1 << 20, None) == -1     # unknown dtype
    assert L.oscar_covariance_device(16, 0, 0, 8, 16, 16, 1 << 20, None) == -1      # no rows
    assert L.oscar_value_covariance_workspace_bytes(10, 0, 8, ctypes.byref(nb)) == -1
    assert L.oscar_value_covariance_workspace_bytes(10, 5, 0, ctypes.byref(nb)) == -1
    assert L.oscar_value_covariance_workspace_bytes(10, 5, 8, None) == -2
    assert L.oscar_value_covariance_device(None, 16, 0, 10, 5, 8, 16, 16, 1 << 20, None) == -2
    assert L.oscar_value_covariance_device(16, 16, 7, 10, 5, 8, 16, 16, 1 << 20, None) == -1
    assert L.oscar_value_covariance_device(16, 16, 0, 10, 0, 8, 16, 16, 1 << 20, None) == -1
    assert L.oscar_value_covariance_device(16, 16, 0, 65535 * 64 + 1, 5, 8, 16, 16, 1 << 20, None) == -1


def test_prefill_arguments_and_workspace_on_the_host(ops):
    L = ops.lib()
    cfg = _cfg(ops)                               # d 128, 32 q / 8 KV heads, group 64, 64 sink + 256 recent
    c = ctypes.byref(cfg.c())
    good = ops.CLayerCache(16, 16, 16, 16, 16, 10, 1)
    nb = ctypes.c_size_t()
    assert L.oscar_prefill_workspace_bytes(c, -1, 10, ctypes.byref(nb)) == -1
    assert L.oscar_prefill_workspace_bytes(c, 1, -1, ctypes.byref(nb)) == -1
    assert L.oscar_prefill_workspace_bytes(c, 1, 10, None) == -2
    # the workspace holds the chunk's rotated queries (fp16 hi and lo, per-group
    # sums) and the rotated BF16 tokens it sees (its own and both windows, K and V
    # as fp16 hi and lo): it does not grow with the cached prefix, which the call
    # does not even take
    al = lambda x: (x + 255) // 256 * 256
    for batch, tq in ((1, 100), (1, 8192), (3, 1000)):
        assert L.oscar_prefill_workspace_bytes(c, batch, tq, ctypes.byref(nb)) == 0
        dense = tq + batch * (64 + 256)
        want = 2 * al(tq * 32 * 128 * 2) + al(tq * 32 * 2 * 4) + 2 * al(dense * 8 * 2 * 128 * 2)
        assert nb.value == want
    args = lambda **kw: dict(dict(q=16, k=16, v=16, total_q=10, cu=16, st=16, rq=16, pt=16, pts=100, batch=1,
                                  mc=10, out=16, ws=None, wsb=0), **kw)

    def call(**kw):
        a = args(**kw)
        return L.oscar_prefill_attention(c, ctypes.byref(good), a["q"], a["k"], a["v"], a["total_q"], a["cu"],
                                         a["st"], a["rq"], a["pt"], a["pts"], a["batch"], a["mc"], a["out"],
                                         a["ws"], a["wsb"], None)

    assert call(batch=0) == 0 and call(total_q=0, mc=0) == 0       # nothing to do
    assert call(batch=-1) == -1 and call(batch=4097) == -1
    assert call(q=None) == -2 and call(out=None) == -2 and call(pt=None) == -2
    assert call(pts=0) == -1
    assert call(mc=0) == -1 and call(mc=11) == -1                  # max_chunk in [1, total_q]
    assert call(ws=None) == -3 and call(ws=16, wsb=1 << 30) == -3  # missing or misaligned workspace


def test_decode_step_arguments_on_the_host(ops):
    L = ops.lib()
    cfg = _cfg(ops)
    c = ctypes.byref(cfg.c())
    good = ops.CLayerCache(16, 16, 16, 16, 16, 10, 1)

    def call(kn=16, vn=16, pts=16, batch=1, msl=16):
        return L.oscar_decode_step(c, ctypes.byref(good), kn, vn, 16, 16, pts, 16, 16, batch, msl, 16, 256,
                                   1 << 20, None)

    assert call(batch=0) == 0                                       # empty batch: no-op
    assert call(batch=-1) == -1 and call(batch=4097) == -1
    assert call(msl=0) == -1
    assert call(pts=8) == -1                                        # pt_stride < max_seq_len
    assert call(kn=None) == -2 and call(vn=None) == -2
