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
