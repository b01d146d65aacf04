"""The binding's C structs are built once and reused; every change on the
Python side (a config field, a cache buffer or size) must give a fresh struct
with the new values.  Host only: the cache's buffers live on the CPU here."""
import numpy as np
import pytest
import torch

from rotated_int2_kv_gb300 import ops


def test_config_struct_follows_fields():
    cfg = ops.Config(128, 32, 8, 64)
    a = cfg.c()
    assert cfg.c() is a                                   # unchanged fields: the same struct
    assert (a.head_dim, a.num_q_heads, a.num_kv_heads, a.group_size) == (128, 32, 8, 64)
    assert a.scale_dtype == ops.SCALE_F16 and a.kv_dtype == ops.DTYPE_BF16
    cfg.group_size = 32
    b = cfg.c()
    assert b is not a and b.group_size == 32
    cfg.scale_fmt = "e4m3"
    assert cfg.c().scale_dtype == ops.SCALE_E4M3
    cfg.kv_dtype = torch.float32
    assert cfg.c().kv_dtype == ops.DTYPE_F32
    cfg.clip_ratio = 0.75
    assert abs(cfg.c().clip_ratio - 0.75) < 1e-7
    cfg.kv_dtype = torch.float16                          # not a supported input type
    with pytest.raises(ValueError):
        cfg.c()
    assert ops.Config(128, 32, 8, 64) == ops.Config(128, 32, 8, 64)   # the memo is not a field


def test_cache_struct_follows_buffers():
    cfg = ops.Config(64, 4, 2, 32)
    R = np.eye(64, dtype=np.float32)
    cache = ops.LayerCache(cfg, 10, 2, R, R, device="cpu")
    a = cache.c()
    assert cache.c() is a
    assert a.records == cache.records.data_ptr() and a.rot_v == cache.rot_v.data_ptr()
    assert (a.num_slots, a.max_reqs) == (10, 2)
    cache.records = torch.zeros_like(cache.records)       # a new buffer: a new struct
    b = cache.c()
    assert b is not a and b.records == cache.records.data_ptr()
    cache.num_slots = 7
    assert cache.c().num_slots == 7


def test_device_check_compares_devices():
    cfg = ops.Config(64, 4, 2, 32)
    R = np.eye(64, dtype=np.float32)
    cache = ops.LayerCache(cfg, 4, 1, R, R, device="cpu")
    assert ops._device_of(cache, torch.zeros(2), None) == torch.device("cpu")
