"""Failure detection on the GPU without a fault: bounded waits report, never hang.

Every pipeline wait of the kernels is an mbarrier wait with a cycle budget
(mbar_wait_bounded); when it runs out the kernel sets OSCAR_DEV_TIMEOUT in the
device status word and returns.  oscar_selftest_bounded_wait runs that same
wait on a barrier nothing completes (a flag that nothing sets), and the test
checks the status bit and that the context still works afterwards.  Decode
with out-of-pool page-table entries is flagged (OSCAR_DEV_BAD_SLOT) and the
offending records are skipped, not read.
"""

import numpy as np
import pytest
import torch

import oracle
from rotated_int2_kv_gb300 import synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports():
    from rotated_int2_kv_gb300 import ops
    ops.device_status(clear=True)
    ops.selftest_bounded_wait(2_000_000, complete=False)     # ~1 ms of SM cycles
    assert ops.device_status(clear=True) & ops.DEV_TIMEOUT
    # a completed barrier is not a timeout
    ops.selftest_bounded_wait(2_000_000, complete=True)
    assert ops.device_status(clear=True) == 0
    # the context is still usable
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2


def test_decode_flags_out_of_pool_slots_without_faulting():
    from rotated_int2_kv_gb300 import ops
    d, Hq, Hkv, G, S, W = 128, 8, 2, 64, 16, 32
    B, L = 2, 900
    Rk, _ = oracle.build_rotation(None, d)
    Rv, _ = oracle.build_rotation(None, d)
    cfg = ops.Config(d, Hq, Hkv, G, S, W, 0.9)
    pool = B * L
    dc = ops.LayerCache(cfg, pool, B, Rk.astype(np.float32), Rv.astype(np.float32))
    pt = synth.page_table(7, B, L, pool).cuda()
    k = torch.randn((B * L, Hkv, d), device="cuda").to(torch.bfloat16)
    cu = torch.tensor([0, L, 2 * L], dtype=torch.int32, device="cuda")
    ops.quantize_append(dc, k, k, cu, torch.zeros(B, dtype=torch.int32, device="cuda"), pt)
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) == 0
    bad = pt.clone()
    bad[0, S + 5] = pool + 10 ** 6         # history position of request 0 outside the pool
    bad[1, S + 7] = -3
    q = torch.randn((B, Hq, d), device="cuda").to(torch.bfloat16)
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    ws = ops.alloc_workspace(cfg, B, L)
    out = ops.decode_attention(dc, q, bad, lens, L, ws)
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) & ops.DEV_BAD_SLOT
    assert torch.isfinite(out).all()
    # the same call with a clean table sets nothing
    ops.decode_attention(dc, q, pt, lens, L, ws)
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) == 0
