"""Host checks of bench.py's workload bookkeeping (no GPU)."""

import importlib
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def _bench():
    import bench
    return importlib.reload(bench)           # fresh module globals per test


def test_default_workload_is_the_batch32_100k_step():
    b = _bench()
    assert (b.B, b.HQ, b.HKV, b.D, b.G) == (32, 32, 8, 128, 64)
    assert b.LB.shape == (32,) and (b.LB == 100_000).all()
    cfg = b.workload_config(640)
    assert cfg["workload"].startswith("Qwen3-8B-shaped decode step (append 1 token + attention), batch 32, "
                                      "context 100000 (64 sink + 99680 INT2 + 256 recent)")
    assert cfg["l2"].startswith("inputs larger than L2 (2.04 GB")


def test_history_bytes_count_records_and_page_table_entries():
    b = _bench()
    # 64 sink and 256 recent tokens are BF16: the history of L tokens is L - 320
    assert b.algorithmic_history_bytes(640, 100_001) == (100_001 - 320) * 644
    assert b.algorithmic_history_bytes(640, 320) == 0
    assert b.algorithmic_history_bytes(640, 100) == 0


def test_ragged_workload_lengths_and_description():
    b = _bench()
    from rotated_int2_kv_gb300 import synth
    lens = synth.ragged_lengths(b.SEED, 8, 65_536, 131_072).astype(np.int64)
    assert ((lens >= 65_536) & (lens <= 131_072)).all()
    b.B, b.HQ, b.HKV, b.D, b.G = 8, 64, 8, 128, 64
    b.LB = lens - 1
    cfg = b.workload_config(640)
    assert "Qwen3-32B-shaped" in cfg["workload"] and "(ragged)" in cfg["workload"]
    assert cfg["context"] == int(lens.max()) - 1
    # tokens of one step: every request at its own length
    s = 3
    assert int((b.LB + s + 1).sum()) == int(lens.sum()) + 8 * s


def test_prefill_only_options():
    b = _bench()
    saved = sys.argv
    try:
        sys.argv = ["bench.py"]
        a = b.parse()
        assert a.prefill_only is None and (a.prefill_prefix, a.prefill_chunk) == (32768, 8192)
        sys.argv = ["bench.py", "--prefill-only", "gqa6-wide", "--prefill-prefix", "8192", "--prefill-chunk", "1024",
                    "--steps", "1"]
        a = b.parse()
        assert (a.prefill_only, a.prefill_prefix, a.prefill_chunk, a.steps) == ("gqa6-wide", 8192, 1024, 1)
        assert not a.calibration_only
        sys.argv = ["bench.py", "--calibration-only", "--steps", "3"]
        a = b.parse()
        assert a.calibration_only and a.steps == 3
    finally:
        sys.argv = saved
