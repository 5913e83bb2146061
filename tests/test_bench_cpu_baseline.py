"""bench.py's host baseline: the oracle spread over single-threaded worker
processes (spawned) on a column sample returns a positive extrapolated layer
time and names the sample."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_oracle_pool_step_on_a_small_sample():
    sample = bench.oracle_prepare("8b_m1_fp8", 0.0005)
    assert all(d["ncol"] >= 8 and d["wq"].shape[0] == d["ncol"] for d in sample)
    pool = bench.OraclePool()
    try:
        us, detail = pool.step("8b_m1_fp8", sample)
    finally:
        pool.close()
    assert us > 0 and "gate_up" in detail and pool.n >= 1

