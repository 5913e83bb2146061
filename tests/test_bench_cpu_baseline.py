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



def test_kernels_per_call_follows_the_workspace_query():
    """The kernel count bench.py reports per layer call (host-side queries
    only): the single kernel for one FP8 token, shrink grid + GEMM for a
    decode tile and for rank 16 at M = 512, and the expand pass besides them
    for M = 512 at rank 64."""
    import precision_gemm_token_gb300 as E
    E.build()
    E.load()
    assert bench.kernels_per_call(0, 1, 28672, 4096, 64) == E.epilora_layer_forward_kernels(0, 1, 4096, 64)
    assert bench.kernels_per_call(1, 32, 28672, 4096, 64) == 2
    assert bench.kernels_per_call(1, 512, 28672, 4096, 16) == 2
    assert bench.kernels_per_call(1, 512, 28672, 4096, 64) == 3
    assert bench.kernels_per_call(0, 2112, 57344, 8192, 16) == 2
