"""The workspace-free layer entry point (epilora_layer_forward_noalloc),
called through the C ABI, against epilora_layer_forward with a caller
workspace: two calls in a row on different batches, each bitwise equal to
the workspace entry point's result on the same inputs; oversize problems are
refused before anything is enqueued.

Kept in the last-collected file so that it also runs after every other GPU
test has used the library on the same device."""
import numpy as np
import pytest
import torch

import precision_gemm_token_gb300 as E
from oracle import epilora_oracle as O
from precision_gemm_token_gb300 import tensors as T
from synth import make_projection

from .gpu_util import FP8, NVFP4, ensure_lib, np32, status_buf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _inputs(fmt, M, K, N, L, r, seed):
    p = make_projection(M, K, N, L, r, seed=seed, idx_mode="uniform", mask_mode="all", device="cuda")
    w = T.quantize_weight(p.W, fmt)
    gx = T.nvfp4_global_scale(p.X) if fmt == NVFP4 else None
    return p, w, gx


def _noalloc(fmt, p, w, gx, Y, st, with_adapters=True):
    M, K = p.X.shape
    L, r = p.A.shape[0], p.A.shape[1]
    A, B = (p.A, p.B) if with_adapters else (None, None)
    return E.epilora_layer_forward_noalloc(fmt, M, w.N, K, p.X, p.X.stride(0), w.codes, w.scale, w.block_scale,
                                           w.global_scale, gx, A, B, L, r, p.idx, p.mask, Y, Y.stride(0), st, None)


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,L,r", [(1, 4096, 1024, 1, 64), (3, 2048, 4096, 2, 16), (33, 1024, 640, 5, 32),
                                       (200, 1024, 1280, 7, 16), (200, 1024, 1280, 7, 64)])
def test_noalloc_matches_workspace_entry(fmt, M, K, N, L, r):
    """Two noalloc calls back to back on one stream, on two different batches
    (activations, indices and mask) through the same weights: each result is
    bitwise the result of epilora_layer_forward with a workspace of its own.
    Both entry points enqueue the same kernels, so any leftover or overlap in
    the shared static scratch would show as a difference."""
    p1, w, gx1 = _inputs(fmt, M, K, N, L, r, seed=M + K)
    p2 = make_projection(M, K, N, L, r, seed=M + K + 1, idx_mode="uniform", mask_mode="random", device="cuda")
    gx2 = T.nvfp4_global_scale(p2.X) if fmt == NVFP4 else None
    p2.A, p2.B = p1.A, p1.B
    assert not torch.equal(p1.X, p2.X)
    st_ref = status_buf()
    refs = [T.layer_forward(p.X, w, p.A, p.B, p.idx, p.mask, x_global_scale=g, status=st_ref)
            for p, g in ((p1, gx1), (p2, gx2))]
    torch.cuda.synchronize()
    assert int(st_ref.item()) == 0

    Y1 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    Y2 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = status_buf()
    before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    assert _noalloc(fmt, p1, w, gx1, Y1, st) == E.EPILORA_OK
    assert _noalloc(fmt, p2, w, gx2, Y2, st) == E.EPILORA_OK
    torch.cuda.synchronize()
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == before
    assert int(st.item()) == 0
    assert torch.equal(Y1, refs[0])
    assert torch.equal(Y2, refs[1])
    ok, info = O.y_within_tolerance(np32(Y1), np32(refs[0]).astype(np.float64))
    assert ok, info


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
def test_noalloc_base_only(fmt):
    M, K, N = 5, 2048, 512
    p, w, gx = _inputs(fmt, M, K, N, 1, 16, seed=3)
    ref = T.layer_forward(p.X, w, x_global_scale=gx)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = status_buf()
    assert _noalloc(fmt, p, w, gx, Y, st, with_adapters=False) == E.EPILORA_OK
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ok, info = O.y_within_tolerance(np32(Y), np32(ref).astype(np.float64))
    assert ok, info


def test_noalloc_refuses_oversize():
    # FP8, M * K = 16 Mi elements: the quantized activations alone exceed the
    # static scratch, so the call must return EPILORA_ERR_WORKSPACE at once
    M, K, N = 1024, 16384, 128
    need = E.epilora_workspace_bytes(FP8, M, K, 16)
    assert need > (8 << 20)
    p, w, _ = _inputs(FP8, M, K, N, 1, 16, seed=5)
    Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = status_buf()
    assert _noalloc(FP8, p, w, None, Y, st) == E.EPILORA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert bool((Y == 0).all())
