"""Parity at the full Llama-shaped sizes, through the fused one-call layer
(the call the benchmark times), on sampled outputs.

Every output Y[t, n] depends only on token t's activations, weight row n and
token t's adapter, so the oracle recomputes a sample of tokens (all of them
up to 64) and of weight rows exactly as it would the whole layer. Checked:
the weight codes / scales of the sampled rows and the activation codes /
scales that the fused call left in its workspace (bit-exact), the partial
sums of S it left there and S from the standalone shrink (both within fp32
rounding of the oracle's S), and Y on the sampled grid within the layer
tolerance.

Cases: the 8B decode layer at M = 1 (one rank-64 adapter) and at M = 32 (32
tenants), FP8; the 8B layer with an NVFP4 base and 128 resident adapters
(Zipf indices) at M = 1, 8, 32, 512 and ranks 16 / 64 / 128; the 70B layer,
FP8, 512 rank-16 adapters, 64 decode tokens plus one 2048-token prefill chunk
with the prefill-only mask."""
import numpy as np
import pytest
import torch

from oracle import epilora_oracle as O
from precision_gemm_token_gb300 import tensors as T
from synth import LLAMA8B_PROJECTIONS, LLAMA70B_PROJECTIONS, make_projection

from .gpu_util import (FP8, NVFP4, ensure_lib, fused_s_partials, np32, npu8, same_codes_e2m1_packed, same_codes_e4m3,
                       status_buf)

pytestmark = pytest.mark.gpu

P8 = {n: (K, N) for n, K, N in LLAMA8B_PROJECTIONS}
P70 = {n: (K, N) for n, K, N in LLAMA70B_PROJECTIONS}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


SYNC_BYTES = 2360576   # EPILORA_WORKSPACE_SYNC_BYTES: the head (counters, tagged exchange regions)


def _r256(v):
    return (v + 255) // 256 * 256


def _sample(n, k, rng, must=()):
    if n <= k:
        return np.arange(n)
    s = set(int(v) for v in must if 0 <= v < n) | {0, n - 1}
    s |= set(int(v) for v in rng.choice(n, size=k - len(s), replace=False))
    return np.array(sorted(s))[:max(k, len(s))]


def _amax(t: torch.Tensor) -> np.ndarray:
    # a max is exact in any order; only the oracle's formula turns it into g
    return np.array([t.abs().max().float().item()], dtype=np.float32)


def run_fullsize(fmt, K, N, M, L, r, idx_mode, seed, mask_mode="all", n_decode=0, n_rows=48, n_cols=64):
    rng = np.random.default_rng(seed)
    p = make_projection(M, K, N, L, r, seed=seed, idx_mode=idx_mode, mask_mode=mask_mode, n_decode=n_decode,
                        device="cuda")
    w = T.quantize_weight(p.W, fmt)
    gx_t = T.nvfp4_global_scale(p.X) if fmt == NVFP4 else None
    ws = T.LayerWorkspace(p.X.device)
    # zero-filled: partial-sum slots the shrink leaves unused then read as 0
    ws.get(fmt, M, K, r, N).zero_()
    st = status_buf()
    Y = T.layer_forward(p.X, w, p.A, p.B, p.idx, p.mask, x_global_scale=gx_t, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    rows = _sample(M, n_rows, rng, must=(n_decode - 1, n_decode))
    cols = _sample(N, n_cols, rng, must=(N - 128, N - 127))
    idx_all, mask_all = p.idx.cpu().numpy(), p.mask.cpu().numpy()
    idx, mask = idx_all[rows], mask_all[rows]
    # only the adapters the sampled tokens use, renumbered
    used = np.unique(idx[(idx >= 0) & (idx < L)])
    remap = {int(l): i for i, l in enumerate(used)}
    idx_s = np.array([remap.get(int(l), -1) for l in idx], dtype=np.int32)
    ui = torch.from_numpy(used.astype(np.int64)).cuda()
    A_s = p.A[ui].float().cpu().numpy() if used.size else np.zeros((1, r, K), np.float32)
    B_s = p.B[ui][:, torch.from_numpy(cols).cuda(), :].float().cpu().numpy() if used.size else \
        np.zeros((1, cols.size, r), np.float32)
    if not used.size:
        idx_s[:] = -1
    x = p.X[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    Wn = p.W[torch.from_numpy(cols).cuda()].float().cpu().numpy()
    cols_t = torch.from_numpy(cols).cuda()
    rows_t = torch.from_numpy(rows).cuda()
    buf = ws.buf
    # workspace: the head (a launch counter that grows by 256 per single-kernel
    # call, nothing else in its first 256 bytes), Xq, scales, S (room for
    # min(8, ceil(K / 1024)) partial sums), and for more than 32 tokens the
    # adapter-sorted row order: row q holds token perm[q]
    off_xq = SYNC_BYTES
    assert int(buf[16:24].view(torch.int64).item()) % 256 == 0
    assert int(buf[:16].count_nonzero().item()) == 0 and int(buf[24:256].count_nonzero().item()) == 0
    xq_bytes = M * K if fmt == FP8 else M * K // 2
    sc_bytes = 4 * M if fmt == FP8 else M * K // 16
    off_perm = off_xq + _r256(xq_bytes) + _r256(sc_bytes) + _r256(M * r * 4 * min(8, -(-K // 1024)))
    if M > 32:
        perm = buf[off_perm:off_perm + 4 * M].view(torch.int32).cpu().numpy()
        assert np.array_equal(np.sort(perm), np.arange(M))
        keys = np.where((idx_all >= 0) & (idx_all < L) & (mask_all != 0), idx_all, L)
        assert np.array_equal(perm, np.lexsort((np.arange(M), keys)))
        row_of = np.empty(M, dtype=np.int64)
        row_of[perm] = np.arange(M)
        qrows_t = torch.from_numpy(row_of[rows]).cuda()
    else:
        qrows_t = torch.from_numpy(rows).cuda()
    if fmt == FP8:
        wq, sw = O.quant_fp8_rows(Wn)
        assert same_codes_e4m3(npu8(w.codes[cols_t]), wq).all()
        assert (np32(w.scale[cols_t]) == sw).all()
        ref = O.layer_fp8(x, wq, sw, A_s, B_s, idx_s, mask)
        xq_gpu = buf[off_xq:off_xq + M * K].view(M, K)[qrows_t]
        sx_gpu = buf[off_xq + _r256(M * K):off_xq + _r256(M * K) + 4 * M].view(torch.float32)[qrows_t]
        assert same_codes_e4m3(npu8(xq_gpu), ref["xq"]).all()
        assert (np32(sx_gpu) == ref["sx"]).all()
    else:
        gw = O.nvfp4_global_scale(_amax(p.W))
        gx = O.nvfp4_global_scale(_amax(p.X))
        assert np32(w.global_scale)[0] == gw and np32(gx_t)[0] == gx
        wq, sbw = O.quant_nvfp4_rows(Wn, gw)
        assert (npu8(w.block_scale[cols_t]) == sbw).all()
        assert same_codes_e2m1_packed(npu8(w.codes[cols_t]), wq).all()
        ref = O.layer_nvfp4(x, gx, wq, sbw, gw, A_s, B_s, idx_s, mask)
        xq_gpu = buf[off_xq:off_xq + M * K // 2].view(M, K // 2)[qrows_t]
        o2 = off_xq + _r256(M * K // 2)
        sb_gpu = buf[o2:o2 + M * K // 16].view(M, K // 16)[qrows_t]
        assert same_codes_e2m1_packed(npu8(xq_gpu), ref["xq"]).all()
        assert (npu8(sb_gpu) == ref["sbx"]).all()
    # S of the same tokens as the fused call left it in its workspace: partial
    # sums over K slices [part][token][r], added here in part order as the
    # GEMM adds them; and from the standalone shrink
    S_ref = ref["S"]
    n_parts = min(8, -(-K // 1024))
    parts = fused_s_partials(buf, fmt, M, K, r)[:, rows_t, :]
    S_fused = parts[0].clone()
    for q in range(1, n_parts):
        S_fused += parts[q]
    S_tol = 1e-5 * max(1.0, float(np.abs(S_ref).max()) if S_ref.size else 1.0) + 1e-6
    for S_gpu in (np32(S_fused).astype(np.float64),
                  np32(T.lora_shrink(p.X, p.A, p.idx, p.mask)[rows_t]).astype(np.float64)):
        s_err = np.abs(S_gpu - S_ref).max() if S_ref.size else 0.0
        assert s_err <= S_tol, s_err
    y = np32(Y[rows_t][:, cols_t])
    ok, info = O.y_within_tolerance(y, ref["Y"])
    assert ok, info
    return info


@pytest.mark.parametrize("proj", list(P8))
def test_8b_decode_m1_fp8_one_adapter(proj):
    K, N = P8[proj]
    run_fullsize(FP8, K, N, M=1, L=1, r=64, idx_mode="single", seed=201)


@pytest.mark.parametrize("proj", list(P8))
def test_8b_decode_m32_fp8_32_tenants(proj):
    K, N = P8[proj]
    run_fullsize(FP8, K, N, M=32, L=32, r=64, idx_mode="per_token", seed=202)


@pytest.mark.parametrize("M,r", [(1, 64), (8, 16), (32, 128), (512, 64)])
@pytest.mark.parametrize("proj", list(P8))
def test_8b_nvfp4_128_adapters_zipf(proj, M, r):
    K, N = P8[proj]
    run_fullsize(NVFP4, K, N, M=M, L=128, r=r, idx_mode="zipf", seed=203 + M)


@pytest.mark.parametrize("proj", list(P70))
def test_70b_fp8_prefill_chunk_and_decode_tokens(proj):
    K, N = P70[proj]
    run_fullsize(FP8, K, N, M=64 + 2048, L=512, r=16, idx_mode="zipf", seed=204, mask_mode="prefill_chunk",
                 n_decode=64)
