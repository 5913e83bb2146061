"""The single-kernel decode path (one persistent launch per fused call for a
few tokens) vs the oracle: shapes whose weight tiles are split between many
thread blocks, ragged weight tiles, a K tail inside the last 128-byte unit,
grids smaller than the GPU, every rank, 1..8 tokens with as many adapters,
masks and inactive tokens; the quantized activations it used and the shrink's
partial sums it left in the workspace; the no-adapter identities; back-to-back
calls sharing a workspace."""
import numpy as np
import pytest
import torch

import precision_gemm_token_gb300 as E
from oracle import epilora_oracle as O
from precision_gemm_token_gb300 import tensors as T
from synth import make_projection

from .gpu_util import (FP8, NVFP4, assert_y_close, ensure_lib, fused_s_partials, np32, npu8, run_case,
                       same_codes_e2m1_packed, same_codes_e4m3, status_buf)

pytestmark = pytest.mark.gpu

SYNC_BYTES = 2360576   # EPILORA_WORKSPACE_SYNC_BYTES: the head (counters, tagged exchange regions)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()
    # the single kernel for both formats (the automatic policy gives NVFP4
    # calls to the shrink grid and the GEMM)
    prev = E.epilora_set_decode_path(E.DECODE_PATH_SINGLE)
    yield
    E.epilora_set_decode_path(prev)


CASES = [
    # M, K, N, L, r, idx_mode, mask_mode       (what it exercises)
    (1, 4096, 4096, 1, 64, "single", "all"),     # o projection: every tile split over ~5 blocks
    (1, 14336, 512, 1, 64, "single", "all"),     # long K, 4 tiles over ~150 blocks
    (8, 2048, 1040, 8, 16, "uniform", "all"),    # 8 tokens, ragged last weight tile (16 rows)
    (5, 1024, 2048, 3, 32, "uniform", "random"),  # mask 0 and no-adapter tokens
    (2, 4096, 768, 2, 128, "uniform", "all"),    # rank 128
    (1, 512, 16, 1, 64, "single", "all"),        # one 16-row tile: a grid of 4 blocks
    (3, 2048, 6144, 4, 16, "uniform", "all"),    # qkv-like width
]


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,L,r,idx_mode,mask_mode", CASES)
def test_single_kernel_matches_oracle(fmt, M, K, N, L, r, idx_mode, mask_mode):
    assert E.epilora_layer_forward_kernels(fmt, M, K, r) == 1
    y, ref, bound, _ = run_case(fmt, M, K, N, L, r, seed=M * 31 + K + N, idx_mode=idx_mode, mask_mode=mask_mode)
    assert_y_close(y, ref, bound, what=(fmt, M, K, N, r))


def test_single_kernel_fp8_k_tail():
    """FP8 with K not a multiple of 128: the last weight unit is zero-filled
    past K by the copy engine and the quantized rows are zero there."""
    for K in (160, 416):
        assert E.epilora_layer_forward_kernels(FP8, 3, K, 16) == 1
        y, ref, bound, _ = run_case(FP8, 3, K, 384, 2, 16, seed=K)
        assert_y_close(y, ref, bound, what=K)


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
def test_single_kernel_base_only(fmt):
    y, ref, bound, _ = run_case(fmt, 4, 2048, 1152, 2, 16, seed=77, use_adapter=False)
    assert_y_close(y, ref, bound)


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
def test_single_kernel_no_adapter_cases_are_bit_exact_base(fmt):
    p = make_projection(5, 1024, 640, 4, 32, seed=17)
    X, W = p.X.cuda(), p.W.cuda()
    w = T.quantize_weight(W, fmt)
    gx = T.nvfp4_global_scale(X) if fmt == NVFP4 else None
    A, B, idx, mask = p.A.cuda(), p.B.cuda(), p.idx.cuda(), p.mask.cuda()
    base = T.layer_forward(X, w, x_global_scale=gx)
    for Yc in (T.layer_forward(X, w, A, torch.zeros_like(B), idx, mask, x_global_scale=gx),
               T.layer_forward(X, w, A, B, idx, torch.zeros_like(mask), x_global_scale=gx),
               T.layer_forward(X, w, A, B, torch.full_like(idx, -1), mask, x_global_scale=gx)):
        assert torch.equal(Yc.float(), base.float())


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,r", [(1, 4096, 2048, 64), (6, 2048, 1024, 32)])
def test_single_kernel_workspace_contents(fmt, M, K, N, r):
    """The activation codes and scales the kernel used (each thread block
    stores the K range it quantized; together they cover the rows) are the
    oracle's bit for bit; the shrink's partial sums over K slices, added in
    part order, are the oracle's S within fp32 rounding; the launch counter
    at bytes [16, 24) of the workspace has moved on by 256 and the rest of
    the counter block is untouched."""
    L = 3
    p = make_projection(M, K, N, L, r, seed=M + K, idx_mode="uniform", device="cuda")
    w = T.quantize_weight(p.W, fmt)
    gx_t = T.nvfp4_global_scale(p.X) if fmt == NVFP4 else None
    ws = T.LayerWorkspace(p.X.device)
    buf = ws.get(fmt, M, K, r)
    buf.fill_(0)
    st = status_buf()
    T.layer_forward(p.X, w, p.A, p.B, p.idx, p.mask, x_global_scale=gx_t, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(buf[16:24].view(torch.int64).item()) == 256    # one launch
    assert int(buf[:16].count_nonzero().item()) == 0 and int(buf[24:256].count_nonzero().item()) == 0
    x, A, B = p.X.float().cpu().numpy(), p.A.float().cpu().numpy(), p.B.float().cpu().numpy()
    idx, mask = p.idx.cpu().numpy(), p.mask.cpu().numpy()
    r256 = lambda v: (v + 255) // 256 * 256  # noqa: E731
    off = SYNC_BYTES
    if fmt == FP8:
        wq, sw = O.quant_fp8_rows(p.W.float().cpu().numpy())
        ref = O.layer_fp8(x, wq, sw, A, B, idx, mask)
        assert same_codes_e4m3(npu8(buf[off:off + M * K].view(M, K)), ref["xq"]).all()
        o2 = off + r256(M * K)
        assert (np32(buf[o2:o2 + 4 * M].view(torch.float32)) == ref["sx"]).all()
    else:
        Wn = p.W.float().cpu().numpy()
        gw = O.nvfp4_global_scale(Wn)
        wq, sbw = O.quant_nvfp4_rows(Wn, gw)
        ref = O.layer_nvfp4(x, O.nvfp4_global_scale(x), wq, sbw, gw, A, B, idx, mask)
        assert same_codes_e2m1_packed(npu8(buf[off:off + M * K // 2].view(M, K // 2)), ref["xq"]).all()
        o2 = off + r256(M * K // 2)
        assert (npu8(buf[o2:o2 + M * K // 16].view(M, K // 16)) == ref["sbx"]).all()
    n_parts = min(8, -(-K // 1024))
    parts = fused_s_partials(buf, fmt, M, K, r)
    S = parts.sum(dim=0) if n_parts == 1 else parts[0].clone()
    for q in range(1, n_parts):
        S += parts[q]
    act = O.active_tokens(idx, mask, L)
    S_ref = ref["S"][act]
    err = np.abs(np32(S).astype(np.float64)[act] - S_ref).max()
    assert err <= 1e-5 * max(1.0, float(np.abs(S_ref).max())) + 1e-6, err


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
def test_single_kernel_chain_shares_workspace(fmt):
    """Single-kernel calls of different shapes back to back on one stream
    (each a programmatic dependent of the one before, sharing the workspace
    counters), eagerly and replayed from a CUDA graph three times: bitwise
    equal to isolated calls; the launch counter ends at 256 per launch."""
    shapes = [(1, 4096, 6144, 1, 64), (1, 4096, 4096, 1, 64), (1, 4096, 28672, 1, 64), (1, 14336, 4096, 1, 64),
              (4, 2048, 1024, 3, 16)]
    cases = []
    for i, (M, K, N, L, r) in enumerate(shapes):
        p = make_projection(M, K, N, L, r, seed=90 + i, device="cuda")
        w = T.quantize_weight(p.W, fmt)
        gx = T.nvfp4_global_scale(p.X) if fmt == NVFP4 else None
        ref = T.layer_forward(p.X, w, p.A, p.B, p.idx, p.mask, x_global_scale=gx)
        cases.append((p, w, gx, ref))
    torch.cuda.synchronize()
    ws = T.LayerWorkspace("cuda")
    for M, K, N, L, r in shapes:
        ws.get(fmt, M, K, r)
    outs = [torch.empty_like(c[3]) for c in cases]

    def run(stream=None):
        for (p, w, gx, _), Y in zip(cases, outs):
            T.layer_forward(p.X, w, p.A, p.B, p.idx, p.mask, x_global_scale=gx, workspace=ws, Y=Y, stream=stream)

    run()
    torch.cuda.synchronize()
    for c, Y in zip(cases, outs):
        assert torch.equal(Y, c[3])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(s)
    for _ in range(3):
        for Y in outs:
            Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for c, Y in zip(cases, outs):
            assert torch.equal(Y, c[3])
    assert int(ws.buf[16:24].view(torch.int64).item()) == 256 * 4 * len(shapes)   # 1 eager run + 3 replays


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    """A wait that runs out, made on the host: with the library's test hook on,
    the shrink items of the single kernel publish nothing, so every thread
    block that finishes a tile waits for S until its bounded wait gives up
    (about a second). 2 tokens at rank 128 over 8 K slices make 512 items,
    more than thread blocks (every block takes several). The call returns
    EPILORA_ERR_TIMEOUT in the status word, every block still exits (the
    launch counter moves on by 256), and with the hook off the next call on
    the same stream and workspace is correct."""
    M, K, N, L, r = 2, 8192, 1024, 2, 128
    assert E.epilora_layer_forward_kernels(FP8, M, K, r) == 1
    p = make_projection(M, K, N, L, r, seed=5, device="cuda")
    w = T.quantize_weight(p.W, FP8)
    ref = T.layer_forward(p.X, w, p.A, p.B, p.idx, p.mask)
    ws = T.LayerWorkspace("cuda")
    buf = ws.get(FP8, M, K, r)
    st = status_buf()
    torch.cuda.synchronize()
    E.epilora_test_drop_shrink_results(True)
    try:
        T.layer_forward(p.X, w, p.A, p.B, p.idx, p.mask, workspace=ws, status=st)
        torch.cuda.synchronize()
    finally:
        E.epilora_test_drop_shrink_results(False)
    assert int(st.item()) == E.EPILORA_ERR_TIMEOUT
    assert int(buf[16:24].view(torch.int64).item()) == 256
    st.zero_()
    Y = T.layer_forward(p.X, w, p.A, p.B, p.idx, p.mask, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(Y, ref)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_single_kernel_fp8_codes_bit_exact_over_magnitudes(seed):
    """The single kernel's FP8 activation codes and scales against the
    oracle's IEEE-division quantizer, bit for bit, on rows whose values span
    many binades (log-uniform magnitudes, random signs, exact zeros, values
    that land on E4M3 rounding ties), including a row whose scale is below
    2^-100."""
    rng = np.random.default_rng(100 + seed)
    M, K, N = 4, 4096, 256
    mag = np.exp2(rng.uniform(-30, 12, (M, K)))
    x = (np.sign(rng.standard_normal((M, K))) * mag).astype(np.float32)
    x[1] *= np.float32(1e-3)
    x[2, ::7] = 0.0
    # row 3: tiny values (amax ~ 1e-33: scale < 2^-100)
    x[3] = (rng.standard_normal(K) * 1e-34).astype(np.float32)
    X = torch.from_numpy(x).to(torch.bfloat16).cuda()
    xr = X.float().cpu().numpy()
    # ties: half-way values between E4M3 neighbours after the scale
    amax0 = float(np.abs(xr[0]).max())
    s0 = np.float32(np.float32(amax0) / np.float32(448.0))
    for j, code_mid in enumerate((1.0625, 2.125, 9.0 / 8 * 3, 0.5 + 1.0 / 32)):
        v = torch.tensor([code_mid * float(s0)], dtype=torch.float32).to(torch.bfloat16)
        X[0, 10 + j] = v.item()
    xr = X.float().cpu().numpy()
    assert E.epilora_layer_forward_kernels(FP8, M, K, 0) == 1
    W = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    w = T.quantize_weight(W, FP8)
    ws = T.LayerWorkspace("cuda")
    buf = ws.get(FP8, M, K, 0)
    T.layer_forward(X, w, workspace=ws)
    torch.cuda.synchronize()
    codes, sc = O.quant_fp8_rows(xr)
    off = SYNC_BYTES
    r256 = lambda v: (v + 255) // 256 * 256  # noqa: E731
    got = npu8(buf[off:off + M * K].view(M, K))
    got_s = np32(buf[off + r256(M * K):off + r256(M * K) + 4 * M].view(torch.float32))
    assert (got_s == sc).all()
    assert same_codes_e4m3(got, codes).all(), np.argwhere(~same_codes_e4m3(got, codes))[:5]
