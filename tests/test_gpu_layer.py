"""GPU layer (quantizer -> shrink -> tcgen05 GEMM with the LoRA epilogue as
the shrink's programmatic dependent) vs the oracle, on FP8 and NVFP4 bases.

Shapes span several 128-row weight tiles, every token-tile width (16..256
columns), ragged token and weight tails, split-K clusters of 1..8 CTAs, and
the degenerate cases: no adapter, zero B, mask 0, out-of-range index."""
import numpy as np
import pytest
import torch

from oracle import epilora_oracle as O
from oracle import fpformats as F
from precision_gemm_token_gb300 import tensors as T
from synth import make_projection

from .gpu_util import FP8, NVFP4, assert_y_close, ensure_lib, np32, run_case, status_buf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


SHAPES = [
    # M, K, N, L, r        (token tile / split-K it exercises)
    (4, 512, 1024, 4, 16),      # the small parity workload: BT 16, 2-CTA cluster split
    (1, 512, 1024, 1, 64),      # single token
    (4, 256, 1024, 4, 16),      # one K stage per CTA
    (16, 1024, 2048, 8, 32),    # 4-CTA clusters
    (17, 512, 144, 4, 16),      # ragged tokens (BT 32) and a partial 16-row weight tile
    (31, 2048, 256, 2, 128),    # 8-CTA clusters, rank 128
    (32, 4096, 512, 32, 64),    # one token per tenant
    (33, 512, 272, 4, 16),      # BT 64, ragged weight tile
    (100, 512, 384, 5, 32),     # BT 128, no split
    (130, 256, 256, 3, 16),     # BT 256
    (300, 512, 272, 7, 64),     # two 256-token tiles, ragged both ways
    (160, 512, 384, 9, 128),    # wide tiles at rank 128
]


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,L,r", SHAPES)
def test_layer_matches_oracle(fmt, M, K, N, L, r):
    if fmt == NVFP4 and K % 256:
        pytest.skip("NVFP4 GEMM needs K % 256 == 0")
    y, ref, bound, _ = run_case(fmt, M, K, N, L, r, seed=M * 7 + N)
    assert_y_close(y, ref, bound, what=(fmt, M, K, N))


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
def test_layer_mask_prefill_chunk(fmt):
    y, ref, bound, _ = run_case(fmt, 40, 512, 256, 6, 16, seed=5, idx_mode="zipf", mask_mode="prefill_chunk",
                                n_decode=8)
    assert_y_close(y, ref, bound)


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("r", [16, 32, 64, 128])
def test_wide_tiles_prefill_chunk_one_adapter_runs(fmt, r):
    """Wide (256-token) tiles whose columns are long one-adapter runs, mask-0
    decode tokens and a ragged last tile: the one-adapter, no-adapter and
    mixed 16-column chunks of the wide epilogue."""
    y, ref, bound, _ = run_case(fmt, 600, 512, 384, 64, r, seed=11 + r, idx_mode="zipf", mask_mode="prefill_chunk",
                                n_decode=40)
    assert_y_close(y, ref, bound, what=(fmt, r))


WIDE_PERSISTENT = [
    # M, K, N, L, r, idx_mode, mask_mode     (more 256-token tiles than SMs: the
    # persistent two-accumulator kernel for FP8)
    (520, 256, 7168, 8, 16, "uniform", "all"),           # mixed-adapter chunks, ragged token tile
    (520, 256, 7152, 64, 32, "zipf", "prefill_chunk"),   # one-adapter runs, mask-0 tokens, ragged weight tile
    (1000, 512, 5120, 16, 64, "zipf", "all"),            # rank 64
    (520, 256, 3072, 24, 128, "zipf", "all"),            # rank 128 (the two-CTA kernel for both formats)
    (520, 256, 7168, 8, 0, "uniform", "all"),            # no adapter
]


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,L,r,idx_mode,mask_mode", WIDE_PERSISTENT)
def test_wide_grids_larger_than_the_gpu(fmt, M, K, N, L, r, idx_mode, mask_mode):
    use = r > 0
    y, ref, bound, _ = run_case(fmt, M, K, N, L, r if use else 16, seed=3 + r, idx_mode=idx_mode,
                                mask_mode=mask_mode, n_decode=24 if mask_mode == "prefill_chunk" else 0,
                                use_adapter=use)
    assert_y_close(y, ref, bound, what=(fmt, M, N, r))


EPILOGUE_TERM = [
    # M, K, N, L, r, idx_mode, mask_mode    (wide tiles whose epilogue computes the
    # adapter term: a workspace without room for the expand pass)
    (100, 512, 384, 5, 32, "uniform", "all"),            # 128-token tiles, TF32 tensor-core term
    (300, 512, 272, 7, 64, "uniform", "all"),            # CUDA-core term, ragged both ways
    (160, 512, 384, 9, 128, "zipf", "all"),              # rank 128
    (600, 512, 384, 64, 16, "zipf", "prefill_chunk"),    # one-adapter runs, mask-0 tokens
    (1000, 512, 5120, 16, 64, "zipf", "all"),            # persistent FP8 kernel, rank 64
    (80, 6144, 128, 6, 64, "zipf", "prefill_chunk"),     # shrink split over K slices
]


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,L,r,idx_mode,mask_mode", EPILOGUE_TERM)
def test_wide_epilogue_term_matches_oracle(fmt, M, K, N, L, r, idx_mode, mask_mode):
    """The adapter term computed in the GEMM's epilogue (the path a call
    takes when its workspace has no room for the expand pass's fp32 term)."""
    if fmt == NVFP4 and K % 256:
        pytest.skip("NVFP4 GEMM needs K % 256 == 0")
    y, ref, bound, _ = run_case(fmt, M, K, N, L, r, seed=17 + M + r, idx_mode=idx_mode, mask_mode=mask_mode,
                                n_decode=8 if mask_mode == "prefill_chunk" else 0, epilogue_term=True)
    assert_y_close(y, ref, bound, what=(fmt, M, N, r))


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,L,r,idx_mode", [
    (300, 512, 272, 7, 64, "uniform"),     # 128-token tiles (NVFP4), ragged weight tile
    (100, 512, 384, 5, 64, "zipf"),        # 128-token tiles, both formats
    (160, 512, 384, 9, 128, "zipf"),       # rank 128
    (40, 4096, 256, 3, 64, "uniform"),     # few tiles: split-K clusters, the element-wise epilogue
    (33, 512, 208, 40, 32, "uniform"),     # one-token runs, ragged weight tile
    (700, 256, 384, 3, 32, "zipf"),        # runs longer than a round of 32 rows
])
def test_expand_pass_and_epilogue_term_both_match_oracle(fmt, M, K, N, L, r, idx_mode):
    """The same inputs through the expand pass (workspace of
    epilora_layer_workspace_bytes) and through the epilogue's own term: both
    within the arithmetic bound of the oracle, and every element of Y the
    same to within that bound of each other."""
    y_x, ref, bound, _ = run_case(fmt, M, K, N, L, r, seed=M + N + r, idx_mode=idx_mode)
    y_e, ref_e, _, _ = run_case(fmt, M, K, N, L, r, seed=M + N + r, idx_mode=idx_mode, epilogue_term=True)
    assert np.array_equal(ref["Y"], ref_e["Y"])
    assert_y_close(y_x, ref, bound, what=("expand", fmt, M, r))
    assert_y_close(y_e, ref, bound, what=("epilogue", fmt, M, r))
    assert (np.abs(y_x.astype(np.float64) - y_e) <= 2 * bound).all()


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,L,r,idx_mode,mask_mode", [
    (48, 4096, 256, 4, 16, "zipf", "prefill_chunk"),      # token blocks over 2 K slices
    (80, 6144, 128, 6, 64, "zipf", "prefill_chunk"),      # rank 64, 3 K slices, ragged last block
    (64, 4096, 256, 8, 32, "uniform", "all"),             # blocks with many adapters: per-token CTAs + zeroed parts
])
def test_wide_shrink_split_over_k(fmt, M, K, N, L, r, idx_mode, mask_mode):
    """More than 32 tokens with K long enough for the shrink to split it:
    token-block CTAs on the tensor cores write partial sums per K slice (and
    zero them for blocks taken token by token); the GEMM adds them in order."""
    y, ref, bound, _ = run_case(fmt, M, K, N, L, r, seed=M + r, idx_mode=idx_mode, mask_mode=mask_mode,
                                n_decode=8 if mask_mode == "prefill_chunk" else 0)
    assert_y_close(y, ref, bound, what=(fmt, M, K, r))


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,r,ends", [
    (4, 512, 640, 16, [384, 512, 640]),          # decode tile, split-K cluster, three slices
    (24, 1024, 384, 64, [256, 384]),             # 32-token decode tile, two slices, rank 64
    (300, 512, 640, 32, [384, 512, 640]),        # wide tiles (two CTAs per SM), three slices
    (520, 256, 26112, 16, [18432, 22272, 26112]),   # more tiles than 4 per SM: persistent kernel (FP8)
])
def test_multi_slice_projection(fmt, M, K, N, r, ends):
    """Fused projections with one adapter pair per slice (qkv, gate_up): the
    columns of slice s use its rank-r block of A and of S."""
    L = 6
    rng = np.random.default_rng(M + N)
    X = torch.tensor(rng.standard_normal((M, K)), dtype=torch.bfloat16)
    W = torch.tensor(0.02 * rng.standard_normal((N, K)), dtype=torch.bfloat16)
    A = torch.tensor(rng.standard_normal((L, len(ends) * r, K)) / np.sqrt(K), dtype=torch.bfloat16)
    B = torch.tensor(0.01 * rng.standard_normal((L, N, r)), dtype=torch.bfloat16)
    idx = torch.tensor(rng.integers(-1, L, size=M), dtype=torch.int32)
    mask = torch.tensor(rng.integers(0, 2, size=M), dtype=torch.uint8)
    x, Wn, An, Bn = (t.float().numpy() for t in (X, W, A, B))
    w = T.quantize_weight(W.cuda(), fmt)
    st = status_buf()
    if fmt == FP8:
        wq, sw = O.quant_fp8_rows(Wn)
        ref = O.layer_fp8(x, wq, sw, An, Bn, idx.numpy(), mask.numpy(), slice_end=ends)
        xv = F.e4m3_decode(ref["xq"]) * ref["sx"][:, None].astype(np.float64)
        wv = F.e4m3_decode(wq) * sw[:, None].astype(np.float64)
        gx = None
    else:
        gw = O.nvfp4_global_scale(Wn)
        wq, sbw = O.quant_nvfp4_rows(Wn, gw)
        gxv = O.nvfp4_global_scale(x)
        gx = torch.tensor([gxv], dtype=torch.float32, device="cuda")
        ref = O.layer_nvfp4(x, gxv, wq, sbw, gw, An, Bn, idx.numpy(), mask.numpy(), slice_end=ends)
        xv = O.dequant_nvfp4_rows(ref["xq"], ref["sbx"], gxv)
        wv = O.dequant_nvfp4_rows(wq, sbw, gw)
    Y = T.layer_forward_slices(X.cuda(), w, A.cuda(), B.cuda(), idx.cuda(), ends, mask=mask.cuda(),
                               x_global_scale=gx, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # bound: bf16 rounding + fp32 accumulation of every product term
    mag = np.abs(xv) @ np.abs(wv).T
    S = np.abs(ref["S"])
    act = O.active_tokens(idx.numpy(), mask.numpy(), L)
    start = 0
    for s_i, end in enumerate(ends):
        for t in np.nonzero(act)[0]:
            mag[t, start:end] += np.abs(Bn[int(idx[t]), start:end]) @ S[t, s_i * r:(s_i + 1) * r]
        start = end
    bound = 2.0 ** -8 * np.abs(ref["Y"]) + 1e-5 * mag + 1e-30
    assert_y_close(np32(Y), ref, bound, what=(fmt, M, N, ends))


def test_fp8_integer_codes_exact():
    """Rows whose amax is 448 quantize with scale 1; with small-integer values
    the codes are those integers, the fp32 accumulation is exact and Y must be
    the bf16 rounding of the exact integer result."""
    rng = np.random.default_rng(11)
    M, K, N = 20, 512, 384
    x = rng.integers(-2, 3, (M, K)).astype(np.float32)
    w = rng.integers(-2, 3, (N, K)).astype(np.float32)
    x[:, 0] = 448.0          # the 448s meet small values only: |Y| < 2^12
    w[:, 1] = 448.0
    X = torch.from_numpy(x).to(torch.bfloat16).cuda()
    W = torch.from_numpy(w).to(torch.bfloat16).cuda()
    wt = T.quantize_weight(W, FP8)
    assert (np32(wt.scale) == 1.0).all()
    Y = T.layer_forward(X, wt)
    exact = x.astype(np.int64) @ w.astype(np.int64).T
    want = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).float().numpy()
    assert (np32(Y) == want).all()


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
def test_no_adapter_cases_are_bit_exact_base(fmt):
    p = make_projection(24, 512, 512, 4, 16, seed=7)
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
@pytest.mark.parametrize("M", [7, 29, 300])   # single kernel; one decode tile; several adapter-sorted wide tiles
def test_permutation_and_determinism(fmt, M):
    p = make_projection(M, 1024, 640, 5, 32, seed=8, mask_mode="random")
    X, W = p.X.cuda(), p.W.cuda()
    w = T.quantize_weight(W, fmt)
    gx = T.nvfp4_global_scale(X) if fmt == NVFP4 else None
    A, B, idx, mask = p.A.cuda(), p.B.cuda(), p.idx.cuda(), p.mask.cuda()
    Y1 = T.layer_forward(X, w, A, B, idx, mask, x_global_scale=gx)
    Y2 = T.layer_forward(X, w, A, B, idx, mask, x_global_scale=gx)
    assert torch.equal(Y1, Y2)
    perm = torch.randperm(M, generator=torch.Generator().manual_seed(1)).cuda()
    Yp = T.layer_forward(X[perm].contiguous(), w, A, B, idx[perm].contiguous(), mask[perm].contiguous(),
                         x_global_scale=gx)
    assert torch.equal(Yp, Y1[perm])


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,L,r", [(16, 1024, 512, 4, 64),
                                       (2, 14336, 256, 2, 64),     # shrink split over 4 K slices
                                       (1, 8192, 256, 1, 128)])    # 2 K slices, rank 128
def test_adapter_contribution_with_zero_base(fmt, M, K, N, L, r):
    """All-zero weights: Y is bf16 of the adapter term alone."""
    y, ref, _, _ = run_case(fmt, M, K, N, L, r, seed=9, zero_w=True)
    d = ref["delta"]
    assert np.linalg.norm(y - d) / np.linalg.norm(d) <= 1e-2


def test_gemm_with_h_given_matches_fused():
    """The standalone GEMM (S already in memory, ordinary launch) equals the
    two-kernel fused call bit for bit (12 tokens: more than the single-kernel
    path takes)."""
    import precision_gemm_token_gb300 as E
    assert E.epilora_layer_forward_kernels(FP8, 12, 1024, 32) == 2
    p = make_projection(12, 1024, 512, 4, 32, seed=10)
    X, W = p.X.cuda(), p.W.cuda()
    w = T.quantize_weight(W, FP8)
    A, B, idx, mask = p.A.cuda(), p.B.cuda(), p.idx.cuda(), p.mask.cuda()
    Yf = T.layer_forward(X, w, A, B, idx, mask)
    Xq, sx = T.quant_act(X, FP8)
    S = T.lora_shrink(X, A, idx, mask)
    torch.cuda.synchronize()
    Yg = T.gemm_lora_epilogue(Xq, sx, w, 12, 1024, S=S, B=B, idx=idx, mask=mask, pdl_dependent=False)
    assert torch.equal(Yf, Yg)


@pytest.mark.parametrize("fmt,M,K,N,r", [
    (FP8, 8, 2048, 512, 32),        # decode tile
    (FP8, 520, 256, 26112, 16),     # more than 4 wide tiles per SM: the persistent kernel
    (NVFP4, 8, 2048, 512, 32),
])
def test_standalone_shrink_then_dependent_gemm(fmt, M, K, N, r):
    """epilora_lora_shrink, then on the same stream epilora_gemm_lora_epilogue
    launched as its programmatic dependent: the GEMM may start while the
    shrink still runs, but reads S, idx and mask only after it; Y equals an
    ordinary launch's bit for bit (S starts out as NaN each time)."""
    import precision_gemm_token_gb300 as E
    p = make_projection(M, K, N, 6, r, seed=M + N)
    X, W = p.X.cuda(), p.W.cuda()
    A, B, idx, mask = p.A.cuda(), p.B.cuda(), p.idx.cuda(), p.mask.cuda()
    w = T.quantize_weight(W, fmt)
    gx = T.nvfp4_global_scale(X) if fmt == NVFP4 else None
    Xq, xs = T.quant_act(X, fmt, global_scale=gx)
    st = status_buf()
    outs = []
    for pdl in (False, True):
        S = torch.full((M, r), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        rc = E.epilora_lora_shrink(X, M, K, X.stride(0), A, A.shape[0], r, idx, mask, S, st, None)
        assert rc == E.EPILORA_OK
        outs.append(T.gemm_lora_epilogue(Xq, xs, w, M, K, S=S, B=B, idx=idx, mask=mask, x_global_scale=gx,
                                         pdl_dependent=pdl, status=st))
        torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert not torch.isnan(outs[0].float()).any()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("M,r", [(6, 16), (40, 64)])   # decode tile; wide tiles with the expand pass
def test_out_of_range_index_in_gemm(M, r):
    p = make_projection(M, 512, 256, 3, r, seed=12)
    idx = p.idx.clone()
    idx[2] = 5
    st = status_buf()
    X, W = p.X.cuda(), p.W.cuda()
    w = T.quantize_weight(W, FP8)
    Y = T.layer_forward(X, w, p.A.cuda(), p.B.cuda(), idx.cuda(), p.mask.cuda(), status=st)
    base = T.layer_forward(X, w)
    torch.cuda.synchronize()
    assert int(st.item()) == -1
    assert torch.equal(Y[2], base[2])


def test_empty_batch_is_a_noop():
    w = T.quantize_weight(torch.randn(256, 512, device="cuda").to(torch.bfloat16), FP8)
    X = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    Y = T.layer_forward(X, w)
    assert Y.shape == (0, 256)


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
def test_back_to_back_calls_share_workspace_and_replay_in_a_graph(fmt):
    """Consecutive fused calls (each a programmatic dependent of the one
    before) that share one workspace, eagerly and captured in a CUDA graph,
    give bitwise the results of isolated calls."""
    shapes = [(1, 4096, 1024, 1, 64), (3, 2048, 4096, 2, 16), (1, 14336, 1024, 1, 64), (1, 4096, 6144, 1, 64),
              (17, 1024, 512, 4, 32)]
    cases = []
    for i, (M, K, N, L, r) in enumerate(shapes):
        p = make_projection(M, K, N, L, r, seed=40 + i)
        X, W = p.X.cuda(), p.W.cuda()
        w = T.quantize_weight(W, fmt)
        gx = T.nvfp4_global_scale(X) if fmt == NVFP4 else None
        args = (X, w, p.A.cuda(), p.B.cuda(), p.idx.cuda(), p.mask.cuda(), gx)
        ref = T.layer_forward(*args[:6], x_global_scale=gx)       # own workspace
        torch.cuda.synchronize()
        cases.append((args, ref))
    ws = T.LayerWorkspace("cuda")
    for M, K, N, L, r in shapes:
        ws.get(fmt, M, K, r, N)
    outs = [torch.empty_like(ref) for _, ref in cases]

    def run(stream=None):
        for (args, _), Y in zip(cases, outs):
            T.layer_forward(*args[:6], x_global_scale=args[6], workspace=ws, Y=Y, stream=stream)

    run()
    torch.cuda.synchronize()
    for (_, ref), Y in zip(cases, outs):
        assert torch.equal(Y, ref)
    for Y in outs:
        Y.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(s)
    for _ in range(2):
        for Y in outs:
            Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for (_, ref), Y in zip(cases, outs):
            assert torch.equal(Y, ref)


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M", [1, 40])
def test_prepared_layer_equals_layer_forward(fmt, M):
    """tensors.PreparedLayer (arguments bound once) re-enqueues the same call:
    with X's contents refreshed in place between calls, Y equals a fresh
    layer_forward call bit for bit, on the single-kernel and the two-kernel
    paths."""
    p = make_projection(M, 2048, 1024, 3, 16, seed=11 + M, device="cuda")
    w = T.quantize_weight(p.W, fmt)
    X = p.X.clone()
    gx = T.nvfp4_global_scale(X) if fmt == NVFP4 else None
    Y = torch.empty((M, 1024), dtype=torch.bfloat16, device="cuda")
    st = status_buf()
    call = T.PreparedLayer(X, w, p.A, p.B, p.idx, p.mask, x_global_scale=gx, workspace=T.LayerWorkspace("cuda"),
                           status=st, Y=Y)
    g = torch.Generator(device="cuda").manual_seed(M)
    for step in range(3):
        X.copy_(torch.randn(X.shape, generator=g, device="cuda").to(torch.bfloat16))
        if gx is not None:
            gx.copy_(T.nvfp4_global_scale(X))
        call()
        ref = T.layer_forward(X, w, p.A, p.B, p.idx, p.mask, x_global_scale=gx)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(Y, ref), (fmt, M, step)
