"""Pins of the oracle's quantizers, shrink, base GEMM and epilogue against
closed forms, exact integer arithmetic, the explicit merged update W + BA,
token permutation, the no-adapter cases and brute-force loops on tiny shapes."""
import numpy as np
import pytest

from oracle import epilora_oracle as O
from oracle import fpformats as F
from synth import make_projection
from synth.inputs import small_integer_tensor

F32 = np.float32


# ------------------------------------------------------------------ quantizers
def test_fp8_quant_closed_form_row():
    # amax 448 -> scale exactly 1, codes are the values themselves
    x = np.array([[448.0, 1.0, -2.0, 0.5, 0.0, -448.0, 3.0, 0.015625]], F32)
    codes, s = O.quant_fp8_rows(x)
    assert s[0] == F32(1.0)
    assert (F.e4m3_decode(codes[0]) == x[0]).all()


def test_fp8_quant_amax_element_hits_448_and_scale_formula():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((64, 512)).astype(F32) * F32(3)
    codes, s = O.quant_fp8_rows(x)
    for t in range(64):
        j = np.argmax(np.abs(x[t]))
        assert (codes[t, j] & 0x7F) == 0x7E                 # +-448
        assert s[t] == F32(F32(np.abs(x[t]).max()) / F32(448.0))
        # every code within range and dequantized values within half a step
        xh = F.e4m3_decode(codes[t]) * np.float64(s[t])
        assert np.all(np.abs(xh - x[t]) <= np.abs(x[t]) / 16 + np.float64(s[t]) * 2.0 ** -10)


def test_fp8_quant_zero_row_uses_floor():
    codes, s = O.quant_fp8_rows(np.zeros((2, 32), F32))
    assert (codes & 0x7F == 0).all()
    assert s[0] == F32(F32(1e-12) / F32(448.0))


def test_fp8_quant_roundtrip_exact():
    """quantize -> dequantize in fp32 -> requantize with the same scale gives
    the same codes."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((32, 256)).astype(F32)
    codes, s = O.quant_fp8_rows(x)
    xh = (F.e4m3_decode(codes).astype(F32) * s[:, None]).astype(F32)
    codes2 = F.e4m3_encode(F.e4m3_round((xh / s[:, None]).astype(F32)))
    same = (codes == codes2) | ((codes & 0x7F) == 0) & ((codes2 & 0x7F) == 0)
    assert same.all()


def test_nvfp4_quant_closed_form_blocks():
    x = np.zeros((1, 32), F32)
    x[0, :4] = [6.0, 3.0, -1.5, 0.5]           # block 0: amax 6
    x[0, 16:20] = [1.0, -1.0, 0.5, 0.0]        # block 1: amax 1
    for g in (F32(1.0), F32(2.0), F32(0.5)):
        packed, sb = O.quant_nvfp4_rows(x, g)
        codes = F.unpack_e2m1(packed)[0]
        # block 0: sb = e4m3(6/6*g) = g (exact), codes = x * g / g
        assert F.e4m3_decode(sb[0, 0]) == g
        assert (F.e2m1_decode(codes[:4]) == x[0, :4]).all()
        # block 1: sb = e4m3(1/6*g); amax element encodes to 6
        assert F.e2m1_decode(codes[16]) == 6.0 and F.e2m1_decode(codes[17]) == -6.0
        xh = O.dequant_nvfp4_rows(packed, sb, g)
        assert np.allclose(xh[0, :4], x[0, :4], rtol=0, atol=0)


def test_nvfp4_quant_zero_block_and_amax_hits_6():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((16, 128)).astype(F32)
    x[3, 16:32] = 0
    g = O.nvfp4_global_scale(x)
    assert g == F32(F32(2688.0) / F32(np.abs(x).max()))
    packed, sb = O.quant_nvfp4_rows(x, g)
    codes = F.unpack_e2m1(packed)
    assert sb[3, 1] == 0 and (codes[3, 16:32] & 7 == 0).all()
    xb = np.abs(x).reshape(16, 8, 16)
    for t in range(16):
        for b in range(8):
            if sb[t, b] == 0:
                continue
            j = np.argmax(xb[t, b])
            assert (codes[t, b * 16 + j] & 7) == 7                  # |code| = 6


def test_nvfp4_global_scale_closed_forms():
    """The encode multiplier g = 448 * 6 / amax (reading O3) through what it
    implies rather than its formula: a tensor whose amax is 2688 = 448 * 6
    needs no scaling (g = 1), one whose amax is 6 gets g = 448 exactly, and in
    every case the block holding the tensor's amax gets the largest E4M3 block
    scale (code 0x7E = 448), its amax element the E2M1 code +-6, and that
    element dequantizes back to the amax. A dropped factor 6, a missing 448
    or a decode-direction g (amax / 2688) breaks one of these."""
    rng = np.random.default_rng(21)
    base = rng.standard_normal((4, 64)).astype(F32)
    for amax, g_want in ((F32(2688.0), F32(1.0)), (F32(6.0), F32(448.0)), (F32(0.75), F32(3584.0))):
        x = (base / np.abs(base).max() * amax).astype(F32)
        t, k = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        x[t, k] = amax if x[t, k] > 0 else -amax
        g = O.nvfp4_global_scale(x)
        assert g == g_want, (amax, g)
        packed, sb = O.quant_nvfp4_rows(x, g)
        codes = F.unpack_e2m1(packed)
        assert sb[t, k // 16] == 0x7E                          # block scale 448: E4M3's largest finite
        assert F.e4m3_decode(sb[t, k // 16]) == 448.0
        assert (codes[t, k] & 7) == 7                          # |E2M1 code| = 6
        xh = O.dequant_nvfp4_rows(packed, sb, g)
        assert xh[t, k] == np.float64(x[t, k])                 # 6 * 448 / g = amax exactly here
    # any tensor: the amax block's scale is 448, the others no larger
    x = (rng.standard_normal((8, 256)) * 0.37).astype(F32)
    g = O.nvfp4_global_scale(x)
    _, sb = O.quant_nvfp4_rows(x, g)
    t, k = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sb[t, k // 16] == 0x7E
    assert (F.e4m3_decode(sb) <= 448.0).all()


def test_nvfp4_dequant_error_bound():
    """Each element is within half an E2M1 step of the block-scaled grid, the
    block scale within half an E4M3 step: |x - xhat| <= |x|/4*(1+1/16) + slack."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((8, 256)).astype(F32)
    g = O.nvfp4_global_scale(x)
    packed, sb = O.quant_nvfp4_rows(x, g)
    xh = O.dequant_nvfp4_rows(packed, sb, g)
    step = F.e4m3_decode(sb).repeat(16, axis=1) / np.float64(g)   # scale of one E2M1 unit
    assert np.all(np.abs(xh - x) <= 0.5 * 2 * step + 1e-12)      # half of the coarsest step (2 units)


# ------------------------------------------------------------------ shrink
def test_shrink_integer_inputs_exact():
    rng = np.random.default_rng(4)
    M, K, L, r = 7, 96, 3, 8
    x = small_integer_tensor(rng, (M, K), -8, 8)
    A = small_integer_tensor(rng, (L, r, K), -8, 8)
    idx = np.array([0, 2, 1, -1, 2, 0, 1], np.int32)
    mask = np.array([1, 1, 0, 1, 1, 1, 1], np.uint8)
    S = O.shrink(x, A, idx, mask)
    xi, Ai = x.astype(np.int64), A.astype(np.int64)
    for t in range(M):
        if idx[t] < 0 or mask[t] == 0:
            assert (S[t] == 0).all()
        else:
            assert (S[t] == Ai[idx[t]] @ xi[t]).all()


def test_shrink_bruteforce_loops():
    rng = np.random.default_rng(5)
    M, K, L, r = 3, 16, 2, 4
    x = rng.standard_normal((M, K))
    A = rng.standard_normal((L, r, K))
    idx = np.array([1, 0, 1], np.int32)
    S = O.shrink(x, A, idx, None)
    for t in range(M):
        for j in range(r):
            s = 0.0
            for k in range(K):
                s += x[t, k] * A[idx[t], j, k]
            assert abs(S[t, j] - s) <= 1e-12 * (1 + abs(s))


# ------------------------------------------------------------------ base GEMM
def test_fp8_base_integer_codes_exact():
    """Small-integer E4M3 codes with unit scales reduce to an integer matmul."""
    rng = np.random.default_rng(6)
    M, N, K = 5, 24, 64
    xi = rng.integers(-8, 9, (M, K))
    wi = rng.integers(-8, 9, (N, K))
    xq = F.e4m3_encode(xi.astype(np.float64))
    wq = F.e4m3_encode(wi.astype(np.float64))
    base = O.base_gemm_fp8(xq, np.ones(M, F32), wq, np.ones(N, F32))
    assert (base == (xi @ wi.T)).all()
    # scales multiply through exactly for powers of two
    base2 = O.base_gemm_fp8(xq, np.full(M, 0.5, F32), wq, np.full(N, 4.0, F32))
    assert (base2 == 2 * (xi @ wi.T)).all()
    # column subset
    cols = np.array([3, 0, 17])
    assert (O.base_gemm_fp8(xq, np.ones(M, F32), wq, np.ones(N, F32), cols) == (xi @ wi[cols].T)).all()


def test_nvfp4_base_integer_codes_exact():
    rng = np.random.default_rng(7)
    M, N, K = 3, 8, 64
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    xv = rng.choice(vals, (M, K)) * rng.choice([-1, 1], (M, K))
    wv = rng.choice(vals, (N, K)) * rng.choice([-1, 1], (N, K))
    xq = F.pack_e2m1(F.e2m1_encode(xv))
    wq = F.pack_e2m1(F.e2m1_encode(wv))
    one = F.e4m3_encode(np.ones((M, K // 16)))
    onew = F.e4m3_encode(np.ones((N, K // 16)))
    base = O.base_gemm_nvfp4(xq, one, F32(1), wq, onew, F32(1))
    assert (base == xv @ wv.T).all()
    two = F.e4m3_encode(np.full((N, K // 16), 2.0))
    assert (O.base_gemm_nvfp4(xq, one, F32(4), wq, two, F32(0.5)) == xv @ wv.T).all()


# ------------------------------------------------------------------ epilogue/layer
def _small_layer(seed=0, M=6, K=64, N=48, L=3, r=8):
    p = make_projection(M, K, N, L, r, seed=seed)
    x = p.X.float().numpy()
    w = p.W.float().numpy()
    wq, sw = O.quant_fp8_rows(w)
    return p, x, wq, sw


def test_delta_equals_merged_update_W_plus_BA():
    """The adapter term equals x . (B_l A_l)^T with the explicit N x K product."""
    p, x, wq, sw = _small_layer()
    A, B = p.A.float().numpy().astype(np.float64), p.B.float().numpy().astype(np.float64)
    idx, mask = p.idx.numpy(), p.mask.numpy()
    ref = O.layer_fp8(x, wq, sw, A, B, idx, mask)
    for t in range(x.shape[0]):
        BA = B[idx[t]] @ A[idx[t]]                   # N x K merged update
        d = BA @ x[t].astype(np.float64)
        assert np.allclose(ref["delta"][t], d, rtol=1e-12, atol=1e-15)


def test_slices_equal_per_slice_merged_updates():
    """Multi-slice projection: the columns of slice s take x . (B_l[cols_s]
    A_l[slice s rows])^T with the explicit merged product of that slice, and
    a single slice is the ordinary layer."""
    rng = np.random.default_rng(7)
    M, K, N, L, r = 5, 64, 48, 3, 4
    ends = [16, 40, 48]
    x = rng.standard_normal((M, K)).astype(np.float32)
    W = (0.02 * rng.standard_normal((N, K))).astype(np.float32)
    A = rng.standard_normal((L, len(ends) * r, K)) / np.sqrt(K)
    B = 0.01 * rng.standard_normal((L, N, r))
    idx = np.array([0, 2, -1, 1, 2])
    mask = np.array([1, 1, 1, 0, 1], dtype=np.uint8)
    wq, sw = O.quant_fp8_rows(W)
    ref = O.layer_fp8(x, wq, sw, A, B, idx, mask, slice_end=ends)
    start = 0
    for s_i, end in enumerate(ends):
        for t in range(M):
            if idx[t] < 0 or mask[t] == 0:
                assert (ref["delta"][t, start:end] == 0).all()
                continue
            BA = B[idx[t], start:end] @ A[idx[t], s_i * r:(s_i + 1) * r]
            assert np.allclose(ref["delta"][t, start:end], BA @ x[t].astype(np.float64), rtol=1e-12, atol=1e-15)
        start = end
    one = O.layer_fp8(x, wq, sw, A[:, :r], B, idx, mask, slice_end=[N])
    assert (one["Y"] == O.layer_fp8(x, wq, sw, A[:, :r], B, idx, mask)["Y"]).all()


def test_zero_B_mask_and_negative_index_give_base():
    p, x, wq, sw = _small_layer(seed=1)
    A, B = p.A.float().numpy(), p.B.float().numpy()
    idx, mask = p.idx.numpy(), p.mask.numpy()
    base = O.base_gemm_fp8(*O.quant_fp8_rows(x), wq, sw)
    assert (O.layer_fp8(x, wq, sw, A, np.zeros_like(B), idx, mask)["Y"] == base).all()
    assert (O.layer_fp8(x, wq, sw, A, B, idx, np.zeros_like(mask))["Y"] == base).all()
    assert (O.layer_fp8(x, wq, sw, A, B, np.full_like(idx, -1), mask)["Y"] == base).all()
    # idx >= L is treated as no adapter too
    assert (O.layer_fp8(x, wq, sw, A, B, np.full_like(idx, 3), mask)["Y"] == base).all()


def test_token_permutation_commutes():
    p, x, wq, sw = _small_layer(seed=2, M=9)
    A, B = p.A.float().numpy(), p.B.float().numpy()
    idx, mask = p.idx.numpy(), np.array([1, 0, 1, 1, 1, 0, 1, 1, 1], np.uint8)
    perm = np.random.default_rng(0).permutation(9)
    y = O.layer_fp8(x, wq, sw, A, B, idx, mask)["Y"]
    yp = O.layer_fp8(x[perm], wq, sw, A, B, idx[perm], mask[perm])["Y"]
    assert (yp == y[perm]).all()


def test_layer_bruteforce_loops_fp8():
    """Triple loops straight from the definitions on a tiny case."""
    rng = np.random.default_rng(8)
    M, K, N, L, r = 3, 32, 5, 2, 4
    x = rng.standard_normal((M, K)).astype(F32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(F32)
    A = rng.standard_normal((L, r, K)) / np.sqrt(K)
    B = rng.standard_normal((L, N, r)) * 0.01
    idx = np.array([1, -1, 0], np.int32)
    mask = np.array([1, 1, 1], np.uint8)
    wq, sw = O.quant_fp8_rows(w)
    ref = O.layer_fp8(x, wq, sw, A, B, idx, mask)
    for t in range(M):
        amax = max(abs(float(v)) for v in x[t])
        st = F32(F32(amax) / F32(448))
        for n in range(N):
            acc = 0.0
            for k in range(K):
                qx = float(F.e4m3_round(np.array([F32(x[t, k] / st)]))[0])
                acc += qx * float(st) * float(F.e4m3_decode(np.array([wq[n, k]]))[0]) * float(sw[n])
            dl = 0.0
            if idx[t] >= 0:
                for j in range(r):
                    h = sum(float(x[t, k]) * A[idx[t], j, k] for k in range(K))
                    dl += h * B[idx[t], n, j]
            want = acc + dl
            assert abs(ref["Y"][t, n] - want) <= 1e-12 * (1 + abs(want)), (t, n)


def test_layer_nvfp4_matches_dequantized_product():
    p = make_projection(4, 64, 32, 2, 4, seed=3)
    x, w = p.X.float().numpy(), p.W.float().numpy()
    gw, gx = O.nvfp4_global_scale(w), O.nvfp4_global_scale(x)
    wq, sbw = O.quant_nvfp4_rows(w, gw)
    A, B = p.A.float().numpy(), p.B.float().numpy()
    ref = O.layer_nvfp4(x, gx, wq, sbw, gw, A, B, p.idx.numpy(), p.mask.numpy())
    xq, sbx = O.quant_nvfp4_rows(x, gx)
    xh = O.dequant_nvfp4_rows(xq, sbx, gx)
    wh = O.dequant_nvfp4_rows(wq, sbw, gw)
    assert np.allclose(ref["base"], xh @ wh.T, rtol=1e-12, atol=1e-14)


def test_tolerance_helper():
    ref = np.array([1.0, -2.0, 0.0, 1e-6])
    ok, _ = O.y_within_tolerance(ref * (1 + 1e-3), ref)
    assert ok
    ok, _ = O.y_within_tolerance(ref * 1.05, ref)
    assert not ok


# ------------------------------------------------------------------ stored FP8 adapters
def test_adapter_fp8_integer_rows_exact():
    """Rows whose amax is 448 get scale 1: small integers are their own codes,
    the dequantized table equals the original, and the layer's adapter term on
    integer activations is the exact integer product."""
    rng = np.random.default_rng(31)
    L, r, K, N, M = 3, 8, 64, 48, 5
    A = rng.integers(-8, 9, (L, r, K)).astype(F32)
    A[:, :, 0] = 448.0
    B = rng.integers(-4, 5, (L, N, r)).astype(F32)
    B[:, :, 1] = -448.0
    for T in (A, B):
        codes, sc = O.quant_adapter_fp8(T)
        assert (sc == F32(1.0)).all()
        assert (O.dequant_adapter_fp8(codes, sc) == T).all()
    x = rng.integers(-3, 4, (M, K)).astype(F32)
    idx = np.array([0, 2, -1, 1, 2], np.int32)
    S = O.shrink(x, O.dequant_adapter_fp8(*O.quant_adapter_fp8(A)), idx, None)
    d = O.expand(S, O.dequant_adapter_fp8(*O.quant_adapter_fp8(B)), idx, None)
    xi, Ai, Bi = x.astype(np.int64), A.astype(np.int64), B.astype(np.int64)
    for t in range(M):
        if idx[t] < 0:
            assert (d[t] == 0).all()
            continue
        want = Bi[idx[t]] @ (Ai[idx[t]] @ xi[t])
        assert (d[t] == want.astype(np.float64)).all()


def test_adapter_fp8_roundtrip_and_error_bound():
    """Requantizing the dequantized table gives the same codes; every element
    is within half an E4M3 step of the original (relative 2^-4 for normal
    values, plus the subnormal step 2^-9 times the row scale)."""
    rng = np.random.default_rng(32)
    T = (rng.standard_normal((4, 16, 256)) / 16).astype(F32)
    codes, sc = O.quant_adapter_fp8(T)
    deq = O.dequant_adapter_fp8(codes, sc)
    c2, s2 = O.quant_adapter_fp8(deq.astype(F32))
    assert (s2 == sc).all()
    assert ((c2 == codes) | (((c2 & 0x7F) == 0) & ((codes & 0x7F) == 0))).all()
    err = np.abs(deq - T)
    assert (err <= np.abs(T) / 16 + sc[:, :, None].astype(np.float64) * 2.0 ** -10).all()
    # each row's amax element is exactly +-448 scaled
    j = np.argmax(np.abs(T), axis=2)
    assert ((np.take_along_axis(codes, j[:, :, None], 2) & 0x7F) == 0x7E).all()


def test_adapter_fp8_layer_is_merged_update_of_dequantized_tables():
    """The layer with stored adapters equals the base plus x (B^ A^)^T from the
    explicit merged N x K matrix of the dequantized tables (tiny shapes)."""
    p = make_projection(6, 64, 40, 3, 16, seed=33)
    x, W = p.X.float().numpy(), p.W.float().numpy()
    Ah = O.dequant_adapter_fp8(*O.quant_adapter_fp8(p.A.float().numpy()))
    Bh = O.dequant_adapter_fp8(*O.quant_adapter_fp8(p.B.float().numpy()))
    wq, sw = O.quant_fp8_rows(W)
    ref = O.layer_fp8(x, wq, sw, Ah, Bh, p.idx.numpy(), p.mask.numpy())
    act = O.active_tokens(p.idx.numpy(), p.mask.numpy(), 3)
    for t in range(6):
        merged = Bh[int(p.idx[t])] @ Ah[int(p.idx[t])] if act[t] else np.zeros((40, 64))
        want = merged @ x[t].astype(np.float64)
        assert np.allclose(ref["delta"][t], want, rtol=1e-12, atol=1e-15)
    # zero adapters: codes 0, the floor scale, no adapter term
    codes, sc = O.quant_adapter_fp8(np.zeros((2, 4, 32), F32))
    assert ((codes & 0x7F) == 0).all() and (sc == F32(F32(1e-12) / F32(448.0))).all()

