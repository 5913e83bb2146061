"""Oracle for the multi-tenant LoRA linear layer of a decode step.

TEST INFRASTRUCTURE ONLY: a plain, slow, obviously correct CPU restatement of
what the layer computes. Only tests, the smoke check and the benchmark's CPU
baseline may import it; the CUDA library never does, and this module shares
no code, table or constant generator with it.

What is computed (EpiLoRA: "Fusing Many LoRA Adapters into Low-Precision GEMMs
for Serving and RL"):

  Y[t, :] = dequant( Q(X)[t, :] . Q(W)^T ) + mask[t] * (x_t . A[idx_t]^T) . B[idx_t]^T

* §Background and motivation › The cost of the separate adapter path:
  the down-projection ("shrink") is h = x A^T and the up-projection
  ("expand") adds h B^T to the layer's output.
* §Design › Multi-adapter kernels › K1 and K2: activations are quantized per
  token for the low-precision base GEMM, h is computed from the *bf16*
  activations (not the quantized ones), and the GEMM's epilogue applies the
  weight and activation scales and then adds each token's h B^T.
* PreFT: Prefill-only finetuning (pith.science summary), Core claim: the
  adapter is applied to prefill tokens only and skipped for decode tokens ->
  a per-token mask.

Readings taken where the pages are silent (each also listed in the design
notes):
  O1  FP8 per-token scale: s_t = fl32(max(amax_t, 1e-12) / 448) with IEEE
      round-to-nearest float32 division; code = E4M3_rn_satfinite(fl32(x / s_t)).
  O2  an all-zero token row uses the 1e-12 floor, so its codes are all 0.
  O3  NVFP4: g is the encode multiplier (g = 448*6 / amax of the tensor);
      per 16-element block: sb = E4M3_rn_sat(fl32(fl32(amax_b / 6) * g));
      sb == 0 -> all codes 0, else code = E2M1_rn_sat(fl32(x * fl32(g / sb)));
      dequantized value = E2M1(code) * sb / g.
  O5  FP8 weight scale per output channel, fp32 [N].
  O6  h is kept in (at least) fp32; here fp64.
  O7  the LoRA scaling alpha/r is folded into B.
  O8  idx < 0 or mask == 0 -> base only.
  O10 a prefill chunk is one request: one adapter for all of its tokens.

Everything downstream of the quantizers is float64.
"""
from __future__ import annotations

import numpy as np

from .fpformats import (
    e2m1_decode,
    e2m1_encode,
    e2m1_round,
    e4m3_decode,
    e4m3_encode,
    e4m3_round,
    pack_e2m1,
    unpack_e2m1,
)

F32 = np.float32
FP8_AMAX_FLOOR = F32(1e-12)
E4M3_MAX_F32 = F32(448.0)
E2M1_MAX_F32 = F32(6.0)
NVFP4_BLOCK = 16


# ---------------------------------------------------------------------------
# S1: per-token FP8 activation quantizer (readings O1, O2)
# ---------------------------------------------------------------------------
def quant_fp8_rows(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Quantize each row of x (float32 holding bf16 values) to E4M3 codes.

    Returns (codes uint8 [M, K], scale float32 [M]). The same routine gives the
    per-output-channel weight scales when applied to W's rows (reading O5).
    """
    x = np.asarray(x, dtype=F32)
    amax = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], F32)
    scale = (np.maximum(amax, FP8_AMAX_FLOOR) / E4M3_MAX_F32).astype(F32)   # float32 division
    q = (x / scale[:, None]).astype(F32)                                     # float32 division
    codes = e4m3_encode(e4m3_round(q))
    return codes, scale


def dequant_fp8_rows(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    return e4m3_decode(codes) * np.asarray(scale, dtype=np.float64)[:, None]


# ---------------------------------------------------------------------------
# S1': NVFP4 activation (and weight) quantizer (reading O3)
# ---------------------------------------------------------------------------
def nvfp4_global_scale(t: np.ndarray) -> np.float32:
    """Encode multiplier g = 448 * 6 / amax(t) of a whole tensor (reading O3)."""
    amax = F32(np.max(np.abs(np.asarray(t, dtype=F32)))) if np.size(t) else F32(0)
    amax = max(amax, FP8_AMAX_FLOOR)
    return F32(F32(448.0 * 6.0) / F32(amax))


def quant_nvfp4_rows(x: np.ndarray, g) -> tuple[np.ndarray, np.ndarray]:
    """Quantize rows of x into packed E2M1 codes and E4M3 block scales.

    Returns (packed uint8 [M, K/2] with element 2i in the low nibble,
             block scale codes uint8 [M, K/16]).
    """
    x = np.asarray(x, dtype=F32)
    M, K = x.shape
    if K % NVFP4_BLOCK:
        raise ValueError("K must be a multiple of 16")
    g = F32(g)
    xb = x.reshape(M, K // NVFP4_BLOCK, NVFP4_BLOCK)
    amax_b = np.max(np.abs(xb), axis=2)
    t1 = (amax_b / F32(6.0)).astype(F32)                     # float32 division
    t2 = (t1 * g).astype(F32)                                 # float32 multiply
    sb = e4m3_round(t2)                                       # block scale value (>= 0)
    sb_code = e4m3_encode(sb)
    sb32 = sb.astype(F32)                                     # exact (E4M3 fits float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(sb32 > 0, (g / np.where(sb32 > 0, sb32, F32(1))).astype(F32), F32(0))
    q = (xb * inv[:, :, None]).astype(F32)                    # float32 multiply
    vals = np.where(sb[:, :, None] > 0, e2m1_round(q), 0.0)
    codes = e2m1_encode(vals).reshape(M, K)
    return pack_e2m1(codes), sb_code


def dequant_nvfp4_rows(packed: np.ndarray, sb_code: np.ndarray, g) -> np.ndarray:
    codes = unpack_e2m1(packed)
    M, K = codes.shape
    v = e2m1_decode(codes).reshape(M, K // NVFP4_BLOCK, NVFP4_BLOCK)
    sb = e4m3_decode(sb_code)
    return (v * sb[:, :, None]).reshape(M, K) / np.float64(F32(g))


# ---------------------------------------------------------------------------
# S2: multi-adapter shrink, h_t = x_t . A[idx_t]^T from the bf16 activations
# ---------------------------------------------------------------------------
def active_tokens(idx: np.ndarray, mask: np.ndarray | None, L: int) -> np.ndarray:
    """Token t carries its adapter iff mask[t] != 0 and 0 <= idx[t] < L (O8)."""
    idx = np.asarray(idx, dtype=np.int64)
    act = (idx >= 0) & (idx < L)
    if mask is not None:
        act &= np.asarray(mask) != 0
    return act


def shrink(x: np.ndarray, A: np.ndarray, idx: np.ndarray, mask: np.ndarray | None) -> np.ndarray:
    """S [M, r] in float64; rows of tokens without an adapter are zero."""
    x = np.asarray(x, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    L, r, _ = A.shape
    M = x.shape[0]
    S = np.zeros((M, r), dtype=np.float64)
    act = active_tokens(idx, mask, L)
    for t in np.nonzero(act)[0]:
        S[t] = A[int(idx[t])] @ x[t]
    return S


# ---------------------------------------------------------------------------
# S3 + S5: base GEMM on dequantized operands, epilogue adds S . B[idx]^T
# ---------------------------------------------------------------------------
def expand(S: np.ndarray, B: np.ndarray, idx: np.ndarray, mask: np.ndarray | None) -> np.ndarray:
    """delta [M, N] = S[t] . B[idx_t]^T for active tokens, else 0."""
    B = np.asarray(B, dtype=np.float64)
    L, N, r = B.shape
    M = S.shape[0]
    delta = np.zeros((M, N), dtype=np.float64)
    act = active_tokens(idx, mask, L)
    for t in np.nonzero(act)[0]:
        delta[t] = B[int(idx[t])] @ S[t]
    return delta


def base_gemm_fp8(xq: np.ndarray, sx: np.ndarray, wq: np.ndarray, sw: np.ndarray,
                  cols: np.ndarray | None = None) -> np.ndarray:
    """base[t, n] = sum_k xhat[t,k] * what[n,k] for FP8 operands (float64).

    The code products are summed first (exact in float64 for these formats and
    sizes) and the two scales applied after, which is the same real number.
    `cols` restricts the output to those columns n.
    """
    xv = e4m3_decode(xq)
    if cols is not None:
        wq, sw = wq[cols], np.asarray(sw)[cols]
    wv = e4m3_decode(wq)
    acc = xv @ wv.T
    return acc * np.asarray(sx, dtype=np.float64)[:, None] * np.asarray(sw, dtype=np.float64)[None, :]


def base_gemm_nvfp4(xq: np.ndarray, sbx: np.ndarray, gx, wq: np.ndarray, sbw: np.ndarray, gw,
                    cols: np.ndarray | None = None) -> np.ndarray:
    """base[t, n] for NVFP4 operands: block-scaled code products summed, then
    divided by both encode multipliers (reading O3)."""
    xv = dequant_nvfp4_rows(xq, sbx, F32(1.0))          # code * block scale, no global scale
    if cols is not None:
        wq, sbw = wq[cols], sbw[cols]
    wv = dequant_nvfp4_rows(wq, sbw, F32(1.0))
    acc = xv @ wv.T
    return acc / (np.float64(F32(gx)) * np.float64(F32(gw)))


def expand_slices(S: np.ndarray, B: np.ndarray, idx: np.ndarray, mask: np.ndarray | None,
                  slice_end) -> np.ndarray:
    """Multi-slice projection (EpiLoRA, §Design › Multi-adapter kernels: a
    fused projection carries one adapter per slice): output columns
    [slice_end[s-1], slice_end[s]) take S[:, s*r:(s+1)*r] . B[idx_t][n]^T."""
    B = np.asarray(B, dtype=np.float64)
    r = B.shape[2]
    delta = np.zeros((S.shape[0], B.shape[1]), dtype=np.float64)
    start = 0
    for s, end in enumerate(slice_end):
        delta[:, start:end] = expand(S[:, s * r:(s + 1) * r], B[:, start:end, :], idx, mask)
        start = end
    return delta


def layer_fp8(x: np.ndarray, wq: np.ndarray, sw: np.ndarray, A: np.ndarray, B: np.ndarray,
              idx: np.ndarray, mask: np.ndarray | None, cols: np.ndarray | None = None, slice_end=None):
    """Reference Y (float64) of the FP8 layer plus its parts.

    Returns dict(Y, base, delta, S, xq, sx). With `cols`, Y/base/delta hold only
    those output columns. With `slice_end` (no `cols`), A is [L, n * r, K] and
    the columns of slice s use its rank-r block (expand_slices).
    """
    xq, sx = quant_fp8_rows(x)
    base = base_gemm_fp8(xq, sx, wq, sw, cols)
    S = shrink(x, A, idx, mask)
    if slice_end is not None:
        delta = expand_slices(S, B, idx, mask, slice_end)
        return dict(Y=base + delta, base=base, delta=delta, S=S, xq=xq, sx=sx)
    Bc = B if cols is None else np.asarray(B)[:, cols, :]
    delta = expand(S, Bc, idx, mask)
    return dict(Y=base + delta, base=base, delta=delta, S=S, xq=xq, sx=sx)


def layer_nvfp4(x: np.ndarray, gx, wq: np.ndarray, sbw: np.ndarray, gw, A: np.ndarray,
                B: np.ndarray, idx: np.ndarray, mask: np.ndarray | None,
                cols: np.ndarray | None = None, slice_end=None):
    xq, sbx = quant_nvfp4_rows(x, gx)
    base = base_gemm_nvfp4(xq, sbx, gx, wq, sbw, gw, cols)
    S = shrink(x, A, idx, mask)
    if slice_end is not None:
        delta = expand_slices(S, B, idx, mask, slice_end)
        return dict(Y=base + delta, base=base, delta=delta, S=S, xq=xq, sbx=sbx)
    Bc = B if cols is None else np.asarray(B)[:, cols, :]
    delta = expand(S, Bc, idx, mask)
    return dict(Y=base + delta, base=base, delta=delta, S=S, xq=xq, sbx=sbx)


# ---------------------------------------------------------------------------
# Stored low-precision adapters (EpiLoRA, §Design › Multi-adapter kernels ›
# K1 and K2: adapters may be stored in FP8 and dequantized in registers).
# Reading P9: each row of A [L, r, K] (one rank over K) and of B [L, N, r] (one
# output channel over r) is kept as E4M3 codes with one fp32 scale, quantized
# with the arithmetic of the FP8 activation rows (readings O1, O2); the layer
# is the plain layer on the dequantized tables.
# ---------------------------------------------------------------------------
def quant_adapter_fp8(T: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Adapter table [L, R, C] -> (E4M3 codes uint8 [L, R, C], fp32 scale [L, R])."""
    T = np.asarray(T, dtype=F32)
    L, R, C = T.shape
    codes, scale = quant_fp8_rows(T.reshape(L * R, C))
    return codes.reshape(L, R, C), scale.reshape(L, R)


def dequant_adapter_fp8(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """float64 [L, R, C]: code value times its row's scale."""
    L, R, C = codes.shape
    return dequant_fp8_rows(codes.reshape(L * R, C), np.asarray(scale).reshape(L * R)).reshape(L, R, C)


# ---------------------------------------------------------------------------
# Acceptance bar for bf16 outputs (reading O13 of the stated 2e-2 bound)
# ---------------------------------------------------------------------------
def y_within_tolerance(y: np.ndarray, ref: np.ndarray, rel: float = 2e-2) -> tuple[bool, dict]:
    """|y - ref| <= rel * (|ref| + 1e-2 * rms(ref)) elementwise and
    max|y - ref| / max|ref| <= rel."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(y - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bound = rel * (np.abs(ref) + 1e-2 * rms)
    ok_elem = bool(np.all(err <= bound))
    mx = float(np.max(np.abs(ref))) if ref.size else 0.0
    max_rel = float(np.max(err)) / mx if mx > 0 else float(np.max(err)) if err.size else 0.0
    return ok_elem and max_rel <= rel, dict(max_err=float(err.max()) if err.size else 0.0,
                                            max_rel=max_rel, worst_ratio=float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0)
