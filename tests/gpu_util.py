"""Helpers shared by the GPU parity tests: run the CUDA path through the C
ABI, run the oracle on the same seeded inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import precision_gemm_token_gb300 as E
from oracle import epilora_oracle as O
from oracle import fpformats as F
from precision_gemm_token_gb300 import tensors as T
from synth import make_projection

FP8, NVFP4 = E.FMT_FP8, E.FMT_NVFP4


def ensure_lib():
    E.build()
    E.load()


def np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def npu8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.uint8)


def same_codes_e4m3(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Equal codes, or both a zero of either sign."""
    return (a == b) | (((a & 0x7F) == 0) & ((b & 0x7F) == 0))


def same_codes_e2m1_packed(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ua, ub = F.unpack_e2m1(a), F.unpack_e2m1(b)
    return (ua == ub) | (((ua & 0x7) == 0) & ((ub & 0x7) == 0))


def status_buf(dev="cuda"):
    return torch.zeros(1, dtype=torch.int32, device=dev)


def oracle_weight(fmt, W_np, g=None):
    if fmt == FP8:
        return O.quant_fp8_rows(W_np)
    return O.quant_nvfp4_rows(W_np, g)


def check_weight_parity(fmt, w: T.QuantWeight, W_np: np.ndarray, rows=None):
    """GPU weight quantization == oracle's, bit for bit (on `rows` if given)."""
    if fmt == FP8:
        wq, sw = O.quant_fp8_rows(W_np if rows is None else W_np)
        gq = npu8(w.codes if rows is None else w.codes[rows])
        gs = np32(w.scale if rows is None else w.scale[rows])
        assert same_codes_e4m3(gq, wq).all()
        assert (gs == sw).all()
        return wq, sw, None
    raise NotImplementedError


def tight_bound(ref: dict, xv: np.ndarray, wv: np.ndarray, B: np.ndarray, idx, mask, cols=None):
    """|y - ref| allowed by the arithmetic: bf16 output rounding (2^-8 of |ref|
    covers RNE with margin) plus fp32 accumulation of every product term
    (1e-5 of the sum of their magnitudes covers K <= 28672 fp32 additions)."""
    mag = np.abs(xv) @ np.abs(wv).T
    S = np.abs(ref["S"])
    Bc = B if cols is None else B[:, cols, :]
    act = O.active_tokens(idx, mask, B.shape[0])
    for t in np.nonzero(act)[0]:
        mag[t] += np.abs(Bc[int(idx[t])]) @ S[t]
    return 2.0 ** -8 * np.abs(ref["Y"]) + 1e-5 * mag + 1e-30


def assert_y_close(y: np.ndarray, ref: dict, bound: np.ndarray | None = None, what=""):
    ok, info = O.y_within_tolerance(y, ref["Y"])
    assert ok, (what, info)
    if bound is not None:
        err = np.abs(y.astype(np.float64) - ref["Y"])
        bad = err > bound
        assert not bad.any(), (what, np.argwhere(bad)[:5], float((err / bound).max()))


def layer_forward_epilogue_term(X, w, A, B, idx, mask, x_global_scale=None, status=None):
    """epilora_layer_forward with a workspace of epilora_workspace_bytes: the
    GEMM's epilogue computes the adapter term itself (no expand pass)."""
    M, K = X.shape
    L, r = A.shape[0], A.shape[1]
    need = E.epilora_workspace_bytes(w.fmt, M, K, r)
    buf = torch.zeros(need, dtype=torch.uint8, device=X.device)
    Y = torch.empty((M, w.N), dtype=torch.bfloat16, device=X.device)
    E.check(E.epilora_layer_forward(w.fmt, M, w.N, K, X, X.stride(0), w.codes, w.scale, w.block_scale,
                                    w.global_scale, x_global_scale, A, B, L, r, idx, mask, Y, Y.stride(0), buf,
                                    need, status, None), "layer_forward")
    return Y


def run_case(fmt, M, K, N, L, r, seed=0, idx_mode="uniform", mask_mode="all", n_decode=0, zero_w=False,
             use_adapter=True, epilogue_term=False):
    """Run GPU and oracle on the same inputs; returns (Y_gpu np, ref dict, bound, inputs).
    epilogue_term: the workspace leaves no room for the expand pass, so that
    wide tiles compute the adapter term in the GEMM's epilogue."""
    p = make_projection(M, K, N, L, r, seed=seed, idx_mode=idx_mode, mask_mode=mask_mode, n_decode=n_decode)
    W = torch.zeros_like(p.W) if zero_w else p.W
    Xg, Wg = p.X.cuda(), W.cuda()
    w = T.quantize_weight(Wg, fmt)
    x, Wn = p.X.float().numpy(), W.float().numpy()
    A, B = p.A.float().numpy(), p.B.float().numpy()
    idx, mask = p.idx.numpy(), p.mask.numpy()
    gx = None
    if fmt == FP8:
        wq, sw = O.quant_fp8_rows(Wn)
        assert same_codes_e4m3(npu8(w.codes), wq).all() and (np32(w.scale) == sw).all()
        ref = O.layer_fp8(x, wq, sw, A, B, idx, mask) if use_adapter else O.layer_fp8(
            x, wq, sw, A, np.zeros_like(B), idx, mask)
        xv = F.e4m3_decode(ref["xq"]) * ref["sx"][:, None].astype(np.float64)
        wv = F.e4m3_decode(wq) * sw[:, None].astype(np.float64)
    else:
        gw = O.nvfp4_global_scale(Wn)
        wq, sbw = O.quant_nvfp4_rows(Wn, gw)
        assert np32(w.global_scale)[0] == gw
        assert (npu8(w.block_scale) == sbw).all() and same_codes_e2m1_packed(npu8(w.codes), wq).all()
        gxv = O.nvfp4_global_scale(x)
        gx = torch.tensor([gxv], dtype=torch.float32, device="cuda")
        Bref = B if use_adapter else np.zeros_like(B)
        ref = O.layer_nvfp4(x, gxv, wq, sbw, gw, A, Bref, idx, mask)
        xv = O.dequant_nvfp4_rows(ref["xq"], ref["sbx"], gxv)
        wv = O.dequant_nvfp4_rows(wq, sbw, gw)
    st = status_buf()
    if use_adapter and epilogue_term:
        Y = layer_forward_epilogue_term(Xg, w, p.A.cuda(), p.B.cuda(), p.idx.cuda(), p.mask.cuda(), x_global_scale=gx,
                                        status=st)
    elif use_adapter:
        Y = T.layer_forward(Xg, w, p.A.cuda(), p.B.cuda(), p.idx.cuda(), p.mask.cuda(), x_global_scale=gx, status=st)
    else:
        Y = T.layer_forward(Xg, w, x_global_scale=gx, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bound = tight_bound(ref, xv, wv, B if use_adapter else np.zeros_like(B), idx, mask)
    return np32(Y), ref, bound, (p, w, gx)


HEAD_BYTES = 2360576          # EPILORA_WORKSPACE_SYNC_BYTES
HEAD_S_OFFSET = 1280 + 256 * 8 * 128 * 8   # tagged S partial sums of the single-kernel path in the head


def _r256(v):
    return (v + 255) // 256 * 256


def fused_s_partials(buf: torch.Tensor, fmt: int, M: int, K: int, r: int) -> torch.Tensor:
    """The partial sums of S over K slices [n_parts, M, r] that a fused call
    left in its workspace `buf` (zero where a slice was not used, if the
    workspace was zero-filled): in the head as (value, tag) pairs for the
    single-kernel path, else as floats after the quantized activations."""
    n_parts = min(8, -(-K // 1024))
    if E.epilora_layer_forward_kernels(fmt, M, K, r) == 1:
        w = buf[HEAD_S_OFFSET:HEAD_S_OFFSET + n_parts * M * r * 8].view(torch.int32).view(n_parts, M, r, 2)
        return w[..., 0].contiguous().view(torch.float32)
    xq_bytes = M * K if fmt == FP8 else M * K // 2
    sc_bytes = 4 * M if fmt == FP8 else M * K // 16
    off = HEAD_BYTES + _r256(xq_bytes) + _r256(sc_bytes)
    return buf[off:off + n_parts * M * r * 4].view(torch.float32).view(n_parts, M, r)

