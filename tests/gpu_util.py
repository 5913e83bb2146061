"""Helpers shared by the GPU parity tests: run the CUDA path through the C
ABI, run the oracle on the same seeded inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import precision_gemm_token_gb300 as E
from oracle import epilora_oracle as O
from oracle import fpformats as F
from precision_gemm_token_gb300 import tensors as T

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
