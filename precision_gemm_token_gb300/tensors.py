"""Tensor-level helpers over the C ABI: allocate outputs with torch on the
inputs' device, call the binding, raise on a non-OK status. No arithmetic of
the layer happens here; every step runs in libepilora.so's kernels."""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import _binding as E


def _u8(shape, dev):
    return torch.empty(shape, dtype=torch.uint8, device=dev)


@dataclass
class QuantWeight:
    fmt: int
    codes: torch.Tensor                         # uint8 [N, K] (FP8) or [N, K/2] (NVFP4)
    scale: Optional[torch.Tensor] = None        # fp32 [N] (FP8)
    block_scale: Optional[torch.Tensor] = None  # uint8 [N, K/16] (NVFP4)
    global_scale: Optional[torch.Tensor] = None  # fp32 [1] (NVFP4)

    @property
    def N(self):
        return self.codes.shape[0]


def nvfp4_global_scale(T: torch.Tensor, stream=None) -> torch.Tensor:
    g = torch.empty(1, dtype=torch.float32, device=T.device)
    E.check(E.epilora_nvfp4_global_scale(T, T.numel(), g, stream), "epilora_nvfp4_global_scale")
    return g


def quant_act(X: torch.Tensor, fmt: int, global_scale: Optional[torch.Tensor] = None, status=None, stream=None):
    """X bf16 [M, K] -> (codes, scale or block scale)."""
    M, K = X.shape
    dev = X.device
    if fmt == E.FMT_FP8:
        q, s = _u8((M, K), dev), torch.empty(M, dtype=torch.float32, device=dev)
        E.check(E.epilora_quant_act(fmt, X, M, K, X.stride(0), q, s, None, None, status, stream), "quant_act")
        return q, s
    q, sb = _u8((M, K // 2), dev), _u8((M, K // 16), dev)
    E.check(E.epilora_quant_act(fmt, X, M, K, X.stride(0), q, None, sb, global_scale, status, stream), "quant_act")
    return q, sb


def quant_act_into(X: torch.Tensor, fmt: int, Xq, scale, global_scale=None, status=None, stream=None):
    """quant_act into caller-owned outputs (codes, and the FP8 scales or the
    NVFP4 block scales)."""
    M, K = X.shape
    if fmt == E.FMT_FP8:
        rc = E.epilora_quant_act(fmt, X, M, K, X.stride(0), Xq, scale, None, None, status, stream)
    else:
        rc = E.epilora_quant_act(fmt, X, M, K, X.stride(0), Xq, None, scale, global_scale, status, stream)
    E.check(rc, "quant_act")


def quantize_weight(W: torch.Tensor, fmt: int, stream=None) -> QuantWeight:
    """Load-time quantization of a bf16 weight [N, K] with the same kernels:
    FP8 per-output-channel scales, or NVFP4 with g_w from W's amax."""
    if fmt == E.FMT_FP8:
        q, s = quant_act(W, fmt, stream=stream)
        return QuantWeight(fmt, q, scale=s)
    g = nvfp4_global_scale(W, stream)
    q, sb = quant_act(W, fmt, global_scale=g, stream=stream)
    return QuantWeight(fmt, q, block_scale=sb, global_scale=g)


def lora_shrink(X, A, idx, mask=None, status=None, stream=None) -> torch.Tensor:
    M, K = X.shape
    L, r, _ = A.shape
    S = torch.empty((M, r), dtype=torch.float32, device=X.device)
    E.check(E.epilora_lora_shrink(X, M, K, X.stride(0), A, L, r, idx, mask, S, status, stream), "lora_shrink")
    return S


@dataclass
class Fp8Adapters:
    """Adapter tables stored as E4M3 codes with one fp32 scale per row."""
    Aq: torch.Tensor        # uint8 [L, r, K]
    a_scale: torch.Tensor   # fp32 [L, r]
    Bq: torch.Tensor        # uint8 [L, N, r]
    b_scale: torch.Tensor   # fp32 [L, N]


def quantize_adapters_fp8(A: torch.Tensor, B: torch.Tensor, stream=None) -> Fp8Adapters:
    """Load-time quantization of bf16 adapter tables A [L, r, K] and B [L, N, r]
    with the FP8 row quantizer (one scale per row of each table)."""
    L, r, K = A.shape
    N = B.shape[1]
    Aq, sa = quant_act(A.reshape(L * r, K), E.FMT_FP8, stream=stream)
    Bq, sb = quant_act(B.reshape(L * N, r), E.FMT_FP8, stream=stream)
    return Fp8Adapters(Aq.view(L, r, K), sa.view(L, r), Bq.view(L, N, r), sb.view(L, N))


def layer_forward_fp8_adapters(X, w: QuantWeight, ad: Fp8Adapters, idx, mask=None, x_global_scale=None,
                               workspace: Optional[LayerWorkspace] = None, status=None, stream=None, Y=None):
    """epilora_layer_forward_fp8_adapters: the layer with stored FP8 adapters."""
    M, K = X.shape
    N = w.N
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    L, r = ad.Aq.shape[0], ad.Aq.shape[1]
    ws = workspace or LayerWorkspace(X.device)
    buf = ws.get(w.fmt, M, K, r)
    rc = E.epilora_layer_forward_fp8_adapters(w.fmt, M, N, K, X, X.stride(0), w.codes, w.scale, w.block_scale,
                                              w.global_scale, x_global_scale, ad.Aq, ad.a_scale, ad.Bq, ad.b_scale,
                                              L, r, idx, mask, Y, Y.stride(0), buf, ws.need(w.fmt, M, K, r), status,
                                              stream)
    E.check(rc, "layer_forward_fp8_adapters")
    return Y


def lora_shrink_into(X, A, idx, mask, S, status=None, stream=None):
    """lora_shrink into a caller-owned S [M, r] fp32."""
    M, K = X.shape
    L, r, _ = A.shape
    E.check(E.epilora_lora_shrink(X, M, K, X.stride(0), A, L, r, idx, mask, S, status, stream), "lora_shrink")


def gemm_lora_epilogue(Xq, x_scale, w: QuantWeight, M, K, S=None, B=None, idx=None, mask=None,
                       x_global_scale=None, pdl_dependent=False, status=None, stream=None, Y=None):
    N = w.N
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=w.codes.device)
    L, r = (B.shape[0], B.shape[2]) if B is not None else (1, 16)
    if w.fmt == E.FMT_FP8:
        rc = E.epilora_gemm_lora_epilogue(w.fmt, M, N, K, Xq, x_scale, None, None, w.codes, w.scale, None, None,
                                          S, B, L, r, idx, mask, Y, Y.stride(0), pdl_dependent, status, stream)
    else:
        rc = E.epilora_gemm_lora_epilogue(w.fmt, M, N, K, Xq, None, x_scale, x_global_scale, w.codes, None,
                                          w.block_scale, w.global_scale, S, B, L, r, idx, mask, Y, Y.stride(0),
                                          pdl_dependent, status, stream)
    E.check(rc, "gemm_lora_epilogue")
    return Y


class LayerWorkspace:
    """Caller-owned workspace for epilora_layer_forward (grown on demand).
    Zero-filled when (re)allocated: the library wants the head of the
    workspace zero before the first call and keeps it valid after each."""

    def __init__(self, device):
        self.device = torch.device(device)
        self.buf = torch.zeros(0, dtype=torch.uint8, device=self.device)
        self._need = {}     # (fmt, M, N, K, r) -> bytes, asked of the library once per shape

    def need(self, fmt, M, K, r, N=None) -> int:
        """Bytes a call of this shape uses: epilora_layer_workspace_bytes
        when N is given (batches of more than 32 tokens with adapters then
        take the expand pass), else epilora_workspace_bytes."""
        key = (fmt, M, N, K, r)
        need = self._need.get(key)
        if need is None:
            need = E.epilora_workspace_bytes(fmt, M, K, r) if N is None else \
                E.epilora_layer_workspace_bytes(fmt, M, N, K, r)
            self._need[key] = need
        return need

    def get(self, fmt, M, K, r, N=None) -> torch.Tensor:
        need = self.need(fmt, M, K, r, N)
        if self.buf.numel() < need:
            self.buf = torch.zeros(max(need, 256), dtype=torch.uint8, device=self.device)
        return self.buf


def layer_forward_slices(X, w: QuantWeight, A, B, idx, slice_end, mask=None, x_global_scale=None,
                         workspace: Optional[LayerWorkspace] = None, status=None, stream=None, Y=None):
    """Multi-slice projection: A [L, n_slices * r, K], B [L, N, r]; output
    columns [slice_end[s-1], slice_end[s]) use slice s's adapter pair."""
    M, K = X.shape
    N = w.N
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    n = len(slice_end)
    L, r = A.shape[0], B.shape[2]
    ws = workspace or LayerWorkspace(X.device)
    buf = ws.get(w.fmt, M, K, n * r, N)
    rc = E.epilora_layer_forward_slices(w.fmt, M, N, K, X, X.stride(0), w.codes, w.scale, w.block_scale,
                                        w.global_scale, x_global_scale, A, B, L, r, n, slice_end, idx, mask, Y,
                                        Y.stride(0), buf, ws.need(w.fmt, M, K, n * r, N), status, stream)
    E.check(rc, "layer_forward_slices")
    return Y


def layer_forward(X, w: QuantWeight, A=None, B=None, idx=None, mask=None, x_global_scale=None,
                  workspace: Optional[LayerWorkspace] = None, status=None, stream=None, Y=None):
    M, K = X.shape
    N = w.N
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    L, r = (A.shape[0], A.shape[1]) if A is not None else (1, 16)
    ws = workspace or LayerWorkspace(X.device)
    rr = r if A is not None else 0
    buf = ws.get(w.fmt, M, K, rr, N)
    rc = E.epilora_layer_forward(w.fmt, M, N, K, X, X.stride(0), w.codes, w.scale, w.block_scale, w.global_scale,
                                 x_global_scale, A, B, L, r, idx, mask, Y, Y.stride(0), buf,
                                 ws.need(w.fmt, M, K, rr, N), status, stream)
    E.check(rc, "layer_forward")
    return Y


class PreparedLayer:
    """epilora_layer_forward with every argument bound once (the device
    addresses of the given tensors, the sizes, the workspace and the stream):
    each call enqueues the same layer again with a single C call, no per-call
    argument conversion. The tensors must stay alive and in place (a caller
    refreshes X's contents, e.g. with one copy per step, and reads Y)."""

    def __init__(self, X, w: QuantWeight, A=None, B=None, idx=None, mask=None, x_global_scale=None,
                 workspace: Optional[LayerWorkspace] = None, status=None, stream=None, Y=None):
        M, K = X.shape
        N = w.N
        if Y is None:
            Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
        L, r = (A.shape[0], A.shape[1]) if A is not None else (1, 16)
        ws = workspace or LayerWorkspace(X.device)
        rr = r if A is not None else 0
        buf = ws.get(w.fmt, M, K, rr, N)
        p = lambda t: None if t is None else t.data_ptr()   # noqa: E731
        if stream is None:
            stream = torch.cuda.current_stream(X.device)
        s = stream if isinstance(stream, int) else stream.cuda_stream
        self.Y = Y
        self._keep = (X, w, A, B, idx, mask, x_global_scale, buf, status, Y)
        self._fn = E.load().epilora_layer_forward
        self._args = (w.fmt, M, N, K, p(X), X.stride(0), p(w.codes), p(w.scale), p(w.block_scale), p(w.global_scale),
                      p(x_global_scale), p(A), p(B), L, r, p(idx), p(mask), p(Y), Y.stride(0), p(buf),
                      ws.need(w.fmt, M, K, rr, N), p(status), s)

    def __call__(self):
        rc = self._fn(*self._args)
        if rc != E.EPILORA_OK:
            E.check(rc, "layer_forward")
        return self.Y
