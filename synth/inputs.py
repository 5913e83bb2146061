"""Seeded input generators for the multi-tenant LoRA linear layer.

Value laws (per projection, drawn in fp32 and rounded to bf16 where the
layer's input is bf16):

* activations X ~ N(0, 1)                      -> bf16 [M, K]
* weights W ~ N(0, 0.02^2)                     -> bf16 [N, K], the unquantized
  checkpoint (quantized at load time by whichever side consumes it; this
  module does not quantize)
* adapter down-projections A ~ N(0, 1/K)       -> bf16 [L, r, K]
* adapter up-projections   B ~ N(0, 0.01^2)    -> bf16 [L, N, r]
* token -> adapter slot index: uniform, one-per-tenant, or truncated
  Zipf(s) over the L resident slots              -> int32 [M]
* prefill mask: all ones, or "decode tokens first (mask 0), then one prefill
  chunk (mask 1) that shares one adapter"        -> uint8 [M]

Small inputs are drawn on the host with numpy's PCG64 so that they are
identical on every machine. Full-size Llama-shaped layers (hundreds of MB to
GB of weights) are drawn on the GPU with torch's seeded Philox generator; the
oracle then reads back only the rows it needs.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

# (name, K, N) of the four linear projections of one decoder layer.
LLAMA8B_PROJECTIONS = (
    ("qkv", 4096, 6144),
    ("o", 4096, 4096),
    ("gate_up", 4096, 28672),
    ("down", 14336, 4096),
)
LLAMA70B_PROJECTIONS = (
    ("qkv", 8192, 10240),
    ("o", 8192, 8192),
    ("gate_up", 8192, 57344),
    ("down", 28672, 8192),
)

W_STD = 0.02
B_STD = 0.01


@dataclass
class ProjectionInputs:
    X: torch.Tensor          # bf16 [M, K]
    W: torch.Tensor          # bf16 [N, K] unquantized weights
    A: torch.Tensor          # bf16 [L, r, K]
    B: torch.Tensor          # bf16 [L, N, r]
    idx: torch.Tensor        # int32 [M]; -1 = no adapter
    mask: torch.Tensor       # uint8 [M]; 0 = adapter skipped for this token

    @property
    def shape(self):
        M, K = self.X.shape
        L, r, _ = self.A.shape
        return M, K, self.W.shape[0], L, r


def zipf_probabilities(L: int, s: float) -> np.ndarray:
    """Truncated Zipf over ranks 1..L: P(k) proportional to k^-s."""
    w = np.arange(1, L + 1, dtype=np.float64) ** (-s)
    return w / w.sum()


def zipf_indices(rng: np.random.Generator, M: int, L: int, s: float = 1.1) -> np.ndarray:
    """Rank k is mapped to adapter slot k-1 (slot 0 is the most popular)."""
    return rng.choice(L, size=M, p=zipf_probabilities(L, s)).astype(np.int32)


def _index_and_mask(rng: np.random.Generator, M: int, L: int, idx_mode: str,
                    mask_mode: str, n_decode: int) -> tuple[np.ndarray, np.ndarray]:
    if idx_mode == "uniform":
        idx = rng.integers(0, L, size=M, dtype=np.int64).astype(np.int32)
    elif idx_mode == "per_token":          # token t uses its own tenant's slot t
        if M > L:
            raise ValueError("per_token indices need M <= L")
        idx = np.arange(M, dtype=np.int32)
    elif idx_mode == "zipf":
        idx = zipf_indices(rng, M, L)
    elif idx_mode == "single":
        idx = np.zeros(M, dtype=np.int32)
    elif idx_mode == "none":
        idx = np.full(M, -1, dtype=np.int32)
    else:
        raise ValueError(f"unknown idx_mode {idx_mode!r}")

    if mask_mode == "all":
        mask = np.ones(M, dtype=np.uint8)
    elif mask_mode == "none":
        mask = np.zeros(M, dtype=np.uint8)
    elif mask_mode == "prefill_chunk":
        # decode tokens first (adapter skipped), then one prefill request whose
        # tokens all carry one adapter drawn from the same index law.
        if not 0 <= n_decode <= M:
            raise ValueError("n_decode out of range")
        mask = np.zeros(M, dtype=np.uint8)
        mask[n_decode:] = 1
        if n_decode < M:
            idx[n_decode:] = idx[n_decode]
    elif mask_mode == "random":
        mask = rng.integers(0, 2, size=M, dtype=np.int64).astype(np.uint8)
    else:
        raise ValueError(f"unknown mask_mode {mask_mode!r}")
    return idx, mask


def make_projection(M: int, K: int, N: int, L: int, r: int, *, seed: int = 0,
                    idx_mode: str = "uniform", mask_mode: str = "all",
                    n_decode: int = 0, device: str = "cpu",
                    x_std: float = 1.0, w_std: float = W_STD,
                    b_std: float = B_STD, gen: Optional[str] = None) -> ProjectionInputs:
    """Draw one projection's inputs.

    gen = "numpy" (default on cpu) draws everything with PCG64(seed) on the
    host; gen = "torch" (default on cuda) draws the large tensors with torch's
    Philox generator on `device`. Index and mask always come from PCG64(seed)
    so they are the same for both generators.
    """
    if gen is None:
        gen = "numpy" if device == "cpu" else "torch"
    rng = np.random.Generator(np.random.PCG64(seed))
    idx, mask = _index_and_mask(rng, M, L, idx_mode, mask_mode, n_decode)

    if gen == "numpy":
        X = rng.standard_normal((M, K), dtype=np.float32) * np.float32(x_std)
        W = rng.standard_normal((N, K), dtype=np.float32) * np.float32(w_std)
        A = rng.standard_normal((L, r, K), dtype=np.float32) * np.float32(1.0 / np.sqrt(K))
        B = rng.standard_normal((L, N, r), dtype=np.float32) * np.float32(b_std)
        t = lambda a: torch.from_numpy(a).to(device)  # noqa: E731
        Xt, Wt = t(X).to(torch.bfloat16), t(W).to(torch.bfloat16)
        At, Bt = t(A).to(torch.bfloat16), t(B).to(torch.bfloat16)
    elif gen == "torch":
        g = torch.Generator(device=device)
        g.manual_seed(int(seed) * 7919 + 17)
        Xt = (torch.randn((M, K), generator=g, device=device) * x_std).to(torch.bfloat16)
        Wt = (torch.randn((N, K), generator=g, device=device) * w_std).to(torch.bfloat16)
        At = (torch.randn((L, r, K), generator=g, device=device) * (1.0 / np.sqrt(K))).to(torch.bfloat16)
        Bt = (torch.randn((L, N, r), generator=g, device=device) * b_std).to(torch.bfloat16)
    else:
        raise ValueError(f"unknown generator {gen!r}")

    return ProjectionInputs(
        X=Xt.contiguous(), W=Wt.contiguous(), A=At.contiguous(), B=Bt.contiguous(),
        idx=torch.from_numpy(idx).to(device), mask=torch.from_numpy(mask).to(device))


def small_integer_tensor(rng: np.random.Generator, shape, lo: int, hi: int) -> np.ndarray:
    """Integer-valued float32 tensor (exact in bf16 for |v| <= 256)."""
    return rng.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.float32)
