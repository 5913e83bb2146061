"""Stored FP8 adapters (epilora_layer_forward_fp8_adapters) vs the oracle on
the dequantized tables: the codes and row scales from the GPU quantizer bit
for bit, then the layer within the arithmetic bound, on the single-kernel
path (a few tokens) and on the shrink grid + GEMM path (up to 32 tokens,
the streamed-B decode epilogue); ranks 16..128, several adapters, masked and
adapter-less tokens; batches past 32 tokens are refused."""
import numpy as np
import pytest
import torch

import precision_gemm_token_gb300 as E
from oracle import epilora_oracle as O
from oracle import fpformats as F
from precision_gemm_token_gb300 import tensors as T
from synth import make_projection

from .gpu_util import FP8, NVFP4, assert_y_close, ensure_lib, np32, npu8, same_codes_e4m3, status_buf, tight_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()
    # the cases marked "single kernel" take it in both formats
    prev = E.epilora_set_decode_path(E.DECODE_PATH_SINGLE)
    yield
    E.epilora_set_decode_path(prev)


CASES = [
    # M, K, N, L, r, idx_mode, mask_mode
    (1, 4096, 1024, 1, 64, "single", "all"),      # single kernel
    (4, 2048, 768, 3, 16, "uniform", "random"),   # single kernel, rank 16 rows of B
    (2, 2048, 256, 2, 128, "uniform", "all"),     # single kernel, rank 128
    (12, 1024, 512, 4, 32, "uniform", "random"),  # shrink grid + GEMM, 16-token decode tile
    (32, 4096, 512, 32, 64, "per_token", "all"),  # 32 tenants, 32-token decode tile
]


@pytest.mark.parametrize("fmt", [FP8, NVFP4], ids=["fp8", "nvfp4"])
@pytest.mark.parametrize("M,K,N,L,r,idx_mode,mask_mode", CASES)
def test_fp8_adapters_match_oracle(fmt, M, K, N, L, r, idx_mode, mask_mode):
    p = make_projection(M, K, N, L, r, seed=M * 13 + r, idx_mode=idx_mode, mask_mode=mask_mode)
    X, W = p.X.cuda(), p.W.cuda()
    w = T.quantize_weight(W, fmt)
    ad = T.quantize_adapters_fp8(p.A.cuda(), p.B.cuda())
    x, Wn = p.X.float().numpy(), W.float().cpu().numpy()
    A, B = p.A.float().numpy(), p.B.float().numpy()
    idx, mask = p.idx.numpy(), p.mask.numpy()
    # the stored tables: the FP8 row quantizer's codes and scales, bit for bit
    Aq, sa = O.quant_adapter_fp8(A)
    Bq, sb = O.quant_adapter_fp8(B)
    assert same_codes_e4m3(npu8(ad.Aq), Aq).all() and (np32(ad.a_scale) == sa).all()
    assert same_codes_e4m3(npu8(ad.Bq), Bq).all() and (np32(ad.b_scale) == sb).all()
    Ah, Bh = O.dequant_adapter_fp8(Aq, sa), O.dequant_adapter_fp8(Bq, sb)
    gx = None
    if fmt == FP8:
        wq, sw = O.quant_fp8_rows(Wn)
        ref = O.layer_fp8(x, wq, sw, Ah, Bh, idx, mask)
        xv = F.e4m3_decode(ref["xq"]) * ref["sx"][:, None].astype(np.float64)
        wv = F.e4m3_decode(wq) * sw[:, None].astype(np.float64)
    else:
        gw = O.nvfp4_global_scale(Wn)
        wq, sbw = O.quant_nvfp4_rows(Wn, gw)
        gxv = O.nvfp4_global_scale(x)
        gx = torch.tensor([gxv], dtype=torch.float32, device="cuda")
        ref = O.layer_nvfp4(x, gxv, wq, sbw, gw, Ah, Bh, idx, mask)
        xv = O.dequant_nvfp4_rows(ref["xq"], ref["sbx"], gxv)
        wv = O.dequant_nvfp4_rows(wq, sbw, gw)
    st = status_buf()
    Y = T.layer_forward_fp8_adapters(X, w, ad, p.idx.cuda(), p.mask.cuda(), x_global_scale=gx, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_y_close(np32(Y), ref, tight_bound(ref, xv, wv, Bh, idx, mask), what=(fmt, M, K, N, r))


def test_fp8_adapters_refuse_wide_batches():
    p = make_projection(33, 512, 256, 2, 16, seed=1)
    w = T.quantize_weight(p.W.cuda(), FP8)
    ad = T.quantize_adapters_fp8(p.A.cuda(), p.B.cuda())
    with pytest.raises(E.EpiloraError) as ei:
        T.layer_forward_fp8_adapters(p.X.cuda(), w, ad, p.idx.cuda(), p.mask.cuda())
    assert ei.value.status == E.EPILORA_ERR_UNSUPPORTED


@pytest.mark.parametrize("M", [1, 16])
def test_fp8_adapters_zero_base_isolates_the_adapter_term(M):
    """All-zero weights: Y is bf16 of the stored adapters' term alone, against
    the oracle's term from the dequantized tables (1e-2 relative), and the
    stored tables' term against the bf16 tables' term (the price of storing
    them in FP8, reported beside the speed: a few percent)."""
    K, N, L, r = 4096, 512, 4, 64
    p = make_projection(M, K, N, L, r, seed=40 + M)
    W = torch.zeros_like(p.W).cuda()
    w = T.quantize_weight(W, FP8)
    ad = T.quantize_adapters_fp8(p.A.cuda(), p.B.cuda())
    Y = T.layer_forward_fp8_adapters(p.X.cuda(), w, ad, p.idx.cuda(), p.mask.cuda())
    x, A, B = p.X.float().numpy(), p.A.float().numpy(), p.B.float().numpy()
    idx, mask = p.idx.numpy(), p.mask.numpy()
    Ah = O.dequant_adapter_fp8(*O.quant_adapter_fp8(A))
    Bh = O.dequant_adapter_fp8(*O.quant_adapter_fp8(B))
    d_q = O.expand(O.shrink(x, Ah, idx, mask), Bh, idx, mask)
    d_bf = O.expand(O.shrink(x, A, idx, mask), B, idx, mask)
    y = np32(Y).astype(np.float64)
    assert np.linalg.norm(y - d_q) / np.linalg.norm(d_q) <= 1e-2
    rel_fp8_vs_bf16 = np.linalg.norm(d_q - d_bf) / np.linalg.norm(d_bf)
    assert rel_fp8_vs_bf16 <= 0.05, rel_fp8_vs_bf16
