"""GPU quantizers vs the oracle: codes and scales bit-exact (FP8 per token,
NVFP4 per 16-block), exhaustive over every bf16 value in range, plus the
global-scale helper."""
import numpy as np
import pytest
import torch

from oracle import epilora_oracle as O
from oracle import fpformats as F
from precision_gemm_token_gb300 import tensors as T
from synth import make_projection

from .gpu_util import FP8, NVFP4, ensure_lib, np32, npu8, same_codes_e2m1_packed, same_codes_e4m3, status_buf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _bf16_rows(rng, M, K, std=1.0):
    return torch.from_numpy((rng.standard_normal((M, K)) * std).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("M,K,std", [(4, 512, 1.0), (1, 4096, 1.0), (33, 14336, 3.0), (7, 32, 1e-3),
                                     (64, 1024, 100.0), (2, 40960, 1.0)])
def test_fp8_quant_bit_exact(M, K, std):
    rng = np.random.default_rng(M * 1000 + K)
    X = _bf16_rows(rng, M, K, std)
    X[0, :] = 0                                   # all-zero token uses the floor
    Xg = X.cuda()
    q, s = T.quant_act(Xg, FP8)
    oq, os_ = O.quant_fp8_rows(X.float().numpy())
    assert (np32(s) == os_).all()
    assert same_codes_e4m3(npu8(q), oq).all()


def test_fp8_quant_strided_rows():
    rng = np.random.default_rng(3)
    big = _bf16_rows(rng, 5, 640).cuda()
    X = big[:, :512]                              # ldx = 640 > K
    q, s = T.quant_act(X, FP8)
    oq, os_ = O.quant_fp8_rows(np32(X))
    assert (np32(s) == os_).all() and same_codes_e4m3(npu8(q), oq).all()


def test_fp8_conversion_exhaustive_over_bf16():
    """Rows whose amax is 448 have scale exactly 1, so the codes are the
    conversion of every bf16 value in [-448, 448] itself."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 448)]
    K = 1024
    n = (vals.size + K - 2) // (K - 1)
    rows = np.zeros((n, K), np.float32)
    flat = np.zeros(n * (K - 1), np.float32)
    flat[:vals.size] = vals
    rows[:, 1:] = flat.reshape(n, K - 1)
    rows[:, 0] = 448.0
    X = torch.from_numpy(rows).to(torch.bfloat16)
    assert (X.float().numpy() == rows).all()
    q, s = T.quant_act(X.cuda(), FP8)
    assert (np32(s) == 1.0).all()
    oq = F.fp32_to_e4m3_code(rows)
    assert same_codes_e4m3(npu8(q), oq).all()


@pytest.mark.parametrize("M,K", [(4, 512), (1, 4096), (32, 14336), (3, 32)])
def test_nvfp4_quant_bit_exact(M, K):
    rng = np.random.default_rng(M + K)
    X = _bf16_rows(rng, M, K)
    X[0, 16:32] = 0                               # a zero block
    Xg = X.cuda()
    g = T.nvfp4_global_scale(Xg)
    og = O.nvfp4_global_scale(X.float().numpy())
    assert np32(g)[0] == og
    q, sb = T.quant_act(Xg, NVFP4, global_scale=g)
    oq, osb = O.quant_nvfp4_rows(X.float().numpy(), og)
    assert (npu8(sb) == osb).all()
    assert same_codes_e2m1_packed(npu8(q), oq).all()


def test_nvfp4_conversion_exhaustive_over_bf16():
    """g = 1 and a 6 in every block give block scale 1 and multiplier 1, so the
    codes are the E2M1 conversion of every bf16 value in [-6, 6]."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 6)]
    per = 15
    nb = (vals.size + per - 1) // per
    blocks = np.zeros((nb, 16), np.float32)
    flat = np.zeros(nb * per, np.float32)
    flat[:vals.size] = vals
    blocks[:, 1:] = flat.reshape(nb, per)
    blocks[:, 0] = 6.0
    K = 512
    nb_pad = (nb + K // 16 - 1) // (K // 16) * (K // 16)
    allb = np.zeros((nb_pad, 16), np.float32)
    allb[:nb] = blocks
    allb[nb:, 0] = 6.0
    rows = allb.reshape(-1, K)
    X = torch.from_numpy(rows).to(torch.bfloat16).cuda()
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    q, sb = T.quant_act(X, NVFP4, global_scale=g)
    assert (npu8(sb) == 0x38).all()               # E4M3 1.0
    oq = F.pack_e2m1(F.fp32_to_e2m1_code(rows))
    assert same_codes_e2m1_packed(npu8(q), oq).all()


def test_nvfp4_bad_global_scale_records_status():
    X = torch.ones((2, 64), dtype=torch.bfloat16, device="cuda")
    st = status_buf()
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    q, sb = T.quant_act(X, NVFP4, global_scale=g, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -1
    assert (npu8(sb) == 0).all() and (npu8(q) == 0).all()


def test_weight_quant_matches_oracle_fp8_and_nvfp4():
    p = make_projection(4, 512, 1024, 4, 16, seed=0)
    W = p.W.to(torch.bfloat16)
    Wn = W.float().numpy()
    w8 = T.quantize_weight(W.cuda(), FP8)
    oq, os_ = O.quant_fp8_rows(Wn)
    assert (np32(w8.scale) == os_).all() and same_codes_e4m3(npu8(w8.codes), oq).all()
    w4 = T.quantize_weight(W.cuda(), NVFP4)
    og = O.nvfp4_global_scale(Wn)
    assert np32(w4.global_scale)[0] == og
    oq4, osb4 = O.quant_nvfp4_rows(Wn, og)
    assert (npu8(w4.block_scale) == osb4).all() and same_codes_e2m1_packed(npu8(w4.codes), oq4).all()


def test_quant_deterministic():
    rng = np.random.default_rng(9)
    X = _bf16_rows(rng, 16, 4096).cuda()
    a = T.quant_act(X, FP8)
    b = T.quant_act(X, FP8)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
