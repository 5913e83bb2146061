"""GPU shrink vs the oracle: exact on integer inputs, within fp32 accumulation
error otherwise, masks / no-adapter / out-of-range indices, determinism and
position independence."""
import numpy as np
import pytest
import torch

from oracle import epilora_oracle as O
from precision_gemm_token_gb300 import tensors as T
from synth import make_projection
from synth.inputs import small_integer_tensor

from .gpu_util import ensure_lib, np32, status_buf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def test_shrink_integer_exact():
    rng = np.random.default_rng(0)
    M, K, L, r = 9, 512, 3, 16
    x = small_integer_tensor(rng, (M, K), -8, 8)
    A = small_integer_tensor(rng, (L, r, K), -8, 8)
    idx = np.array([0, 2, 1, -1, 2, 0, 1, 2, 2], np.int32)
    mask = np.array([1, 1, 0, 1, 1, 1, 1, 1, 0], np.uint8)
    S = T.lora_shrink(torch.from_numpy(x).to(torch.bfloat16).cuda(), torch.from_numpy(A).to(torch.bfloat16).cuda(),
                      torch.from_numpy(idx).cuda(), torch.from_numpy(mask).cuda())
    assert (np32(S) == O.shrink(x, A, idx, mask)).all()


@pytest.mark.parametrize("M,K,L,r,mode", [(4, 512, 4, 16, "uniform"), (1, 4096, 1, 64, "single"),
                                          (32, 4096, 32, 64, "per_token"), (5, 14336, 8, 128, "uniform"),
                                          (64, 1024, 16, 32, "zipf")])
def test_shrink_matches_oracle(M, K, L, r, mode):
    p = make_projection(M, K, 16, L, r, seed=M + K, idx_mode=mode, mask_mode="random" if M > 8 else "all")
    S = T.lora_shrink(p.X.cuda(), p.A.cuda(), p.idx.cuda(), p.mask.cuda())
    x, A = p.X.float().numpy(), p.A.float().numpy()
    ref = O.shrink(x, A, p.idx.numpy(), p.mask.numpy())
    # fp32 accumulation of K products: bound by K * 2^-24 * sum |x a|
    mag = np.zeros_like(ref)
    act = O.active_tokens(p.idx.numpy(), p.mask.numpy(), L)
    for t in np.nonzero(act)[0]:
        mag[t] = np.abs(A[p.idx[t]]) @ np.abs(x[t])
    err = np.abs(np32(S) - ref)
    assert (err <= 1e-5 * mag + 1e-30).all(), float((err / (mag + 1e-30)).max())
    assert (np32(S)[~act] == 0).all()


def test_shrink_no_mask_pointer_means_all_active():
    p = make_projection(6, 512, 16, 3, 16, seed=1)
    S = T.lora_shrink(p.X.cuda(), p.A.cuda(), p.idx.cuda(), None)
    ref = O.shrink(p.X.float().numpy(), p.A.float().numpy(), p.idx.numpy(), None)
    assert np.allclose(np32(S), ref, rtol=1e-4, atol=1e-5)


def test_shrink_out_of_range_index_records_status():
    p = make_projection(4, 512, 16, 3, 16, seed=2)
    idx = p.idx.clone()
    idx[1] = 3                                  # == L
    st = status_buf()
    S = T.lora_shrink(p.X.cuda(), p.A.cuda(), idx.cuda(), p.mask.cuda(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -1
    assert (np32(S)[1] == 0).all()


def test_shrink_deterministic_and_position_independent():
    p = make_projection(16, 4096, 16, 4, 64, seed=3)
    X, A, idx, mask = p.X.cuda(), p.A.cuda(), p.idx.cuda(), p.mask.cuda()
    S1 = T.lora_shrink(X, A, idx, mask)
    S2 = T.lora_shrink(X, A, idx, mask)
    assert torch.equal(S1, S2)
    perm = torch.randperm(16, generator=torch.Generator().manual_seed(0)).cuda()
    S3 = T.lora_shrink(X[perm].contiguous(), A, idx[perm].contiguous(), mask[perm].contiguous())
    assert torch.equal(S3, S1[perm])
