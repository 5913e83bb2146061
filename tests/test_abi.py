"""The C-ABI library builds, loads and exports every symbol include/epilora.h
declares; host-side argument validation rejects bad calls before any launch.
No compute call is made here."""
import ctypes
import os
import re

import pytest

import precision_gemm_token_gb300 as E
from precision_gemm_token_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "epilora.h")


def _declared():
    txt = open(HEADER).read()
    return re.findall(r"EPILORA_API\s+[\w\s\*]+?\b(epilora_\w+)\s*\(", txt)


@pytest.fixture(scope="module")
def lib():
    E.build()
    return E.load()


def test_header_declares_the_abi():
    names = _declared()
    for n in ("epilora_quant_act", "epilora_lora_shrink", "epilora_gemm_lora_epilogue", "epilora_layer_forward",
              "epilora_workspace_bytes", "epilora_status_string", "epilora_abi_version",
              "epilora_nvfp4_global_scale"):
        assert n in names
    assert len(names) == len(set(names))


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(E.LIB_PATH)
    for n in _declared():
        assert hasattr(raw, n), n
    # the binding wraps exactly the declared set
    assert set(_binding.SIGNATURES) == set(_declared())


def test_only_abi_symbols_are_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", E.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == set(_declared()), exported ^ set(_declared())


def test_status_strings(lib):
    assert E.epilora_abi_version() == 1
    for code, name in [(0, "EPILORA_OK"), (-1, "EPILORA_ERR_INVALID_ARG"), (-2, "EPILORA_ERR_UNSUPPORTED"),
                       (-3, "EPILORA_ERR_CUDA"), (-4, "EPILORA_ERR_TIMEOUT"), (-5, "EPILORA_ERR_WORKSPACE")]:
        assert E.epilora_status_string(code) == name
    assert E.epilora_status_string(12345) == "EPILORA_UNKNOWN_STATUS"


def test_workspace_bytes(lib):
    r256 = lambda v: (v + 255) // 256 * 256  # noqa: E731
    sync = 2360576                # the head: counters and exchange regions of the single-kernel path
    # counters, Xq, scales, then S with room for ceil(K / 1024) partial sums (at most 8)
    assert E.epilora_workspace_bytes(0, 4, 512, 16) == sync + r256(4 * 512) + r256(16) + r256(4 * 16 * 4)
    assert E.epilora_workspace_bytes(1, 4, 512, 16) == sync + r256(4 * 256) + r256(4 * 32) + r256(4 * 16 * 4)
    assert E.epilora_workspace_bytes(0, 4, 512, 0) == sync + r256(4 * 512) + r256(16)
    assert E.epilora_workspace_bytes(0, 2, 14336, 64) == sync + r256(2 * 14336) + r256(8) + r256(2 * 64 * 4 * 8)
    assert E.epilora_workspace_bytes(0, 1, 40960, 16) == sync + r256(40960) + r256(4) + r256(16 * 4 * 8)
    assert E.epilora_workspace_bytes(0, 3, 4096, 32) == sync + r256(3 * 4096) + r256(12) + r256(3 * 32 * 4 * 4)
    # more than 32 tokens with adapters: plus the adapter-sorted row order (int32 per token)
    assert E.epilora_workspace_bytes(0, 64, 512, 16) == sync + r256(64 * 512) + r256(256) + r256(64 * 16 * 4) + \
        r256(256)
    assert E.epilora_workspace_bytes(0, 64, 512, 0) == sync + r256(64 * 512) + r256(256)
    assert E.epilora_workspace_bytes(0, 0, 512, 16) == 0
    assert E.epilora_workspace_bytes(7, 4, 512, 16) == 0


def test_layer_workspace_bytes(lib):
    r256 = lambda v: (v + 255) // 256 * 256   # noqa: E731
    # more than 32 tokens with adapters of rank >= 32: plus the expand pass's fp32 [M, N] term
    for fmt, M, N, K, r in [(0, 64, 512, 512, 32), (1, 300, 272, 512, 64), (0, 33, 130, 256, 128)]:
        assert E.epilora_layer_workspace_bytes(fmt, M, N, K, r) == \
            E.epilora_workspace_bytes(fmt, M, K, r) + r256(M * N * 4)
    # decode batches, rank 16 and base-only calls: the same as epilora_workspace_bytes
    for fmt, M, N, K, r in [(0, 32, 512, 512, 16), (1, 4, 4096, 4096, 64), (0, 64, 512, 512, 0),
                            (0, 64, 512, 512, 16)]:
        assert E.epilora_layer_workspace_bytes(fmt, M, N, K, r) == E.epilora_workspace_bytes(fmt, M, K, r)
    assert E.epilora_layer_workspace_bytes(0, 0, 512, 512, 16) == 0
    assert E.epilora_layer_workspace_bytes(7, 64, 512, 512, 16) == 0
    assert E.epilora_layer_workspace_bytes(0, 64, -1, 512, 16) == 0


def test_layer_forward_kernels(lib):
    """One persistent kernel for a few tokens (FP8: M * K <= 16384; NVFP4:
    bf16 rows within one 40 KB ring slot; M <= 8) while two weight stages
    still fit beside the per-call buffers; else two. The automatic policy
    gives the single kernel the FP8 calls only."""
    k = E.epilora_layer_forward_kernels
    assert E.epilora_set_decode_path(E.DECODE_PATH_AUTO) == E.DECODE_PATH_AUTO
    assert k(0, 1, 4096, 64) == 1 and k(1, 1, 4096, 64) == 2
    assert E.epilora_set_decode_path(E.DECODE_PATH_TWO) == E.DECODE_PATH_AUTO
    assert k(0, 1, 4096, 64) == 2 and k(1, 1, 4096, 64) == 2
    with pytest.raises(E.EpiloraError):
        E.epilora_set_decode_path(3)
    assert E.epilora_set_decode_path(E.DECODE_PATH_SINGLE) == E.DECODE_PATH_TWO
    assert k(0, 1, 14336, 0) == 1 and k(0, 1, 16384, 64) == 1 and k(0, 1, 16416, 0) == 2
    assert k(0, 4, 4096, 64) == 1 and k(0, 5, 4096, 0) == 2 and k(0, 8, 2048, 16) == 1 and k(0, 9, 512, 0) == 2
    assert k(1, 1, 14336, 64) == 1 and k(1, 2, 8192, 64) == 1 and k(1, 8, 2048, 16) == 1
    assert k(1, 2, 14336, 64) == 2 and k(1, 8, 4096, 16) == 2           # bf16 rows beyond one ring slot
    assert k(0, 8, 2048, 512) == 1 and k(1, 8, 2048, 512) == 2          # S rows crowd out a weight stage
    assert k(1, 1, 4128, 0) == 2                                         # NVFP4 wants K % 256 == 0
    assert k(0, 32, 4096, 0) == 2 and k(0, 0, 4096, 0) == 0 and k(2, 1, 4096, 0) == 0 and k(0, 1, 100, 0) == 0
    E.epilora_set_decode_path(E.DECODE_PATH_AUTO)


# ---------------------------------------------------------------------------
# Validation: every call below is invalid, so it must return before touching
# the GPU. Fake (aligned, never dereferenced) addresses are used, which is
# only safe where no device exists to launch on.
# ---------------------------------------------------------------------------
def _no_gpu():
    import torch
    return not torch.cuda.is_available()


FAKE = 0x10000
INVALID, UNSUP, WS = -1, -2, -5


@pytest.mark.skipif(not _no_gpu(), reason="fake-pointer validation runs only where nothing can launch")
@pytest.mark.parametrize("kw,want", [
    (dict(fmt=2), INVALID),
    (dict(K=40), INVALID),             # FP8: K % 16
    (dict(fmt=1, K=48, x_scale=None, x_block_scale=FAKE, x_global_scale=FAKE), INVALID),   # NVFP4: K % 32
    (dict(K=0), INVALID),
    (dict(M=-1), INVALID),
    (dict(ldx=500), INVALID),          # ldx < K
    (dict(ldx=516), INVALID),          # ldx % 8
    (dict(X=FAKE + 8), INVALID),       # misaligned
    (dict(x_scale=None), INVALID),
])
def test_quant_validation(lib, kw, want):
    a = dict(fmt=0, X=FAKE, M=4, K=512, ldx=512, Xq=FAKE, x_scale=FAKE, x_block_scale=None, x_global_scale=None)
    a.update(kw)
    assert E.epilora_quant_act(a["fmt"], a["X"], a["M"], a["K"], a["ldx"], a["Xq"], a["x_scale"],
                               a["x_block_scale"], a["x_global_scale"], None, 0) == want


@pytest.mark.skipif(not _no_gpu(), reason="fake-pointer validation runs only where nothing can launch")
def test_quant_nvfp4_needs_global_scale(lib):
    assert E.epilora_quant_act(1, FAKE, 4, 512, 512, FAKE, None, FAKE, None, None, 0) == INVALID
    assert E.epilora_quant_act(1, FAKE, 0, 512, 512, None, None, None, FAKE, None, 0) == 0   # M == 0: no-op


@pytest.mark.skipif(not _no_gpu(), reason="fake-pointer validation runs only where nothing can launch")
@pytest.mark.parametrize("kw", [dict(r=8), dict(r=48), dict(L=0), dict(K=100), dict(S=None), dict(idx=None),
                                dict(A=FAKE + 4)])
def test_shrink_validation(lib, kw):
    a = dict(X=FAKE, M=4, K=512, ldx=512, A=FAKE, L=4, r=16, idx=FAKE, mask=None, S=FAKE)
    a.update(kw)
    assert E.epilora_lora_shrink(a["X"], a["M"], a["K"], a["ldx"], a["A"], a["L"], a["r"], a["idx"], a["mask"],
                                 a["S"], None, 0) == INVALID


@pytest.mark.skipif(not _no_gpu(), reason="fake-pointer validation runs only where nothing can launch")
@pytest.mark.parametrize("kw,want", [
    (dict(N=100), INVALID), (dict(N=0), INVALID), (dict(ldy=1000), INVALID), (dict(ldy=1028), INVALID),
    (dict(r=24), INVALID), (dict(Y=FAKE + 2), INVALID), (dict(w_scale=None), INVALID),
    (dict(fmt=1, K=544, xbs=FAKE, xgs=FAKE, wbs=FAKE, wgs=FAKE), UNSUP),   # NVFP4 needs K % 256
    (dict(fmt=1, xbs=FAKE, xgs=None, wbs=FAKE, wgs=FAKE), INVALID),
])
def test_gemm_validation(lib, kw, want):
    a = dict(fmt=0, M=4, N=1024, K=512, Xq=FAKE, xs=FAKE, xbs=None, xgs=None, Wq=FAKE, w_scale=FAKE, wbs=None,
             wgs=None, S=FAKE, B=FAKE, L=4, r=16, idx=FAKE, mask=None, Y=FAKE, ldy=1024)
    a.update(kw)
    assert E.epilora_gemm_lora_epilogue(a["fmt"], a["M"], a["N"], a["K"], a["Xq"], a["xs"], a["xbs"], a["xgs"],
                                        a["Wq"], a["w_scale"], a["wbs"], a["wgs"], a["S"], a["B"], a["L"], a["r"],
                                        a["idx"], a["mask"], a["Y"], a["ldy"], 0, None, 0) == want


@pytest.mark.skipif(not _no_gpu(), reason="fake-pointer validation runs only where nothing can launch")
def test_layer_forward_workspace_checks(lib):
    need = E.epilora_workspace_bytes(0, 4, 512, 16)
    args = lambda ws, nbytes: (0, 4, 1024, 512, FAKE, 512, FAKE, FAKE, None, None, None, FAKE, FAKE, 4, 16,  # noqa
                               FAKE, None, FAKE, 1024, ws, nbytes, None, 0)
    assert E.epilora_layer_forward(*args(None, need)) == WS
    assert E.epilora_layer_forward(*args(FAKE, need - 1)) == WS
    assert E.epilora_layer_forward(*args(FAKE + 16, need)) == WS      # 256-byte alignment


@pytest.mark.skipif(not _no_gpu(), reason="fake-pointer validation runs only where nothing can launch")
@pytest.mark.parametrize("n,ends,A,want", [
    (0, [1024], FAKE, INVALID),                     # no slice
    (5, [128, 256, 384, 512, 1024], FAKE, INVALID),  # more than 4 slices
    (2, [512, 512], FAKE, INVALID),                 # not ascending
    (2, [500, 1024], FAKE, INVALID),                # inner end not a multiple of 128
    (2, [512, 896], FAKE, INVALID),                 # last end != N
    (2, [512, 1024], None, INVALID),                # A required
])
def test_layer_forward_slices_validation(lib, n, ends, A, want):
    need = E.epilora_workspace_bytes(0, 4, 512, 16 * max(n, 1))
    rc = E.epilora_layer_forward_slices(0, 4, 1024, 512, FAKE, 512, FAKE, FAKE, None, None, None, A, FAKE, 4, 16, n,
                                        ends, FAKE, None, FAKE, 1024, FAKE, need, None, 0)
    assert rc == want


@pytest.mark.skipif(not _no_gpu(), reason="fake-pointer validation runs only where nothing can launch")
def test_layer_forward_slices_workspace_sized_for_all_slices(lib):
    """The workspace of a sliced call holds S rows of n_slices * r floats."""
    small = E.epilora_workspace_bytes(0, 4, 512, 16)
    big = E.epilora_workspace_bytes(0, 4, 512, 48)
    assert big > small
    args = lambda nbytes: (0, 4, 1024, 512, FAKE, 512, FAKE, FAKE, None, None, None, FAKE, FAKE, 4, 16, 3,  # noqa
                           [384, 768, 1024], FAKE, None, FAKE, 1024, FAKE, nbytes, None, 0)
    assert E.epilora_layer_forward_slices(*args(small)) == WS
