"""ctypes binding of libepilora.so: the C ABI of include/epilora.h, same names.

Argument marshalling only. Every data argument may be a torch tensor (its
data_ptr() is passed), a raw integer device address, or None (NULL). `stream`
may be a torch.cuda.Stream, a raw cudaStream_t integer, or None for torch's
current stream on the current device. Each function returns the library's
int status; `check()` turns a non-zero status into an exception.

There is no fallback: if the library has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

EPILORA_OK = 0
EPILORA_ERR_INVALID_ARG = -1
EPILORA_ERR_UNSUPPORTED = -2
EPILORA_ERR_CUDA = -3
EPILORA_ERR_TIMEOUT = -4
EPILORA_ERR_WORKSPACE = -5
FMT_FP8 = 0
FMT_NVFP4 = 1

_c_int, _vp, _sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t

# name -> (restype, argtypes), in the order of include/epilora.h
SIGNATURES = {
    "epilora_abi_version": (_c_int, []),
    "epilora_status_string": (ctypes.c_char_p, [_c_int]),
    "epilora_quant_act": (_c_int, [_c_int, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp, _vp, _vp]),
    "epilora_nvfp4_global_scale": (_c_int, [_vp, _sz, _vp, _vp]),
    "epilora_lora_shrink": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp, _c_int, _c_int, _vp, _vp, _vp, _vp, _vp]),
    "epilora_gemm_lora_epilogue": (_c_int, [_c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                            _vp, _vp, _c_int, _c_int, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp]),
    "epilora_workspace_bytes": (_sz, [_c_int, _c_int, _c_int, _c_int]),
    "epilora_layer_workspace_bytes": (_sz, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "epilora_layer_forward_kernels": (_c_int, [_c_int, _c_int, _c_int, _c_int]),
    "epilora_test_drop_shrink_results": (_c_int, [_c_int]),
    "epilora_set_decode_path": (_c_int, [_c_int]),
    "epilora_layer_forward": (_c_int, [_c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _vp, _vp, _vp, _vp, _vp,
                                       _vp, _c_int, _c_int, _vp, _vp, _vp, _c_int, _vp, _sz, _vp, _vp]),
    "epilora_layer_forward_fp8_adapters": (_c_int, [_c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _vp, _vp, _vp,
                                                    _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp, _vp, _c_int,
                                                    _vp, _sz, _vp, _vp]),
    "epilora_layer_forward_noalloc": (_c_int, [_c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _vp, _vp, _vp,
                                               _vp, _vp, _vp, _c_int, _c_int, _vp, _vp, _vp, _c_int, _vp, _vp]),
    "epilora_layer_forward_slices": (_c_int, [_c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _vp, _vp, _vp, _vp,
                                              _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp, _c_int, _vp,
                                              _sz, _vp, _vp]),
}

_lib = None


class EpiloraError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_name(status)} ({status})" if what else f"{status_name(status)} ({status})")


def load(path: str | None = None):
    """Load libepilora.so (built in-tree by precision_gemm_token_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libepilora.so is not built ({path}); run precision_gemm_token_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_name(status: int) -> str:
    try:
        return load().epilora_status_string(int(status)).decode()
    except Exception:  # library missing: still name the code
        return {0: "EPILORA_OK", -1: "EPILORA_ERR_INVALID_ARG", -2: "EPILORA_ERR_UNSUPPORTED",
                -3: "EPILORA_ERR_CUDA", -4: "EPILORA_ERR_TIMEOUT", -5: "EPILORA_ERR_WORKSPACE"}.get(status, "?")


def check(status: int, what: str = "") -> None:
    if status != EPILORA_OK:
        raise EpiloraError(status, what)


def epilora_abi_version() -> int:
    return load().epilora_abi_version()


def epilora_status_string(status: int) -> str:
    return load().epilora_status_string(int(status)).decode()


def epilora_quant_act(fmt, X, M, K, ldx, Xq, x_scale, x_block_scale, x_global_scale, status_dev=None,
                      stream=None) -> int:
    return load().epilora_quant_act(fmt, _p(X), M, K, ldx, _p(Xq), _p(x_scale), _p(x_block_scale),
                                    _p(x_global_scale), _p(status_dev), _stream(stream))


def epilora_nvfp4_global_scale(T, n, g_out, stream=None) -> int:
    return load().epilora_nvfp4_global_scale(_p(T), n, _p(g_out), _stream(stream))


def epilora_lora_shrink(X, M, K, ldx, A, L, r, idx, mask, S, status_dev=None, stream=None) -> int:
    return load().epilora_lora_shrink(_p(X), M, K, ldx, _p(A), L, r, _p(idx), _p(mask), _p(S), _p(status_dev),
                                      _stream(stream))


def epilora_gemm_lora_epilogue(fmt, M, N, K, Xq, x_scale, x_block_scale, x_global_scale, Wq, w_scale,
                               w_block_scale, w_global_scale, S, B, L, r, idx, mask, Y, ldy, pdl_dependent=0,
                               status_dev=None, stream=None) -> int:
    return load().epilora_gemm_lora_epilogue(fmt, M, N, K, _p(Xq), _p(x_scale), _p(x_block_scale),
                                             _p(x_global_scale), _p(Wq), _p(w_scale), _p(w_block_scale),
                                             _p(w_global_scale), _p(S), _p(B), L, r, _p(idx), _p(mask), _p(Y), ldy,
                                             int(pdl_dependent), _p(status_dev), _stream(stream))


def epilora_workspace_bytes(fmt, M, K, r) -> int:
    return load().epilora_workspace_bytes(fmt, M, K, r)


def epilora_layer_workspace_bytes(fmt, M, N, K, r) -> int:
    return load().epilora_layer_workspace_bytes(fmt, M, N, K, r)


def epilora_layer_forward_kernels(fmt, M, K, r) -> int:
    return load().epilora_layer_forward_kernels(fmt, M, K, r)


DECODE_PATH_AUTO, DECODE_PATH_SINGLE, DECODE_PATH_TWO = 0, 1, 2


def epilora_set_decode_path(policy: int) -> int:
    """Decode-path policy for later calls (DECODE_PATH_AUTO: the single kernel
    for FP8, the shrink grid and GEMM for NVFP4; _SINGLE: the single kernel
    wherever it can run; _TWO: never). Returns the previous policy."""
    rc = load().epilora_set_decode_path(policy)
    check(rc if rc < 0 else 0, "set_decode_path")
    return rc


def epilora_test_drop_shrink_results(on: bool) -> None:
    """Test hook: the single-kernel path's shrink items publish nothing
    while on (finishers then time out with EPILORA_ERR_TIMEOUT)."""
    load().epilora_test_drop_shrink_results(1 if on else 0)


def epilora_layer_forward(fmt, M, N, K, X, ldx, Wq, w_scale, w_block_scale, w_global_scale, x_global_scale, A, B,
                          L, r, idx, mask, Y, ldy, workspace, workspace_bytes, status_dev=None, stream=None) -> int:
    return load().epilora_layer_forward(fmt, M, N, K, _p(X), ldx, _p(Wq), _p(w_scale), _p(w_block_scale),
                                        _p(w_global_scale), _p(x_global_scale), _p(A), _p(B), L, r, _p(idx),
                                        _p(mask), _p(Y), ldy, _p(workspace), workspace_bytes, _p(status_dev),
                                        _stream(stream))


def epilora_layer_forward_slices(fmt, M, N, K, X, ldx, Wq, w_scale, w_block_scale, w_global_scale, x_global_scale,
                                 A, B, L, r, n_slices, slice_end, idx, mask, Y, ldy, workspace, workspace_bytes,
                                 status_dev=None, stream=None) -> int:
    """slice_end: a sequence of n_slices column ends (host ints)."""
    ends = (ctypes.c_int * max(1, n_slices))(*[int(e) for e in slice_end])
    return load().epilora_layer_forward_slices(fmt, M, N, K, _p(X), ldx, _p(Wq), _p(w_scale), _p(w_block_scale),
                                               _p(w_global_scale), _p(x_global_scale), _p(A), _p(B), L, r,
                                               n_slices, ctypes.cast(ends, ctypes.c_void_p), _p(idx), _p(mask),
                                               _p(Y), ldy, _p(workspace), workspace_bytes, _p(status_dev),
                                               _stream(stream))


def epilora_layer_forward_fp8_adapters(fmt, M, N, K, X, ldx, Wq, w_scale, w_block_scale, w_global_scale,
                                       x_global_scale, Aq, a_scale, Bq, b_scale, L, r, idx, mask, Y, ldy, workspace,
                                       workspace_bytes, status_dev=None, stream=None) -> int:
    return load().epilora_layer_forward_fp8_adapters(fmt, M, N, K, _p(X), ldx, _p(Wq), _p(w_scale), _p(w_block_scale),
                                                     _p(w_global_scale), _p(x_global_scale), _p(Aq), _p(a_scale),
                                                     _p(Bq), _p(b_scale), L, r, _p(idx), _p(mask), _p(Y), ldy,
                                                     _p(workspace), workspace_bytes, _p(status_dev), _stream(stream))


def epilora_layer_forward_noalloc(fmt, M, N, K, X, ldx, Wq, w_scale, w_block_scale, w_global_scale,
                                  x_global_scale, A, B, L, r, idx, mask, Y, ldy, status_dev=None,
                                  stream=None) -> int:
    return load().epilora_layer_forward_noalloc(fmt, M, N, K, _p(X), ldx, _p(Wq), _p(w_scale), _p(w_block_scale),
                                                _p(w_global_scale), _p(x_global_scale), _p(A), _p(B), L, r,
                                                _p(idx), _p(mask), _p(Y), ldy, _p(status_dev), _stream(stream))
