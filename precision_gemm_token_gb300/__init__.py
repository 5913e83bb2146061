"""GB300 (sm_103a) multi-tenant LoRA linear layer of an LLM decode step.

    Y = bf16( dequant(Q(X) . Q(W)^T) + mask * (X . A[idx]^T) . B[idx]^T )

The computation lives in libepilora.so (hand-written CUDA: per-token FP8 /
NVFP4 quantizer, multi-adapter shrink, tcgen05 GEMM with the LoRA epilogue
launched as the shrink's programmatic dependent) behind the C ABI of
include/epilora.h. This package is its ctypes binding (`_binding`, same
function names as the C ABI) plus `tensors`, thin helpers that allocate
outputs with torch and call the binding. There is no CPU fallback.
"""
from ._binding import (  # noqa: F401
    EPILORA_ERR_CUDA,
    EPILORA_ERR_INVALID_ARG,
    EPILORA_ERR_TIMEOUT,
    EPILORA_ERR_UNSUPPORTED,
    EPILORA_ERR_WORKSPACE,
    DECODE_PATH_AUTO,
    DECODE_PATH_SINGLE,
    DECODE_PATH_TWO,
    EPILORA_OK,
    FMT_FP8,
    FMT_NVFP4,
    EpiloraError,
    check,
    epilora_abi_version,
    epilora_gemm_lora_epilogue,
    epilora_layer_forward,
    epilora_layer_forward_fp8_adapters,
    epilora_layer_forward_kernels,
    epilora_test_drop_shrink_results,
    epilora_layer_forward_noalloc,
    epilora_layer_forward_slices,
    epilora_layer_workspace_bytes,
    epilora_lora_shrink,
    epilora_nvfp4_global_scale,
    epilora_quant_act,
    epilora_set_decode_path,
    epilora_status_string,
    epilora_workspace_bytes,
    load,
)
from .build import LIB_PATH, build  # noqa: F401
