// NVFP4 (E2M1 + UE4M3 block scales) instantiations of the tcgen05 GEMM with
// the LoRA epilogue.
#include "gemm.cuh"

namespace epi {
int launch_gemm_nvfp4(const GemmArgs& a) { return launch_gemm_by_m<EPILORA_FMT_NVFP4>(a); }
}  // namespace epi
