// FP8 (E4M3) instantiations of the tcgen05 GEMM with the LoRA epilogue.
#include "gemm.cuh"

namespace epi {
int launch_gemm_fp8(const GemmArgs& a) { return launch_gemm_by_m<EPILORA_FMT_FP8_E4M3>(a); }
}  // namespace epi
