// FP8 (E4M3) instantiations of the tcgen05 GEMM with the LoRA epilogue.
#include "gemm.cuh"

namespace epi {
int launch_gemm_fp8(const GemmArgs& a) { return launch_gemm_by_m<EPILORA_FMT_FP8_E4M3>(a); }
}  // namespace epi

#ifdef EPILORA_GEMM_TRACE
// tuning builds only: copy (and clear) the per-CTA phase timestamps
extern "C" EPILORA_API int epilora_debug_gemm_trace_fp8(void* host_out, int clear) {
  if (cudaMemcpyFromSymbol(host_out, epi::g_gemm_trace, sizeof(epi::g_gemm_trace)) != cudaSuccess) return -3;
  if (clear) {
    static unsigned long long zeros[epi::kTraceSlots][epi::kTraceCtas][16];
    if (cudaMemcpyToSymbol(epi::g_gemm_trace, zeros, sizeof(zeros)) != cudaSuccess) return -3;
    epi::gemm_trace_launches() = 0;
  }
  return 0;
}
#endif
