// Standalone per-token activation quantizer (FP8 E4M3 with a per-token scale;
// NVFP4 E2M1 with E4M3 scales per 16-element block) and the NVFP4 global-scale
// helper. The row arithmetic lives in quant_row.cuh (shared with the
// quantizer CTAs of the fused shrink grid).
//
// EpiLoRA, "Fusing Many LoRA Adapters into Low-Precision GEMMs for Serving and
// RL", §Design › Multi-adapter kernels › K1 and K2: activations are quantized
// once, per token, for the low-precision base GEMM. One CTA per row.
#include "quant_row.cuh"

namespace epi {

namespace {

constexpr int kQuantMaxThreads = 512;
constexpr int kQuantChunks = 8;          // 16-byte chunks of the row held per thread

__global__ void __launch_bounds__(kQuantMaxThreads) quant_fp8_kernel(const __nv_bfloat16* __restrict__ X, int K,
                                                                     int ldx, uint8_t* __restrict__ Xq,
                                                                     float* __restrict__ x_scale) {
  __shared__ float red[kQuantMaxThreads / 32];
  const size_t t = blockIdx.x;
  quant_row_fp8<kQuantChunks>(X + t * static_cast<size_t>(ldx), K, Xq + t * static_cast<size_t>(K), x_scale + t,
                              red);
}

__global__ void __launch_bounds__(256) quant_nvfp4_kernel(const __nv_bfloat16* __restrict__ X, int K, int ldx,
                                                        uint8_t* __restrict__ Xq, uint8_t* __restrict__ sbx,
                                                        const float* __restrict__ gptr, int* status) {
  const size_t t = blockIdx.x;
  const bool ok = quant_row_nvfp4(X + t * static_cast<size_t>(ldx), K, Xq + t * static_cast<size_t>(K / 2),
                                  sbx + t * static_cast<size_t>(K / kNvfp4Block), *gptr);
  if (!ok && threadIdx.x == 0) record_status(status, EPILORA_ERR_INVALID_ARG);
}

// amax of a bf16 tensor into a zero-initialised uint (non-negative floats
// order like their bit patterns, so an integer max is exact and
// order-independent), then g = 2688 / max(amax, floor).
__global__ void __launch_bounds__(256) tensor_amax_kernel(const __nv_bfloat16* __restrict__ T, size_t n,
                                                          unsigned int* out) {
  __shared__ float red[8];
  float amax = 0.0f;
  const size_t nv = n / 8;
  const uint4* v = reinterpret_cast<const uint4*>(T);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nv; i += (size_t)gridDim.x * blockDim.x) {
    float x[8];
    unpack8(__ldg(v + i), x);
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(x[k]));
  }
  if (blockIdx.x == 0) {
    for (size_t i = nv * 8 + threadIdx.x; i < n; i += blockDim.x) amax = fmaxf(amax, fabsf(__bfloat162float(T[i])));
  }
  amax = block_max(amax, red);
  if (threadIdx.x == 0) atomicMax(out, __float_as_uint(amax));
}

__global__ void global_scale_finish_kernel(float* g) {
  const float amax = __uint_as_float(*reinterpret_cast<unsigned int*>(g));
  *g = __fdiv_rn(kE4M3Max * kE2M1Max, fmaxf(amax, kAmaxFloor));
}

// threads per row CTA of the FP8 quantizer: about K/64 (8 chunks each), 32..512
int quant_fp8_threads(int K) {
  int threads = (K / 8 + kQuantChunks - 1) / kQuantChunks;
  threads = (threads + 31) / 32 * 32;
  return threads < 32 ? 32 : threads > kQuantMaxThreads ? kQuantMaxThreads : threads;
}

int quant_carveout_done[2][64] = {{0}};

}  // namespace

int launch_quant(int fmt, const void* X, int M, int K, int ldx, void* Xq, float* x_scale, uint8_t* x_block_scale,
                 const float* x_global_scale, int* status_dev, cudaStream_t stream) {
  if (M == 0) return EPILORA_OK;
  if (prefer_max_shared(reinterpret_cast<const void*>(quant_fp8_kernel), quant_carveout_done[0]) != EPILORA_OK ||
      prefer_max_shared(reinterpret_cast<const void*>(quant_nvfp4_kernel), quant_carveout_done[1]) != EPILORA_OK)
    return EPILORA_ERR_CUDA;
  if (fmt == EPILORA_FMT_FP8_E4M3) {
    quant_fp8_kernel<<<M, quant_fp8_threads(K), 0, stream>>>(static_cast<const __nv_bfloat16*>(X), K, ldx,
                                                              static_cast<uint8_t*>(Xq), x_scale);
  } else {
    quant_nvfp4_kernel<<<M, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(X), K, ldx,
                                              static_cast<uint8_t*>(Xq), x_block_scale, x_global_scale,
                                              status_dev);
  }
  return cudaGetLastError() == cudaSuccess ? EPILORA_OK : EPILORA_ERR_CUDA;
}

int launch_global_scale(const void* T, size_t n, float* g_out, cudaStream_t stream) {
  if (cudaMemsetAsync(g_out, 0, sizeof(float), stream) != cudaSuccess) return EPILORA_ERR_CUDA;
  size_t blocks = (n / 8 + 255) / 256;
  const size_t cap = static_cast<size_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  tensor_amax_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(T), n,
                                                                         reinterpret_cast<unsigned int*>(g_out));
  global_scale_finish_kernel<<<1, 1, 0, stream>>>(g_out);
  return cudaGetLastError() == cudaSuccess ? EPILORA_OK : EPILORA_ERR_CUDA;
}

}  // namespace epi
