// Per-token activation quantizers (FP8 E4M3 with a per-token scale; NVFP4
// E2M1 with E4M3 scales per 16-element block) and the NVFP4 global-scale
// helper.
//
// EpiLoRA, "Fusing Many LoRA Adapters into Low-Precision GEMMs for Serving and
// RL", §Design › Multi-adapter kernels › K1 and K2: activations are quantized
// once, per token, for the low-precision base GEMM. The exact arithmetic
// (IEEE division for the scale and the element / scale quotient, round to
// nearest even with saturation in the conversion) is the reading this library
// takes of "the same per-token scale and rounding"; it is bit-exact and
// deterministic. One CTA per token row; the row is read twice (amax, then
// codes), the second time from L1/L2.
#include "common.cuh"
#include "ptx.cuh"

namespace epi {

namespace {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  return m;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&x)[8]) {
  x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
  x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
  x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

__global__ void __launch_bounds__(kQuantThreads) quant_fp8_kernel(const __nv_bfloat16* __restrict__ X, int K,
                                                                   int ldx, uint8_t* __restrict__ Xq,
                                                                   float* __restrict__ x_scale) {
  __shared__ float red[kQuantThreads / 32];
  const size_t t = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(X + t * static_cast<size_t>(ldx));
  const int nch = K / 8;
  float amax = 0.0f;
  for (int c = threadIdx.x; c < nch; c += kQuantThreads) {
    float x[8];
    unpack8(__ldg(row + c), x);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
  amax = block_max(amax, red);
  const float s = __fdiv_rn(fmaxf(amax, kAmaxFloor), kE4M3Max);
  if (threadIdx.x == 0) x_scale[t] = s;
  uint2* out = reinterpret_cast<uint2*>(Xq + t * static_cast<size_t>(K));
  for (int c = threadIdx.x; c < nch; c += kQuantThreads) {
    float x[8];
    unpack8(__ldg(row + c), x);
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = cvt_e4m3x2(__fdiv_rn(x[2 * i], s), __fdiv_rn(x[2 * i + 1], s));
    out[c] = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
  }
}

__global__ void __launch_bounds__(kQuantThreads) quant_nvfp4_kernel(const __nv_bfloat16* __restrict__ X, int K,
                                                                     int ldx, uint8_t* __restrict__ Xq,
                                                                     uint8_t* __restrict__ sbx,
                                                                     const float* __restrict__ gptr,
                                                                     int* status) {
  const size_t t = blockIdx.x;
  const float g = *gptr;
  const bool g_ok = (g > 0.0f) && isfinite(g);
  if (!g_ok && threadIdx.x == 0) record_status(status, EPILORA_ERR_INVALID_ARG);
  const uint4* row = reinterpret_cast<const uint4*>(X + t * static_cast<size_t>(ldx));
  const int nb = K / kNvfp4Block;
  uint2* out = reinterpret_cast<uint2*>(Xq + t * static_cast<size_t>(K / 2));
  uint8_t* srow = sbx + t * static_cast<size_t>(nb);
  for (int b = threadIdx.x; b < nb; b += kQuantThreads) {
    float x[16];
    {
      float a[8], c[8];
      unpack8(__ldg(row + 2 * b), a);
      unpack8(__ldg(row + 2 * b + 1), c);
#pragma unroll
      for (int i = 0; i < 8; ++i) { x[i] = a[i]; x[8 + i] = c[i]; }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    uint32_t sb = 0, lo = 0, hi = 0;
    if (g_ok) {
      const float t2 = __fmul_rn(__fdiv_rn(amax, kE2M1Max), g);
      sb = cvt_e4m3x2(t2, 0.0f) & 0xFFu;
      const float sbf = e4m3_to_f32(sb);
      if (sbf > 0.0f) {
        const float inv = __fdiv_rn(g, sbf);
        uint32_t by[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) by[i] = cvt_e2m1x2(__fmul_rn(x[2 * i], inv), __fmul_rn(x[2 * i + 1], inv));
        lo = by[0] | (by[1] << 8) | (by[2] << 16) | (by[3] << 24);
        hi = by[4] | (by[5] << 8) | (by[6] << 16) | (by[7] << 24);
      }
    }
    out[b] = make_uint2(lo, hi);
    srow[b] = static_cast<uint8_t>(sb);
  }
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

}  // namespace

int launch_quant(int fmt, const void* X, int M, int K, int ldx, void* Xq, float* x_scale, uint8_t* x_block_scale,
                 const float* x_global_scale, int* status_dev, cudaStream_t stream) {
  if (M == 0) return EPILORA_OK;
  if (fmt == EPILORA_FMT_FP8_E4M3) {
    quant_fp8_kernel<<<M, kQuantThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(X), K, ldx,
                                                        static_cast<uint8_t*>(Xq), x_scale);
  } else {
    quant_nvfp4_kernel<<<M, kQuantThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(X), K, ldx,
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
