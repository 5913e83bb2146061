// Row quantizers shared by the standalone quantizer kernel and the quantizer
// CTAs of the fused shrink grid, so both produce identical codes and scales.
//
// EpiLoRA, "Fusing Many LoRA Adapters into Low-Precision GEMMs for Serving and
// RL", §Design › Multi-adapter kernels › K1 and K2 and › The decode path:
// activations are quantized once per layer with one scale per token (FP8) or
// per 16-element block (NVFP4), by a kernel of their own or by extra thread
// blocks of the shrink. The page fixes only that the codes match the serving
// engine's own activation quantization; the arithmetic read here is IEEE
// round-to-nearest division / multiplication in fp32 and conversions that
// round to nearest even with saturation.
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace epi {

__device__ __forceinline__ void unpack8(const uint4& v, float (&x)[8]) {
  x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
  x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
  x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

// max over the CTA of non-negative values; red holds >= blockDim/32 floats
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = 0.0f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  return m;
}

__device__ __forceinline__ uint2 quant8_e4m3(const uint4& v, float s) {
  float x[8];
  unpack8(v, x);
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = cvt_e4m3x2(__fdiv_rn(x[2 * i], s), __fdiv_rn(x[2 * i + 1], s));
  return make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

// One CTA quantizes one row of K elements to E4M3 with a per-row scale.
// Rows of up to kRowRegChunks * blockDim 16-byte chunks are read from memory
// once (kept in registers); longer rows are read a second time for the codes.
template <int kRowRegChunks>
__device__ __forceinline__ void quant_row_fp8(const __nv_bfloat16* __restrict__ xrow, int K,
                                              uint8_t* __restrict__ qrow, float* __restrict__ scale_out,
                                              float* red) {
  const uint4* row = reinterpret_cast<const uint4*>(xrow);
  const int nch = K / 8;
  const int nt = static_cast<int>(blockDim.x);
  uint4 v[kRowRegChunks];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < kRowRegChunks; ++j) {
    const int c = static_cast<int>(threadIdx.x) + j * nt;
    v[j] = c < nch ? __ldg(row + c) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll 8
  for (int c = static_cast<int>(threadIdx.x) + kRowRegChunks * nt; c < nch; c += nt) {
    float x[8];
    unpack8(__ldg(row + c), x);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int j = 0; j < kRowRegChunks; ++j) {
    float x[8];
    unpack8(v[j], x);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
  amax = block_max(amax, red);
  const float s = __fdiv_rn(fmaxf(amax, kAmaxFloor), kE4M3Max);
  if (threadIdx.x == 0) *scale_out = s;
  uint2* out = reinterpret_cast<uint2*>(qrow);
#pragma unroll
  for (int j = 0; j < kRowRegChunks; ++j) {
    const int c = static_cast<int>(threadIdx.x) + j * nt;
    if (c < nch) out[c] = quant8_e4m3(v[j], s);
  }
#pragma unroll 8
  for (int c = static_cast<int>(threadIdx.x) + kRowRegChunks * nt; c < nch; c += nt)
    out[c] = quant8_e4m3(__ldg(row + c), s);
}

// amax over a whole row by one CTA, loads kept in flight (nothing held).
__device__ __forceinline__ float row_amax_bf16(const __nv_bfloat16* __restrict__ xrow, int K, float* red) {
  const uint4* row = reinterpret_cast<const uint4*>(xrow);
  const int nch = K / 8;
  float amax = 0.0f;
#pragma unroll 8
  for (int c = static_cast<int>(threadIdx.x); c < nch; c += static_cast<int>(blockDim.x)) {
    float x[8];
    unpack8(__ldg(row + c), x);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
  return block_max(amax, red);
}

// E4M3 codes of the row's elements [k0, k1) (multiples of 8) with scale s.
__device__ __forceinline__ void quant_slice_fp8(const __nv_bfloat16* __restrict__ xrow, int k0, int k1,
                                                uint8_t* __restrict__ qrow, float s) {
  const uint4* row = reinterpret_cast<const uint4*>(xrow);
  uint2* out = reinterpret_cast<uint2*>(qrow);
#pragma unroll 4
  for (int c = k0 / 8 + static_cast<int>(threadIdx.x); c < k1 / 8; c += static_cast<int>(blockDim.x))
    out[c] = quant8_e4m3(__ldg(row + c), s);
}

// One CTA quantizes one row to NVFP4: per 16-element block b,
// sb = E4M3(fl32(fl32(amax_b / 6) * g)), codes = E2M1(fl32(x * fl32(g / sb))).
// Blocks [b0, b1) of the row (all of it by default). Returns false if the
// global scale g is not a positive finite number (those blocks are then
// written as zeros).
__device__ __forceinline__ bool quant_row_nvfp4(const __nv_bfloat16* __restrict__ xrow, int K,
                                                uint8_t* __restrict__ qrow, uint8_t* __restrict__ srow, float g,
                                                int b0 = 0, int b1 = -1) {
  const bool g_ok = (g > 0.0f) && isfinite(g);
  const uint4* row = reinterpret_cast<const uint4*>(xrow);
  uint2* out = reinterpret_cast<uint2*>(qrow);
  const int nb = b1 < 0 ? K / kNvfp4Block : b1;
  for (int b = b0 + static_cast<int>(threadIdx.x); b < nb; b += blockDim.x) {
    float x[16];
    {
      float a[8], c[8];
      unpack8(__ldg(row + 2 * b), a);
      unpack8(__ldg(row + 2 * b + 1), c);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[i] = a[i];
        x[8 + i] = c[i];
      }
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
  return g_ok;
}

}  // namespace epi
