// Multi-adapter shrink (LoRA down-projection): S[t, j] = x_t . A[idx_t, j, :],
// optionally with one extra quantizer CTA per token in the same grid.
//
// EpiLoRA, "Fusing Many LoRA Adapters into Low-Precision GEMMs for Serving and
// RL": §Background and motivation › The cost of the separate adapter path
// (h = x A^T), §Design › Multi-adapter kernels › K1 and K2 (h from the bf16
// activations) and › The decode path (the shrink runs as its own small kernel
// that sees a complete x, lets the GEMM launch as its dependent at once, and
// a few extra thread blocks of it quantize the activations). PreFT,
// "Prefill-only finetuning", Core claim: tokens with mask 0 skip the adapter.
//
// One shrink CTA (128 threads) computes kRanksPerCta rank rows for one token.
// Its threads split the K dimension into 16-byte chunks (8 bf16): each chunk
// of x is loaded once and multiplied with the same chunk of the CTA's A rows
// (coalesced 128-bit loads). Partial sums are reduced with a fixed
// xor-butterfly inside each warp and then over the warps in index order, so S
// is bitwise reproducible and independent of the token's position in the
// batch. The CTAs are small (128 threads, at most 64 registers each) so that
// two GEMM CTAs still fit beside one on an SM: the GEMM runs concurrently.
#include "quant_row.cuh"

namespace epi {

namespace {

constexpr int kShrinkThreads = 128;
constexpr int kRanksPerCta = 4;
constexpr int kShrinkQuantChunks = 4;   // row chunks a quantizer thread holds in registers

__device__ __forceinline__ float dot8(const uint4& xv, const uint4& av, float acc) {
  acc = fmaf(bf16_lo(xv.x), bf16_lo(av.x), acc);
  acc = fmaf(bf16_hi(xv.x), bf16_hi(av.x), acc);
  acc = fmaf(bf16_lo(xv.y), bf16_lo(av.y), acc);
  acc = fmaf(bf16_hi(xv.y), bf16_hi(av.y), acc);
  acc = fmaf(bf16_lo(xv.z), bf16_lo(av.z), acc);
  acc = fmaf(bf16_hi(xv.z), bf16_hi(av.z), acc);
  acc = fmaf(bf16_lo(xv.w), bf16_lo(av.w), acc);
  acc = fmaf(bf16_hi(xv.w), bf16_hi(av.w), acc);
  return acc;
}

struct QuantSide {          // quantizer CTAs of the fused grid (fmt < 0: none)
  int fmt;
  uint8_t* Xq;
  float* x_scale;
  uint8_t* x_block_scale;
  const float* x_global_scale;
  uint32_t* x_ready;
};

__global__ void __launch_bounds__(kShrinkThreads, 8) shrink_kernel(const __nv_bfloat16* __restrict__ X, int K,
                                                                    int ldx, const __nv_bfloat16* __restrict__ A,
                                                                    int L, int r, const int32_t* __restrict__ idx,
                                                                    const uint8_t* __restrict__ mask,
                                                                    float* __restrict__ S, int* status,
                                                                    QuantSide qs) {
  // When this grid is itself a programmatic dependent (of the previous layer
  // call on the stream) its CTAs are already resident: wait here for that
  // kernel's completion; x and the workspace are only valid from now on
  // (no-op for an ordinary launch). Then let the dependent GEMM start
  // streaming its weights; it waits for this grid's completion only before
  // its epilogue. Waiting first keeps consecutive calls ordered, so calls may
  // share a workspace.
  pdl_wait_primary();
  pdl_allow_dependents();
  __shared__ float red[kShrinkThreads / 32][kRanksPerCta];

  const size_t t = blockIdx.x;
  int gy = static_cast<int>(blockIdx.y);
  if (qs.fmt >= 0) {
    if (gy == 0) {
      // quantizer CTA of token t
      const __nv_bfloat16* xrow = X + t * static_cast<size_t>(ldx);
      if (qs.fmt == EPILORA_FMT_FP8_E4M3) {
        quant_row_fp8<kShrinkQuantChunks>(xrow, K, qs.Xq + t * static_cast<size_t>(K), qs.x_scale + t, &red[0][0]);
      } else {
        const bool ok = quant_row_nvfp4(xrow, K, qs.Xq + t * static_cast<size_t>(K / 2),
                                        qs.x_block_scale + t * static_cast<size_t>(K / kNvfp4Block),
                                        *qs.x_global_scale);
        if (!ok && threadIdx.x == 0) record_status(status, EPILORA_ERR_INVALID_ARG);
      }
      fence_proxy_async_global();   // the GEMM reads these codes with TMA (async proxy)
      __threadfence();              // this thread's codes are visible GPU-wide ...
      __syncthreads();
      if (threadIdx.x == 0) atomicAdd(qs.x_ready, 1u);   // ... before the row counts as ready
      return;
    }
    gy -= 1;
  }

  const int j0 = gy * kRanksPerCta;
  const int l = idx[t];
  bool act = (l >= 0) && (mask == nullptr || mask[t] != 0);
  if (l >= L) {
    if (gy == 0 && threadIdx.x == 0) record_status(status, EPILORA_ERR_INVALID_ARG);
    act = false;
  }
  float* srow = S + t * static_cast<size_t>(r) + j0;
  if (!act) {
    if (threadIdx.x < kRanksPerCta) srow[threadIdx.x] = 0.0f;
    return;
  }
  const int nch = K / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(X + t * static_cast<size_t>(ldx));
  const uint4* ar = reinterpret_cast<const uint4*>(A + (static_cast<size_t>(l) * r + j0) * static_cast<size_t>(K));

  float acc[kRanksPerCta];
#pragma unroll
  for (int j = 0; j < kRanksPerCta; ++j) acc[j] = 0.0f;

#pragma unroll 2
  for (int c = threadIdx.x; c < nch; c += blockDim.x) {
    const uint4 xv = __ldg(xr + c);
    uint4 av[kRanksPerCta];
#pragma unroll
    for (int j = 0; j < kRanksPerCta; ++j) av[j] = __ldg(ar + static_cast<size_t>(j) * nch + c);
#pragma unroll
    for (int j = 0; j < kRanksPerCta; ++j) acc[j] = dot8(xv, av[j], acc[j]);
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < kRanksPerCta; ++j) {
    float v = acc[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp][j] = v;
  }
  __syncthreads();
  if (threadIdx.x < kRanksPerCta) {
    float s = 0.0f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += red[w][threadIdx.x];
    srow[threadIdx.x] = s;
  }
}

int shrink_carveout_done[64] = {0};

}  // namespace

int launch_shrink(const void* X, int M, int K, int ldx, const void* A, int L, int r, const int32_t* idx,
                  const uint8_t* mask, float* S, int* status_dev, cudaStream_t stream) {
  if (M == 0) return EPILORA_OK;
  if (prefer_max_shared(reinterpret_cast<const void*>(shrink_kernel), shrink_carveout_done) != EPILORA_OK)
    return EPILORA_ERR_CUDA;
  QuantSide qs{-1, nullptr, nullptr, nullptr, nullptr, nullptr};
  dim3 grid(M, r / kRanksPerCta);
  shrink_kernel<<<grid, kShrinkThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(X), K, ldx,
                                                      static_cast<const __nv_bfloat16*>(A), L, r, idx, mask, S,
                                                      status_dev, qs);
  return cudaGetLastError() == cudaSuccess ? EPILORA_OK : EPILORA_ERR_CUDA;
}

int launch_shrink_quant(const void* X, int M, int K, int ldx, const void* A, int L, int r, const int32_t* idx,
                        const uint8_t* mask, float* S, int fmt, void* Xq, float* x_scale, uint8_t* x_block_scale,
                        const float* x_global_scale, uint32_t* x_ready, int* status_dev, cudaStream_t stream) {
  if (M == 0) return EPILORA_OK;
  if (prefer_max_shared(reinterpret_cast<const void*>(shrink_kernel), shrink_carveout_done) != EPILORA_OK)
    return EPILORA_ERR_CUDA;
  QuantSide qs{fmt, static_cast<uint8_t*>(Xq), x_scale, x_block_scale, x_global_scale, x_ready};
  // launched as a programmatic dependent of whatever precedes it on the
  // stream: its CTAs become resident early and wait (griddepcontrol.wait)
  // for that kernel's completion before touching x or the workspace
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(M, r / kRanksPerCta + 1);
  cfg.blockDim = dim3(kShrinkThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, shrink_kernel, static_cast<const __nv_bfloat16*>(X), K, ldx,
                         static_cast<const __nv_bfloat16*>(A), L, r, idx, mask, S, status_dev, qs) != cudaSuccess)
    return EPILORA_ERR_CUDA;
  return EPILORA_OK;
}

}  // namespace epi
