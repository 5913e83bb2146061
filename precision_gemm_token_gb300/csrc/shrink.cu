// Multi-adapter shrink (LoRA down-projection): S[t, j] = x_t . A[idx_t, j, :].
//
// EpiLoRA, "Fusing Many LoRA Adapters into Low-Precision GEMMs for Serving and
// RL": §Background and motivation › The cost of the separate adapter path
// (h = x A^T), §Design › Multi-adapter kernels › K1 and K2 (h from the bf16
// activations) and › The decode path (the shrink runs as its own small kernel,
// launched without a dependency attribute so it sees a complete x, and lets
// the GEMM launch as its dependent immediately). PreFT, "Prefill-only
// finetuning", Core claim: tokens with mask 0 skip the adapter.
//
// One CTA computes kRanksPerCta rank rows for one token. Its 256 threads split
// the K dimension into 16-byte chunks (8 bf16): each chunk of x is loaded once
// and multiplied with the same chunk of the CTA's A rows (coalesced 128-bit
// loads). Partial sums are reduced with a fixed xor-butterfly inside each warp
// and then over the warps in index order, so S is bitwise reproducible and
// independent of the token's position in the batch.
#include "common.cuh"
#include "ptx.cuh"

namespace epi {

namespace {

constexpr int kShrinkThreads = 256;
constexpr int kRanksPerCta = 8;

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

__global__ void __launch_bounds__(kShrinkThreads) shrink_kernel(const __nv_bfloat16* __restrict__ X, int K, int ldx,
                                                                 const __nv_bfloat16* __restrict__ A, int L, int r,
                                                                 const int32_t* __restrict__ idx,
                                                                 const uint8_t* __restrict__ mask,
                                                                 float* __restrict__ S, int* status) {
  // Let the dependent GEMM start streaming its weights right away; it waits
  // for this grid's completion only before its epilogue.
  pdl_allow_dependents();
  __shared__ float red[kShrinkThreads / 32][kRanksPerCta];

  const size_t t = blockIdx.x;
  const int j0 = blockIdx.y * kRanksPerCta;
  const int l = idx[t];
  bool act = (l >= 0) && (mask == nullptr || mask[t] != 0);
  if (l >= L) {
    if (blockIdx.y == 0 && threadIdx.x == 0) record_status(status, EPILORA_ERR_INVALID_ARG);
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
  for (int c = threadIdx.x; c < nch; c += kShrinkThreads) {
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
#pragma unroll
    for (int w = 0; w < kShrinkThreads / 32; ++w) s += red[w][threadIdx.x];
    srow[threadIdx.x] = s;
  }
}

}  // namespace

int launch_shrink(const void* X, int M, int K, int ldx, const void* A, int L, int r, const int32_t* idx,
                  const uint8_t* mask, float* S, int* status_dev, cudaStream_t stream) {
  if (M == 0) return EPILORA_OK;
  dim3 grid(M, r / kRanksPerCta);
  shrink_kernel<<<grid, kShrinkThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(X), K, ldx,
                                                      static_cast<const __nv_bfloat16*>(A), L, r, idx, mask, S,
                                                      status_dev);
  return cudaGetLastError() == cudaSuccess ? EPILORA_OK : EPILORA_ERR_CUDA;
}

}  // namespace epi
