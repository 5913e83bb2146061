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
// Decode batches (shrink_kernel): one rank CTA (128 threads) computes
// kRanksPerCta rank rows for one token. Its threads split the K dimension
// into 16-byte chunks (8 bf16): each chunk of x is loaded once and multiplied
// with the same chunk of the CTA's A rows (coalesced 128-bit loads). Partial
// sums are reduced with a fixed xor-butterfly inside each warp and then over
// the warps in index order, so S is bitwise reproducible and independent of
// the token's position in the batch. The CTAs are small (128 threads, at
// most 64 registers each) so that the GEMM's CTAs still fit beside them.
// Batches of more than 32 tokens (shrink_block_kernel): blocks of 16
// consecutive tokens that carry at most two adapters go to tensor-core CTAs
// (see there); the others to rank CTAs as above, in the same grid.
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
  int32_t* perm;            // non-null: rows are written in adapter-sorted order, perm[row] = token
};

// Sort key of token t for the adapter-sorted row order: its adapter slot if
// it carries one (idx in [0, L), mask set), else L; ties keep token order.
__device__ __forceinline__ int sort_key(const int32_t* idx, const uint8_t* mask, int L, int t) {
  const int l = idx[t];
  return (l >= 0 && l < L && (mask == nullptr || mask[t] != 0)) ? l : L;
}

// Row of token t in the sorted order: the number of tokens whose (key, index)
// precedes its own (one CTA; every thread takes a strided share of the
// tokens, then a fixed-order reduction).
__device__ __forceinline__ int sorted_row(const int32_t* idx, const uint8_t* mask, int L, int M, int t,
                                          int* red_i) {
  const int key = sort_key(idx, mask, L, t);
  int cnt = 0;
  int u0 = 0;
  if ((reinterpret_cast<uintptr_t>(idx) & 15u) == 0 && (reinterpret_cast<uintptr_t>(mask) & 3u) == 0) {
    // four tokens per load
    const int n4 = M / 4;
#pragma unroll 2
    for (int v = threadIdx.x; v < n4; v += blockDim.x) {
      const int4 iv = reinterpret_cast<const int4*>(idx)[v];
      const uint32_t mv = mask != nullptr ? reinterpret_cast<const uint32_t*>(mask)[v] : 0x01010101u;
      const int ls[4] = {iv.x, iv.y, iv.z, iv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int l = ls[e];
        const int k = (l >= 0 && l < L && ((mv >> (8 * e)) & 0xFFu) != 0u) ? l : L;
        const int u = 4 * v + e;
        cnt += (k < key || (k == key && u < t)) ? 1 : 0;
      }
    }
    u0 = n4 * 4;
  }
#pragma unroll 4
  for (int u = u0 + threadIdx.x; u < M; u += blockDim.x) {
    const int k = sort_key(idx, mask, L, u);
    cnt += (k < key || (k == key && u < t)) ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) red_i[threadIdx.x >> 5] = cnt;
  __syncthreads();
  int total = 0;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += red_i[w];
  __syncthreads();
  return total;
}

// Before the dependency wait: bring this CTA's inputs into L2 (its slice of
// x, and for a rank CTA its A rows of the token's adapter) so that the loads
// after the wait do not queue behind the weight stream of the GEMM that is
// starting meanwhile. Only hints: the index read here may still change (the
// previous kernel may write it); the loads after the wait re-read it.
__device__ __forceinline__ void prefetch_inputs(const __nv_bfloat16* X, int K, int ldx, const __nv_bfloat16* A,
                                                int L, int r, const int32_t* idx, int qparts, int kslice) {
  const size_t t = blockIdx.x;
  int gy = static_cast<int>(blockIdx.y);
  const int parts = qparts > 0 ? qparts : 1;
  if (qparts > 0 && gy < qparts) {
    const int k0 = gy * kslice, k1 = min(K, k0 + kslice);
    if (k1 > k0) prefetch_l2_bulk(X + t * static_cast<size_t>(ldx) + k0, static_cast<uint32_t>((k1 - k0) * 2));
    return;
  }
  gy -= qparts;
  const int groups = r / kRanksPerCta;
  if (groups == 0) return;
  const int part = gy / groups;
  const int j0 = (gy - part * groups) * kRanksPerCta;
  const int k0 = part * kslice, k1 = min(K, (part + 1) * kslice);
  if (k1 <= k0) return;
  int l;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(l) : "l"(idx + t));
  if (l < 0 || l >= L) return;
  prefetch_l2_bulk(X + t * static_cast<size_t>(ldx) + k0, static_cast<uint32_t>((k1 - k0) * 2));
  for (int j = 0; j < kRanksPerCta; ++j)
    prefetch_l2_bulk(A + (static_cast<size_t>(l) * r + j0 + j) * static_cast<size_t>(K) + k0,
                     static_cast<uint32_t>((k1 - k0) * 2));
  (void)parts;
}

// Quantizer CTA of a fused grid: K slice gy of token t (of `parts`), written
// to row q (t, or its place in the adapter-sorted order when qs.perm is set).
template <int kRegChunks>   // 16-byte chunks of the row each thread holds in registers
__device__ __forceinline__ void quant_role(const __nv_bfloat16* __restrict__ X, int K, int ldx,
                                           const int32_t* __restrict__ idx, const uint8_t* __restrict__ mask, int L,
                                           int M, size_t t, int gy, int parts, int kslice, const QuantSide& qs,
                                           int* status, float* red) {
  size_t q = t;
  if (qs.perm != nullptr) {
    q = static_cast<size_t>(sorted_row(idx, mask, L, M, static_cast<int>(t), reinterpret_cast<int*>(red)));
    if (gy == 0 && threadIdx.x == 0) qs.perm[q] = static_cast<int32_t>(t);
  }
  const __nv_bfloat16* xrow = X + t * static_cast<size_t>(ldx);
  const int k0 = gy * kslice;
  const int k1 = min(K, k0 + kslice);
  if (qs.fmt == EPILORA_FMT_FP8_E4M3) {
    if (parts == 1) {
      quant_row_fp8<kRegChunks>(xrow, K, qs.Xq + q * static_cast<size_t>(K), qs.x_scale + q, red);
    } else {
      // every slice CTA takes the whole row's amax (the same exact max)
      const float amax = row_amax_bf16(xrow, K, red);
      const float sc = __fdiv_rn(fmaxf(amax, kAmaxFloor), kE4M3Max);
      if (gy == 0 && threadIdx.x == 0) qs.x_scale[q] = sc;
      if (k0 < k1) quant_slice_fp8(xrow, k0, k1, qs.Xq + q * static_cast<size_t>(K), sc);
    }
  } else {
    const bool ok = quant_row_nvfp4(xrow, K, qs.Xq + q * static_cast<size_t>(K / 2),
                                    qs.x_block_scale + q * static_cast<size_t>(K / kNvfp4Block),
                                    *qs.x_global_scale, k0 / kNvfp4Block, k1 / kNvfp4Block);
    if (!ok && gy == 0 && threadIdx.x == 0) record_status(status, EPILORA_ERR_INVALID_ARG);
  }
}

// Rank CTA: ranks j0 .. j0 + 3 of token t over K slice `part` (kslice
// elements), written to S[part][t][j0 ..]; zeros for a token without an
// active adapter. `red` holds (blockDim.x / 32) * 4 floats.
// x (8 bf16) . a (8 E4M3 codes), accumulated in element order
__device__ __forceinline__ float dot8_e4m3(const uint4& xv, const uint2& av, float acc) {
  const uint32_t w[2] = {av.x, av.y};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float f0 = e4m3_to_f32(w[h] & 0xFFu), f1 = e4m3_to_f32((w[h] >> 8) & 0xFFu);
    const float f2 = e4m3_to_f32((w[h] >> 16) & 0xFFu), f3 = e4m3_to_f32(w[h] >> 24);
    const uint32_t xa = h == 0 ? xv.x : xv.z, xb = h == 0 ? xv.y : xv.w;
    acc = fmaf(bf16_lo(xa), f0, acc);
    acc = fmaf(bf16_hi(xa), f1, acc);
    acc = fmaf(bf16_lo(xb), f2, acc);
    acc = fmaf(bf16_hi(xb), f3, acc);
  }
  return acc;
}

// a_scale != nullptr: A holds E4M3 codes (K bytes per row) and each row's
// fp32 scale multiplies the slice's sum.
__device__ __forceinline__ void rank_role(const __nv_bfloat16* __restrict__ X, int K, int ldx,
                                          const __nv_bfloat16* __restrict__ A, int L, int r,
                                          const int32_t* __restrict__ idx, const uint8_t* __restrict__ mask,
                                          float* __restrict__ S, int* status, int M, size_t t, int j0, int part,
                                          int kslice, bool report, float* red, const float* a_scale = nullptr) {
  const int l = idx[t];
  bool act = (l >= 0) && (mask == nullptr || mask[t] != 0);
  if (l >= L) {
    if (report && threadIdx.x == 0) record_status(status, EPILORA_ERR_INVALID_ARG);
    act = false;
  }
  float* srow = S + (static_cast<size_t>(part) * M + t) * static_cast<size_t>(r) + j0;
  if (!act) {
    if (threadIdx.x < kRanksPerCta) srow[threadIdx.x] = 0.0f;
    return;
  }
  const int c0 = part * kslice / 8;
  const int c1 = min(K, (part + 1) * kslice) / 8;
  const int nch = K / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(X + t * static_cast<size_t>(ldx));
  const size_t arow = (static_cast<size_t>(l) * r + j0) * static_cast<size_t>(K);   // first A row (elements)

  float acc[kRanksPerCta];
#pragma unroll
  for (int j = 0; j < kRanksPerCta; ++j) acc[j] = 0.0f;

  if (a_scale == nullptr) {
    const uint4* ar = reinterpret_cast<const uint4*>(A + arow);
#pragma unroll 2
    for (int c = c0 + static_cast<int>(threadIdx.x); c < c1; c += blockDim.x) {
      const uint4 xv = __ldg(xr + c);
      uint4 av[kRanksPerCta];
#pragma unroll
      for (int j = 0; j < kRanksPerCta; ++j) av[j] = __ldg(ar + static_cast<size_t>(j) * nch + c);
#pragma unroll
      for (int j = 0; j < kRanksPerCta; ++j) acc[j] = dot8(xv, av[j], acc[j]);
    }
  } else {
    const uint2* ar = reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(A) + arow);
#pragma unroll 2
    for (int c = c0 + static_cast<int>(threadIdx.x); c < c1; c += blockDim.x) {
      const uint4 xv = __ldg(xr + c);
      uint2 av[kRanksPerCta];
#pragma unroll
      for (int j = 0; j < kRanksPerCta; ++j) av[j] = __ldg(ar + static_cast<size_t>(j) * nch + c);
#pragma unroll
      for (int j = 0; j < kRanksPerCta; ++j) acc[j] = dot8_e4m3(xv, av[j], acc[j]);
    }
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < kRanksPerCta; ++j) {
    float v = acc[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp * kRanksPerCta + j] = v;
  }
  __syncthreads();
  if (threadIdx.x < kRanksPerCta) {
    float sum = 0.0f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) sum += red[w * kRanksPerCta + threadIdx.x];
    srow[threadIdx.x] = a_scale != nullptr ? sum * __ldg(a_scale + static_cast<size_t>(l) * r + j0 + threadIdx.x) : sum;
  }
}

// grid (M, [parts quantizer CTAs +] (r / 4) * parts rank CTAs); CTA (t, y):
// quantizer slice y of token t, or ranks 4 * (g % (r / 4)) .. + 3 of token t
// over K slice g / (r / 4), g = y - parts. Slices are `kslice` elements
// (a multiple of 256); partial sums go to S[part][t][:].
__global__ void __launch_bounds__(kShrinkThreads, 8) shrink_kernel(const __nv_bfloat16* __restrict__ X, int K,
                                                                    int ldx, const __nv_bfloat16* __restrict__ A,
                                                                    int L, int r, const int32_t* __restrict__ idx,
                                                                    const uint8_t* __restrict__ mask,
                                                                    float* __restrict__ S, int* status,
                                                                    QuantSide qs, int parts, int kslice,
                                                                    int early_release, const float* a_scale) {
  // Let the dependent GEMM launch at once: before it reads anything this grid
  // writes it waits for this grid's completion, and until then it only
  // streams weights. Then, when this grid is itself a programmatic dependent
  // (of the previous call's GEMM), wait for that grid's completion: x, idx,
  // mask and the workspace are only valid from here on (no-op for an
  // ordinary launch).
  if (threadIdx.x == 0) prefetch_inputs(X, K, ldx, A, L, r, idx, qs.fmt >= 0 ? parts : 0, kslice);
  // early_release: the GEMM may launch as soon as every CTA of this grid has
  // started (else as they exit)
  if (early_release) pdl_allow_dependents();
  pdl_wait_primary();
  __shared__ float red[kShrinkThreads / 32][kRanksPerCta];

  const size_t t = blockIdx.x;
  int gy = static_cast<int>(blockIdx.y);
  if (qs.fmt >= 0) {
    if (gy < parts) {
      quant_role<kShrinkQuantChunks>(X, K, ldx, idx, mask, L, static_cast<int>(gridDim.x), static_cast<int>(t), gy,
                                     parts, kslice, qs, status, &red[0][0]);
      __syncthreads();
      return;
    }
    gy -= parts;
  }

  const int groups = r / kRanksPerCta;
  if (groups == 0) return;
  const int part = gy / groups;
  rank_role(X, K, ldx, A, L, r, idx, mask, S, status, static_cast<int>(gridDim.x), t,
            (gy - part * groups) * kRanksPerCta, part, kslice, gy == 0, &red[0][0], a_scale);
}

// Wide batches (M > 32): tokens in blocks of 16 consecutive tokens. A block
// whose active tokens carry at most kBlockAdapters distinct adapters (the
// tokens of a prefill request share one and sit next to each other) is taken
// by one CTA per K slice that computes all r ranks of S for it on the tensor
// cores (m16n8k16 bf16 mma.sync: products of bf16 values are exact in fp32,
// fp32 accumulate), reading a row of the adapter's A once per block instead
// of once per token: one pass per adapter, the x rows of the other tokens
// zeroed; the four warps take consecutive quarters of the slice and their
// partial tiles are added in warp order. Any other block is taken token by
// token by rank CTAs as in shrink_kernel (16 ranks over the whole K each, in
// groups of 4, written to part 0; its block CTAs zero the other parts).
// Grid: nblk * parts block CTAs (block, part) first, then per token its
// quantizer CTA and r / 16 rank CTAs.
constexpr int kBlockTokens = 16;
constexpr int kBlockAdapters = 2;

// distinct active adapters of tokens t0 .. t0 + 15 (< M), for a whole warp
__device__ __forceinline__ int block_adapters(const int32_t* __restrict__ idx, const uint8_t* __restrict__ mask,
                                              int L, int M, int t0) {
  const int lane = threadIdx.x & 31;
  const int t = t0 + (lane & 15);
  int l = -1;
  if (t < M) {
    l = idx[t];
    if (l < 0 || l >= L || (mask != nullptr && mask[t] == 0)) l = -1;
  }
  const unsigned same = __match_any_sync(0xffffffffu, l);
  const bool first = __ffs(same) - 1 == lane;
  return __popc(__ballot_sync(0xffffffffu, first && l >= 0));
}

__global__ void __launch_bounds__(kShrinkThreads, 6) shrink_block_kernel(const __nv_bfloat16* __restrict__ X, int K,
                                                                      int ldx, const __nv_bfloat16* __restrict__ A,
                                                                      int L, int r, const int32_t* __restrict__ idx,
                                                                      const uint8_t* __restrict__ mask,
                                                                      float* __restrict__ S, int* status,
                                                                      QuantSide qs, int M, int parts, int kslice,
                                                                      int early_release) {
  if (early_release) pdl_allow_dependents();
  pdl_wait_primary();
  extern __shared__ float red_dyn[];        // [4 warps][16 tokens][r] (at least 64 floats)
  __shared__ int lsh[kBlockTokens];
  const int nblk = r > 0 ? (M + kBlockTokens - 1) / kBlockTokens : 0;
  const int q = static_cast<int>(blockIdx.x);
  if (q >= nblk * parts) {
    // per token: its quantizer CTA, then its rank CTAs of 16 ranks each (a
    // token of a block with many adapters; four rank groups in turn)
    const int groups = r / 16;
    const int u = q - nblk * parts;
    const int t = u / (1 + groups);
    const int role = u - t * (1 + groups);
    if (role == 0) {
      // rows of up to 8192 elements stay in registers between the amax and the codes
      if (qs.fmt >= 0)
        quant_role<8>(X, K, ldx, idx, mask, L, M, static_cast<size_t>(t), 0, 1, K, qs, status, red_dyn);
      return;
    }
    if (block_adapters(idx, mask, L, M, (t / kBlockTokens) * kBlockTokens) <= kBlockAdapters) return;
    for (int gq = 0; gq < 16 / kRanksPerCta; ++gq) {
      if (gq > 0) __syncthreads();     // the previous group's partial sums are read out
      rank_role(X, K, ldx, A, L, r, idx, mask, S, status, M, static_cast<size_t>(t),
                (role - 1) * 16 + gq * kRanksPerCta, 0, K, role == 1 && gq == 0, red_dyn);
    }
    return;
  }
  const int blk = q / parts;
  const int part = q - blk * parts;
  const int t0 = blk * kBlockTokens;
  if (block_adapters(idx, mask, L, M, t0) > kBlockAdapters) {
    // taken token by token (part 0): zero the other parts
    if (part > 0)
      for (int e = threadIdx.x; e < kBlockTokens * r; e += kShrinkThreads) {
        const int t = t0 + e / r;
        if (t < M) S[(static_cast<size_t>(part) * M + t) * r + (e % r)] = 0.0f;
      }
    return;
  }
  if (threadIdx.x < kBlockTokens) {
    const int t = t0 + static_cast<int>(threadIdx.x);
    int l = -1;
    if (t < M) {
      l = idx[t];
      if (l >= L) {
        if (part == 0) record_status(status, EPILORA_ERR_INVALID_ARG);
        l = -1;
      }
      if (l >= 0 && mask != nullptr && mask[t] == 0) l = -1;
    }
    lsh[threadIdx.x] = l;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int k0 = part * kslice, k1 = min(K, k0 + kslice);
  // K in chunks of 32: lane (g, tq) loads 16 bytes, k = 8 tq .. 8 tq + 7 of
  // the chunk, of its two x rows and of each of its two rank rows; the first
  // half feeds one m16n8k16 MMA and the second half another (the same k order
  // on both operands, so each MMA sums 16 distinct k and the two cover the
  // chunk). 16 ranks per pass over the slice.
  const int nch = (k1 - k0) / 32;
  const int c0 = (nch * warp) / 4, c1 = (nch * (warp + 1)) / 4;
  const int lj = lsh[lane & 15];
  const uint32_t act = __ballot_sync(0xffffffffu, lj >= 0) & 0xffffu;
  float* redw = red_dyn + warp * kBlockTokens * r;
  constexpr int U = 2;     // chunks in flight per lane
  for (int rg = 0; rg < r / 16; ++rg) {
    float c[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) c[nt][i] = 0.0f;
    uint32_t rem = act;
    while (rem != 0u) {
      const int l = lsh[__ffs(rem) - 1];
      const uint32_t rows = __ballot_sync(0xffffffffu, lj == l) & 0xffffu;
      rem &= ~rows;
      const bool ona = (rows >> g) & 1u, onb = (rows >> (g + 8)) & 1u;
      // rows of tokens outside the block's valid range are never "on"
      const uint4* xa =
          reinterpret_cast<const uint4*>(X + static_cast<size_t>(ona ? t0 + g : 0) * ldx + k0 + 8 * tq);
      const uint4* xb =
          reinterpret_cast<const uint4*>(X + static_cast<size_t>(onb ? t0 + g + 8 : 0) * ldx + k0 + 8 * tq);
      const uint4* a0 =
          reinterpret_cast<const uint4*>(A + (static_cast<size_t>(l) * r + rg * 16 + g) * K + k0 + 8 * tq);
      const uint4* a1 = a0 + K;    // 8 rank rows further
      auto chunk = [&](const uint4& va, const uint4& vb, const uint4& w0, const uint4& w1) {
        const uint32_t aA[4] = {va.x, vb.x, va.y, vb.y};
        const uint32_t aB[4] = {va.z, vb.z, va.w, vb.w};
        mma_bf16_m16n8k16(c[0], aA, w0.x, w0.y);
        mma_bf16_m16n8k16(c[0], aB, w0.z, w0.w);
        mma_bf16_m16n8k16(c[1], aA, w1.x, w1.y);
        mma_bf16_m16n8k16(c[1], aB, w1.z, w1.w);
      };
      int ch = c0;
      for (; ch + U <= c1; ch += U) {
        uint4 va[U], vb[U], w0[U], w1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          va[u] = ona ? __ldg(xa + (ch + u) * 4) : make_uint4(0u, 0u, 0u, 0u);
          vb[u] = onb ? __ldg(xb + (ch + u) * 4) : make_uint4(0u, 0u, 0u, 0u);
          w0[u] = __ldg(a0 + (ch + u) * 4);
          w1[u] = __ldg(a1 + (ch + u) * 4);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) chunk(va[u], vb[u], w0[u], w1[u]);
      }
      for (; ch < c1; ++ch) {
        const uint4 va = ona ? __ldg(xa + ch * 4) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 vb = onb ? __ldg(xb + ch * 4) : make_uint4(0u, 0u, 0u, 0u);
        chunk(va, vb, __ldg(a0 + ch * 4), __ldg(a1 + ch * 4));
      }
    }
    // this warp's partial tile [token][rank rg*16 ..]
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int j = rg * 16 + nt * 8 + 2 * tq;
      redw[g * r + j] = c[nt][0];
      redw[g * r + j + 1] = c[nt][1];
      redw[(g + 8) * r + j] = c[nt][2];
      redw[(g + 8) * r + j + 1] = c[nt][3];
    }
  }
  __syncthreads();
  // the warps' partial tiles added in warp order
  const int tile = kBlockTokens * r;
  for (int e = threadIdx.x; e < tile; e += kShrinkThreads) {
    const int tl = e / r;
    const int t = t0 + tl;
    if (t < M) {
      const float v = ((red_dyn[e] + red_dyn[tile + e]) + red_dyn[2 * tile + e]) + red_dyn[3 * tile + e];
      S[(static_cast<size_t>(part) * M + t) * r + (e - tl * r)] = v;
    }
  }
}

constexpr int kShrinkSliceTarget = 1024;   // elements of K per slice when splitting
constexpr int kShrinkMaxParts = 8;

int kslice_for(int K, int parts) {
  const int per = (K + parts - 1) / parts;
  return (per + 255) / 256 * 256;
}

int shrink_carveout_done[64] = {0};

}  // namespace

int shrink_kslice(int K, int parts) { return kslice_for(K, parts); }

int shrink_parts_max(int K) {
  const int p = (K + kShrinkSliceTarget - 1) / kShrinkSliceTarget;
  return p < 1 ? 1 : p > kShrinkMaxParts ? kShrinkMaxParts : p;
}

int shrink_parts(int M, int K, int r) {
  if (M > 32) {
    // token-block CTAs: K slices of about 2048 (ranks <= 64; rank 128 keeps
    // one slice, the wide GEMM then reads S rows straight from memory)
    if (r <= 0 || r > 64) return 1;
    int p = (K + 2047) / 2048;
    if (p > kShrinkMaxParts) p = kShrinkMaxParts;
    while (p > 1 && kslice_for(K, p) * (p - 1) >= K) --p;
    return p < 1 ? 1 : p;
  }
  // split K only while the grid stays small (decode): a token's chain of
  // dependent loads then shortens without adding a wave of CTAs
  const int per_part = M * (r / kRanksPerCta + 1);
  int p = shrink_parts_max(K);
  if (per_part <= num_sms()) {
    // small grid, released at once and run beside the GEMM's CTAs: at most
    // one slice set per SM
    const int cap = num_sms() / per_part;
    if (p > cap) p = cap;
  }
  // (a larger grid runs before the GEMM's CTAs arrive: more, shorter CTAs
  // keep more loads in flight)
  // every slice non-empty
  while (p > 1 && kslice_for(K, p) * (p - 1) >= K) --p;
  return p;
}

int launch_shrink(const void* X, int M, int K, int ldx, const void* A, int L, int r, const int32_t* idx,
                  const uint8_t* mask, float* S, int* status_dev, cudaStream_t stream) {
  if (M == 0) return EPILORA_OK;
  if (prefer_max_shared(reinterpret_cast<const void*>(shrink_kernel), shrink_carveout_done) != EPILORA_OK)
    return EPILORA_ERR_CUDA;
  QuantSide qs{-1, nullptr, nullptr, nullptr, nullptr, nullptr};
  dim3 grid(M, r / kRanksPerCta);
  shrink_kernel<<<grid, kShrinkThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(X), K, ldx,
                                                      static_cast<const __nv_bfloat16*>(A), L, r, idx, mask, S,
                                                      status_dev, qs, 1, K, 1, nullptr);
  return cudaGetLastError() == cudaSuccess ? EPILORA_OK : EPILORA_ERR_CUDA;
}

int launch_shrink_quant(const void* X, int M, int K, int ldx, const void* A, int L, int r, const int32_t* idx,
                        const uint8_t* mask, float* S, int s_parts, int fmt, void* Xq, float* x_scale,
                        uint8_t* x_block_scale, const float* x_global_scale, int32_t* perm, int* status_dev,
                        cudaStream_t stream, const float* a_scale) {
  if (M == 0) return EPILORA_OK;
  if (s_parts < 1 || s_parts > shrink_parts_max(K) || (s_parts > 1 && kslice_for(K, s_parts) * (s_parts - 1) >= K))
    return EPILORA_ERR_INVALID_ARG;
  if (prefer_max_shared(reinterpret_cast<const void*>(shrink_kernel), shrink_carveout_done) != EPILORA_OK)
    return EPILORA_ERR_CUDA;
  if (perm != nullptr && (M <= 32 || idx == nullptr))
    return EPILORA_ERR_INVALID_ARG;
  QuantSide qs{fmt, static_cast<uint8_t*>(Xq), x_scale, x_block_scale, x_global_scale, perm};
  const int kslice = s_parts == 1 ? K : kslice_for(K, s_parts);
  if (M > 32) {
    if (a_scale != nullptr) return EPILORA_ERR_UNSUPPORTED;   // stored FP8 adapters: decode batches only
    // wide batch: M quantizer CTAs, then token-block CTAs (block, K slice)
    const int nblk = r > 0 ? (M + kBlockTokens - 1) / kBlockTokens : 0;
    const long ctas = static_cast<long>(M) + static_cast<long>(nblk) * s_parts +
                      (r > 0 ? static_cast<long>(M) * (r / 16) : 0L);
    if (ctas > (1L << 30)) return EPILORA_ERR_INVALID_ARG;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(kShrinkThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int early = ctas <= num_sms() ? 1 : 0;
    // per-warp partial tiles of a token block (and the quantizers' scratch)
    cfg.dynamicSmemBytes = static_cast<size_t>(4) * kBlockTokens * (r > 4 ? r : 4) * sizeof(float);
    if (cfg.dynamicSmemBytes > 227 * 1024) return EPILORA_ERR_UNSUPPORTED;
    if (cfg.dynamicSmemBytes > 48 * 1024) {
      static int attr_done[64] = {0};
      int dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EPILORA_ERR_CUDA;
      if (attr_done[dev] < static_cast<int>(cfg.dynamicSmemBytes)) {
        if (cudaFuncSetAttribute(shrink_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(cfg.dynamicSmemBytes)) != cudaSuccess)
          return EPILORA_ERR_CUDA;
        attr_done[dev] = static_cast<int>(cfg.dynamicSmemBytes);
      }
    }
    const cudaError_t e = cudaLaunchKernelEx(&cfg, shrink_block_kernel, static_cast<const __nv_bfloat16*>(X), K, ldx,
                                             static_cast<const __nv_bfloat16*>(A), L, r, idx, mask, S, status_dev, qs,
                                             M, s_parts, kslice, early);
    return e == cudaSuccess ? EPILORA_OK : EPILORA_ERR_CUDA;
  }
  // launched as a programmatic dependent of whatever precedes it on the
  // stream: its CTAs become resident early and wait (griddepcontrol.wait)
  // for that kernel's completion before touching x or the workspace
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(M, s_parts + (r / kRanksPerCta) * s_parts);
  // The GEMM is released at CTA start when the grid fits beside it, and for
  // decode batches of any grid size: it then launches once the last CTA has
  // started and streams weights under the shrink's tail. Wide batches
  // release it at exit instead (their shrink is a small share of the layer,
  // and an early GEMM only competes with it for HBM).
  const int early_release =
      M <= 32 || static_cast<int>(cfg.gridDim.x * cfg.gridDim.y) <= num_sms() ? 1 : 0;
  cfg.blockDim = dim3(kShrinkThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, shrink_kernel, static_cast<const __nv_bfloat16*>(X), K, ldx,
                         static_cast<const __nv_bfloat16*>(A), L, r, idx, mask, S, status_dev, qs, s_parts,
                         kslice, early_release, a_scale) != cudaSuccess)
    return EPILORA_ERR_CUDA;
  return EPILORA_OK;
}

}  // namespace epi

