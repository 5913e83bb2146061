// Low-precision base GEMM with the multi-adapter LoRA epilogue ("K2"), on the
// 5th-generation tensor cores of sm_103a.
//
// EpiLoRA, "Fusing Many LoRA Adapters into Low-Precision GEMMs for Serving and
// RL":
//  * §Design › Multi-adapter kernels › K1 and K2 — the GEMM's epilogue applies
//    the weight and activation scales and then adds h_l B_l^T for each group
//    of rows that shares an adapter, reading only the tile's slice of B_l;
//  * › The decode path — the GEMM runs as the shrink's programmatic dependent:
//    it streams its weights while the shrink runs (extra thread blocks of the
//    shrink quantize the activations) and waits for h only before its
//    epilogue; it prefetches B;
//  * › When the overlap hides the adapter — exposure grows when the GEMM has
//    more CTAs than SMs, so decode grids are sized to stay resident.
//
// GB300 design (not the pages' Triton kernel):
//  * swap-AB: weight rows are the MMA's M = 128 side (TMEM lanes), tokens the
//    MMA's N side (BT = 16..256 TMEM columns), so a decode batch of 1..32
//    tokens still issues full-height MMAs while W streams;
//  * one elected thread issues tcgen05.mma (kind::f8f6f4 for E4M3, or
//    kind::mxf4nvf4 block-scaled with UE4M3 scales for NVFP4) on 128-byte
//    swizzled K-major tiles that TMA writes into a multi-stage ring; a stage
//    holds KA 128-byte K atoms of every row; the accumulator lives in TMEM;
//  * the producer fills the ring with weight tiles as soon as the CTA starts;
//    in the fused layer call it waits for the shrink grid (which quantizes the
//    activations) only before its first activation load, so a GEMM that
//    becomes resident while the previous layer call's GEMM drains streams
//    its weights at once;
//  * every weight tile starts its K loop at its own offset, so the CTAs
//    streaming W at the same time do not all read the same column slice;
//  * few output tiles (decode): the K dimension is split over a thread-block
//    cluster of KS CTAs; each CTA stores its fp32 partial rows straight into
//    the shared memory of the CTA that owns them (distributed shared memory),
//    and every owner sums the KS partials in rank order (deterministic, no
//    atomics), each CTA finishing 128/KS rows;
//  * decode tiles whose tokens use several adapters stream the B_l slices of
//    the tile (one 128-byte-swizzled TMA box per adapter) through the same
//    ring right behind the weights; the epilogue warps consume them group by
//    group into an fp32 output tile in shared memory, so the up-projection's
//    bytes keep HBM busy instead of being fetched one token at a time;
//  * the epilogue warps are idle during the main loop: they prefetch B into
//    L2 and load their first B row, execute griddepcontrol.wait (the shrink's
//    completion) and stage S in shared memory before the accumulator is ready.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM allocator
// and MMA issuer (all 32 lanes re-lay NVFP4 scale factors), warps 2..5 =
// epilogue (warp w reads TMEM lane quadrant w % 4).
#pragma once
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace epi {

constexpr int kGemmThreads = 192;
constexpr int kTileN = 128;          // weight rows per tile (MMA M)
constexpr int kAtomBytes = 128;      // bytes of K per 128-B swizzle atom
constexpr int kMaxRank = 128;
constexpr int kEpiBarrier = 1;       // named barrier of the 4 epilogue warps
constexpr int kMaxSplit = 8;         // largest cluster along K
constexpr int kDecodeBT = 32;        // token tiles up to this width use the decode epilogue
// fused call: weight stages issued before the wait for the shrink grid (a
// deep queue of weight reads would delay the shrink grid's own loads), and
// the weight bytes prefetched into L2 over the grid after it
constexpr int kPrewaitStages = 16;
constexpr long kL2AheadBytes = 32L << 20;

struct GemmParams {
  CUtensorMap tmW;    // uint8 [N, Kbytes], box 128 x 128 B, 128-B swizzle
  CUtensorMap tmX;    // uint8 [M, Kbytes], box BT x 128 B, 128-B swizzle
  CUtensorMap tmSW;   // NVFP4: uint8 [N, K/16], box 128 x 16*KA B
  CUtensorMap tmSX;   // NVFP4: uint8 [M, K/16], box BT x 16*KA B
  CUtensorMap tmB;    // streamed B: uint8 [L*N, 2r], box (128/KS) rows x min(2r, 128) B, swizzled
  const float* x_scale;
  const float* w_scale;
  const float* x_gs;
  const float* w_gs;
  const float* S;
  const __nv_bfloat16* B;
  const float* b_scale;  // stored FP8 B: E4M3 codes [L, N, r] bytes with one fp32 scale per row [L, N]; null: bf16
  const int32_t* idx;
  const uint8_t* mask;
  __nv_bfloat16* Y;
  int* status;
  // 1: the quantized activations, their scales, idx and mask are written by
  // the primary grid (the fused shrink grid): the producer streams weights
  // first and executes griddepcontrol.wait before the first activation load,
  // the epilogue warps before reading any token metadata.
  int fused;
  // 1: launched as a programmatic dependent outside the fused call: Xq (and
  // its block scales) may be loaded at once, but x_scale, idx, mask and S only
  // after griddepcontrol.wait (the previous kernel may write them)
  int pdl;
  const int32_t* perm;  // rows of Xq / x_scale are in this token order (perm[row] = token), or identity if null
  int stage_s;          // non-decode tiles: S of the tile's tokens is staged in the ring after the main loop
  // S is the sum of s_parts partial arrays [s_parts][M][r] (split K of the
  // shrink), added in part order
  int s_parts;
  int M, N, K, L, r, ldy;
  int num_kb;         // K stages in total (KA atoms each)
  int ks;             // cluster size along K (1 = no split)
  int stages;         // depth of the smem ring
  int rotate;         // 1: per-tile rotation of the K loop start
  int stream_b;       // 1: tiles with >= 2 adapter groups stream B through the ring
  int b_box_bytes;    // inner box bytes of tmB (32, 64 or 128 = its swizzle span)
  int b_atoms;        // tmB boxes per group (2 when 2r = 256)
  int b_group_bytes;  // ring bytes of one group's boxes (1024-byte aligned)
  int b_groups_per_slot;
  int b_early;        // 1: a decode tile with one adapter group loads its B slice at once into its own buffer
  int l2_ahead;       // fused call: weight stages past the ring to prefetch into L2 while waiting
  int t_tiles, n_tiles;  // persistent wide kernel: token tiles, weight tiles
  // S in memory: rows of s_row floats; a weight tile starting at column n0
  // reads the rank-r block of its slice (the number of slice ends <= n0)
  int s_row;
  int n_slices;
  int slice_end[4];
  int y_stage;        // wide tiles: ring byte offset of the per-warp output staging (-1: 2-byte stores)
  // wide tiles: the adapter term of each sorted row with an adapter, fp32
  // [M][N] (written by the expand pass); null: the epilogue computes it
  const float* yadd;
};

template <int FMT, int BT, int KA>
struct GemmCfg {
  static constexpr bool kFP4 = (FMT == EPILORA_FMT_NVFP4);
  static constexpr bool kDecode = BT <= kDecodeBT;
  static constexpr int kWAtom = kTileN * kAtomBytes;              // 16 KB
  static constexpr int kXAtom = BT * kAtomBytes;                  // multiple of 1 KB
  static constexpr int kWBytes = KA * kWAtom;
  static constexpr int kXBytes = KA * kXAtom;
  static constexpr int kKSteps = 4 * KA;                          // MMAs per stage (32 bytes of K each)
  static constexpr int kSfAtomsB = (BT + 127) / 128;              // scale atoms per K step for tokens
  static constexpr int kSfABytes = kFP4 ? kKSteps * 512 : 0;      // one 512-B atom per K step
  static constexpr int kSfBBytes = kFP4 ? kKSteps * 512 * kSfAtomsB : 0;
  static constexpr int kSfRow = 16 * KA;                          // scale bytes per row and stage
  static constexpr int kSfWRaw = kFP4 ? kTileN * kSfRow : 0;      // TMA box of W scales
  static constexpr int kSfXRaw = kFP4 ? BT * kSfRow : 0;          // TMA box of X scales
  static constexpr int kSfXRawPad = (kSfXRaw + 1023) / 1024 * 1024;
  static constexpr int kStageRaw = kWBytes + kXBytes + kSfABytes + kSfBBytes + kSfWRaw + kSfXRawPad;
  static constexpr int kStageBytes = (kStageRaw + 1023) / 1024 * 1024;
  static constexpr int kStageTx = kWBytes + kXBytes + kSfWRaw + kSfXRaw;   // bytes TMA delivers per stage
  // TMEM: accumulator columns [0, BT); NVFP4 scale columns after it, two slots.
  static constexpr int kSfColsA = 4 * kKSteps;
  static constexpr int kSfColsB = 4 * kKSteps * kSfAtomsB;
  static constexpr int kSfSlotCols = kSfColsA + kSfColsB;
  static constexpr int kTmemNeed = BT + (kFP4 ? 2 * kSfSlotCols : 0);
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
  static constexpr uint32_t kIdesc = kFP4 ? idesc_mxf4nvf4(kTileN, BT) : idesc_f8f6f4_e4m3(kTileN, BT);
  static_assert(BT % 16 == 0 && BT >= 16 && BT <= 256, "token tile");
  static_assert(KA == 1 || KA == 2 || KA == 4, "atoms per stage");
  static_assert(kTmemNeed <= 512, "TMEM");
};

constexpr int kGemmMiscBytes = 4096;

// Split-K reduction buffer: partial rows from every rank of the cluster,
// [rank][token][row within the owner's slice], fp32.
__host__ __device__ constexpr int gemm_red_rows(int ks) { return (kTileN + ks - 1) / ks; }
template <int BT>
__host__ __device__ constexpr int gemm_red_bytes(int ks) {
  return ks > 1 ? ks * BT * gemm_red_rows(ks) * 4 : 0;
}
// Decode-tile region: S rows [BT][r] fp32, output tile [BT][128/ks] fp32,
// token order by adapter group [BT], group starts [BT+1], group adapters [BT],
// group of each ordered token [BT].
__host__ __device__ constexpr int gemm_decode_bytes(int BT, int r, int ks) {
  return BT > kDecodeBT ? 0 : (BT * r * 4 + BT * gemm_red_rows(ks) * 4 + (4 * BT + 4) * 4 + 15) / 16 * 16;
}

// Rank-r block of S that output column n0's slice reads (floats from the
// start of an S row).
__device__ __forceinline__ int s_slice_offset(const GemmParams& p, int n0) {
  int off = 0;
  for (int q = 0; q + 1 < p.n_slices && q < 4; ++q)
    if (n0 >= p.slice_end[q]) off += p.r;
  return off;
}

// Two floats to packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Named barrier of the epilogue warps that also ORs a flag over them.
__device__ __forceinline__ bool epi_bar_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(kEpiBarrier)
      : "memory");
  return r != 0;
}

// S[t] . B[l, n] with the B row in registers: R4 float4 chunks of S (from
// shared or global memory), no per-chunk guards, two accumulators.
template <int R4, bool kSmem>
__device__ __forceinline__ float dot_srow_brow_n(const float4* srow, const uint32_t (&brow)[kMaxRank / 2]) {
  float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
  for (int c = 0; c < R4; ++c) {
    const float4 s4 = kSmem ? srow[c] : __ldcg(srow + c);
    float& d = (c & 1) ? d1 : d0;
    d = fmaf(s4.x, bf16_lo(brow[2 * c]), d);
    d = fmaf(s4.y, bf16_hi(brow[2 * c]), d);
    d = fmaf(s4.z, bf16_lo(brow[2 * c + 1]), d);
    d = fmaf(s4.w, bf16_hi(brow[2 * c + 1]), d);
  }
  return d0 + d1;
}
__device__ __forceinline__ float dot_srow_brow(const float4* srow, const uint32_t (&brow)[kMaxRank / 2], int r,
                                               bool srow_in_smem) {
  if (srow_in_smem) {
    switch (r) {
      case 16: return dot_srow_brow_n<4, true>(srow, brow);
      case 32: return dot_srow_brow_n<8, true>(srow, brow);
      case 64: return dot_srow_brow_n<16, true>(srow, brow);
      default: return dot_srow_brow_n<32, true>(srow, brow);
    }
  }
  switch (r) {
    case 16: return dot_srow_brow_n<4, false>(srow, brow);
    case 32: return dot_srow_brow_n<8, false>(srow, brow);
    case 64: return dot_srow_brow_n<16, false>(srow, brow);
    default: return dot_srow_brow_n<32, false>(srow, brow);
  }
}

// S[t] . B_g[row] for a B row of NC 16-byte chunks held in a swizzled ring
// box (chunk c in atom c >> cpa_log, at position (c & mask) ^ xr), S in
// shared memory; loads independent, two accumulators.
// The same for an E4M3 B row (16 codes per 16-byte chunk, S in chunks of 16).
__device__ __forceinline__ float2 e4m3x2_f32(uint32_t c) {
  uint32_t h2;
  const uint16_t c16 = static_cast<uint16_t>(c & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c16));
  __half2_raw hr;
  hr.x = static_cast<unsigned short>(h2 & 0xFFFFu);
  hr.y = static_cast<unsigned short>(h2 >> 16);
  return __half22float2(__half2(hr));
}
template <int NC>
__device__ __forceinline__ float dot_b_row_e4m3(const uint8_t* gb, int atom_stride, int cpa_log, int mask, int xr,
                                                const float4* srow) {
  float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(gb + (c >> cpa_log) * atom_stride + (((c & mask) ^ xr) << 4));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float& d = (c & 1) ? d1 : d0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 s4 = srow[4 * c + q];
      const float2 lo = e4m3x2_f32(w[q]), hi = e4m3x2_f32(w[q] >> 16);
      d = fmaf(s4.x, lo.x, d);
      d = fmaf(s4.y, lo.y, d);
      d = fmaf(s4.z, hi.x, d);
      d = fmaf(s4.w, hi.y, d);
    }
  }
  return d0 + d1;
}
// S[t] . B_g[row] for the row at gb (bf16 or E4M3 per b_scale), rank r
__device__ __forceinline__ float dot_b_row_any(const uint8_t* gb, int atom_stride, int cpa_log, int mask, int xr,
                                               const float4* srow, int r, bool fp8);

template <int NC>
__device__ __forceinline__ float dot_b_row(const uint8_t* gb, int atom_stride, int cpa_log, int mask, int xr,
                                           const float4* srow) {
  float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(gb + (c >> cpa_log) * atom_stride + (((c & mask) ^ xr) << 4));
    const float4 s0 = srow[2 * c], s1 = srow[2 * c + 1];
    float& d = (c & 1) ? d1 : d0;
    d = fmaf(s0.x, bf16_lo(v.x), d);
    d = fmaf(s0.y, bf16_hi(v.x), d);
    d = fmaf(s0.z, bf16_lo(v.y), d);
    d = fmaf(s0.w, bf16_hi(v.y), d);
    d = fmaf(s1.x, bf16_lo(v.z), d);
    d = fmaf(s1.y, bf16_hi(v.z), d);
    d = fmaf(s1.z, bf16_lo(v.w), d);
    d = fmaf(s1.w, bf16_hi(v.w), d);
  }
  return d0 + d1;
}

__device__ __forceinline__ float dot_b_row_any(const uint8_t* gb, int atom_stride, int cpa_log, int mask, int xr,
                                               const float4* srow, int r, bool fp8) {
  if (fp8) {
    switch (r) {
      case 16: return dot_b_row_e4m3<1>(gb, atom_stride, cpa_log, mask, xr, srow);
      case 32: return dot_b_row_e4m3<2>(gb, atom_stride, cpa_log, mask, xr, srow);
      case 64: return dot_b_row_e4m3<4>(gb, atom_stride, cpa_log, mask, xr, srow);
      default: return dot_b_row_e4m3<8>(gb, atom_stride, cpa_log, mask, xr, srow);
    }
  }
  switch (r) {   // rank 16 / 32 / 64 / 128: a loop without guards per chunk
    case 16: return dot_b_row<2>(gb, atom_stride, cpa_log, mask, xr, srow);
    case 32: return dot_b_row<4>(gb, atom_stride, cpa_log, mask, xr, srow);
    case 64: return dot_b_row<8>(gb, atom_stride, cpa_log, mask, xr, srow);
    default: return dot_b_row<16>(gb, atom_stride, cpa_log, mask, xr, srow);
  }
}

template <int FMT, int BT, int KA>
__global__ void __launch_bounds__(kGemmThreads, 2) gemm_lora_kernel(const __grid_constant__ GemmParams p) {
  using C = GemmCfg<FMT, BT, KA>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stages = p.stages;
  const int ks = p.ks;
  uint8_t* red_buf = smem + static_cast<size_t>(stages) * C::kStageBytes;
  uint8_t* misc = red_buf + gemm_red_bytes<BT>(ks);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(misc);
  uint64_t* empty_bar = full_bar + stages;
  uint64_t* acc_bar = empty_bar + stages;
  uint64_t* meta_bar = acc_bar + 1;           // token metadata and adapter groups are in shared memory
  uint64_t* b_bar = meta_bar + 1;             // the early B slice has landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(b_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* ngroups_s = reinterpret_cast<int*>(tmem_slot + 2);
  float* meta_sx = reinterpret_cast<float*>(tmem_slot + 4);
  int* meta_idx = reinterpret_cast<int*>(meta_sx + BT);       // adapter slot, -1 = none
  int* meta_tok = meta_idx + BT;                               // token of each tile column (row of Y and S)
  float* s_big = reinterpret_cast<float*>(smem);               // non-decode: S rows of the tile, after the main loop
  const int s_ld = p.r + 4;                                    // its row stride in floats (bank-conflict padding)
  // decode region (BT <= kDecodeBT)
  const int RR = gemm_red_rows(ks);           // rows owned per rank (last rank: fewer)
  float* s_stage = reinterpret_cast<float*>(misc + kGemmMiscBytes);   // [token][r]
  // one-group decode tiles: the B slice of the group (1024-byte aligned for the swizzled box)
  uint8_t* b_early_buf = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(misc + kGemmMiscBytes + gemm_decode_bytes(BT, p.r, ks)) + 1023) & ~uintptr_t(1023));
  float* y_tile = s_stage + BT * p.r;                                 // [token][RR]
  int* g_order = reinterpret_cast<int*>(y_tile + BT * RR);            // tokens sorted by group
  int* g_start = g_order + BT;                                        // [group + 1]
  int* g_adapter = g_start + BT + 1;                                  // adapter of each group
  int* g_of = g_adapter + BT;                                         // group of g_order[k]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = ks > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int t0 = blockIdx.y * BT;
  const int n0 = blockIdx.z * kTileN;
  const int kb_begin = (p.num_kb * rank) / ks;
  const int kb_end = (p.num_kb * (rank + 1)) / ks;
  const int nkb = kb_end - kb_begin;
  const int tv = min(BT, p.M - t0);           // valid token columns of this tile
  const float* S_t = p.S != nullptr ? p.S + s_slice_offset(p, n0) : nullptr;   // this tile's slice of S rows
  const int row_lo = ks > 1 ? RR * rank : 0;
  const int row_hi = ks > 1 ? min(kTileN, RR * (rank + 1)) : kTileN;
  const int R = row_hi - row_lo;
  const int et = threadIdx.x - 64;            // epilogue thread 0..127
  // K-loop rotation of this weight tile (fixed per weight tile and the same
  // for every token tile: results stay deterministic and independent of the
  // tokens' positions)
  const int rot = p.rotate ? static_cast<int>((blockIdx.z * 5u) % static_cast<unsigned>(nkb)) : 0;

  auto stage_kb = [&](int i) {
    int kb = i + rot;
    if (kb >= nkb) kb -= nkb;
    return kb + kb_begin;
  };
  // A single token tile reads every weight byte once: the weights then
  // stream with the first eviction priority, so that the activations, S and
  // the adapters' B slices stay in L2 beside them (several token tiles
  // re-read them and keep the default).
  const bool w_once = gridDim.y == 1;
  const uint64_t wpol = l2_policy_evict_first();
  // TMA loads of ring slot s for loop iteration i: weights (+ their scales)
  auto issue_w = [&](int i, int s) {
    uint8_t* st = smem + static_cast<size_t>(s) * C::kStageBytes;
    const int kb = stage_kb(i);
    mbar_arrive_expect_tx(&full_bar[s], C::kStageTx);
    uint8_t* sfw = st + C::kWBytes + C::kXBytes + C::kSfABytes + C::kSfBBytes;
    if (w_once) {
#pragma unroll
      for (int a = 0; a < KA; ++a)
        tma_load_2d_hint(st + a * C::kWAtom, &p.tmW, &full_bar[s], (kb * KA + a) * kAtomBytes, n0, wpol);
      if (C::kFP4) tma_load_2d_hint(sfw, &p.tmSW, &full_bar[s], kb * C::kSfRow, n0, wpol);
    } else {
#pragma unroll
      for (int a = 0; a < KA; ++a)
        tma_load_2d(st + a * C::kWAtom, &p.tmW, &full_bar[s], (kb * KA + a) * kAtomBytes, n0);
      if (C::kFP4) tma_load_2d(sfw, &p.tmSW, &full_bar[s], kb * C::kSfRow, n0);
    }
  };
  // ... and activations (+ their scales)
  auto issue_x = [&](int i, int s) {
    uint8_t* st = smem + static_cast<size_t>(s) * C::kStageBytes;
    const int kb = stage_kb(i);
#pragma unroll
    for (int a = 0; a < KA; ++a)
      tma_load_2d(st + C::kWBytes + a * C::kXAtom, &p.tmX, &full_bar[s], (kb * KA + a) * kAtomBytes, t0);
    if (C::kFP4)
      tma_load_2d(st + C::kWBytes + C::kXBytes + C::kSfABytes + C::kSfBBytes + C::kSfWRaw, &p.tmSX, &full_bar[s],
                  kb * C::kSfRow, t0);
  };

  // ---------------------------------------------------------------- setup
  const int prologue = nkb < stages ? nkb : stages;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(acc_bar, 1);
    mbar_init(meta_bar, 1);
    mbar_init(b_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    // the ring starts empty: stream weights into it before anything else
    auto l2_ahead = [&]() {
      // the next weight stages go to L2 now and come back from there later
      const int ahead_end = min(nkb, prologue + p.l2_ahead);
      for (int i = prologue; i < ahead_end; ++i) {
        const int kb = stage_kb(i);
#pragma unroll
        for (int a = 0; a < KA; ++a) tma_prefetch_l2_2d(&p.tmW, (kb * KA + a) * kAtomBytes, n0);
        if (C::kFP4) tma_prefetch_l2_2d(&p.tmSW, kb * C::kSfRow, n0);
      }
    };
    // fused call: only the first kPrewaitStages weight stages before the wait
    const int prewait = p.fused ? min(prologue, kPrewaitStages) : prologue;
    for (int i = 0; i < prewait; ++i) issue_w(i, i);
    if (p.fused) {
      // the shrink grid quantizes the activations: its completion (and that
      // of everything before it) makes them visible
      pdl_wait_primary();
      fence_proxy_async_global();
      // activations of the stages already requested first (the MMA waits for
      // them), then the rest of the ring, then the L2 prefetch
      for (int i = 0; i < prewait; ++i) issue_x(i, i);
      for (int i = prewait; i < prologue; ++i) {
        issue_w(i, i);
        issue_x(i, i);
      }
      l2_ahead();
    } else {
      for (int i = 0; i < prologue; ++i) issue_x(i, i);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  // Token metadata of the tile (scales, adapter slots) and, for decode tiles,
  // the adapter groups: by the four epilogue warps. In the fused call it is
  // read in the main-loop phase, once the shrink grid has completed (set-up
  // then needs no global loads); otherwise during set-up.
  auto build_meta = [&]() {
    for (int i = et; i < BT; i += 128) {
      const int row = t0 + i;             // row of the quantized activations
      float sx = 0.0f;
      int l = -1;
      int tok = row;
      if (row < p.M) {
        if (p.perm != nullptr) tok = p.perm[row];
        if (!C::kFP4) sx = p.x_scale[row];
        if (p.S != nullptr) {
          const int li = p.idx[tok];
          const bool on = li >= 0 && li < p.L && (p.mask == nullptr || p.mask[tok] != 0);
          if (li >= p.L) record_status(p.status, EPILORA_ERR_INVALID_ARG);
          l = on ? li : -1;
        }
      }
      meta_sx[i] = sx;
      meta_idx[i] = l;
      meta_tok[i] = tok;
    }
    asm volatile("bar.sync %0, 128;" ::"r"(kEpiBarrier) : "memory");
    if (C::kDecode) {
      if (warp == 2) {
        // adapter groups of the tile (lane t = token t, BT <= 32), numbered in
        // order of first appearance, and the tokens sorted by group (stable)
        const unsigned full = 0xffffffffu;
        const int l = lane < tv ? meta_idx[lane] : -1;
        const unsigned act = __ballot_sync(full, l >= 0);
        const unsigned same = __match_any_sync(full, l);       // lanes holding the same adapter
        const int leader = __ffs(same) - 1;                    // its first token
        const bool is_leader = l >= 0 && leader == lane;
        const unsigned leaders = __ballot_sync(full, is_leader);
        const int gid = __popc(leaders & ((1u << leader) - 1u));
        const int cnt = is_leader ? __popc(same) : 0;
        int incl = cnt;                                        // inclusive scan of group sizes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(full, incl, o);
          if (lane >= o) incl += n;
        }
        const int start = __shfl_sync(full, incl - cnt, leader);
        if (l >= 0) {
          const int pos = start + __popc(same & ((1u << lane) - 1u));
          g_order[pos] = lane;
          g_of[pos] = gid;
        }
        if (is_leader) {
          g_adapter[gid] = l;
          g_start[gid] = start;
        }
        if (lane == 0) {
          g_start[__popc(leaders)] = __popc(act);
          *ngroups_s = __popc(leaders);
        }
      }
    } else if (et == 0) {
      *ngroups_s = 0;
    }
    asm volatile("bar.sync %0, 128;" ::"r"(kEpiBarrier) : "memory");   // groups visible to all four warps
  };
  if (warp >= 2 && !p.fused && !p.pdl) build_meta();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // every CTA of the cluster has started once this phase completes (its wait
  // comes before the first store into a peer's shared memory)
  if (ks > 1) cluster_arrive_relaxed();
  // Decode tiles stream their B slices through the ring, behind the weights.
  // The group count is known to the epilogue warps once they have built the
  // metadata, and to the producer once meta_bar has completed.
  int ngroups = 0;
  bool sb = false;
  const int gps = p.b_groups_per_slot;
  int n_bslots = 0;       // ring loads carrying B slices
  int n_loads = nkb;
  bool b_early_on = false;  // the tile's only group comes through b_early_buf instead of the ring
  auto set_groups = [&]() {
    ngroups = *ngroups_s;
    sb = C::kDecode && p.stream_b && ngroups >= 1 && p.S != nullptr;
    b_early_on = sb && p.b_early && ngroups == 1;
    n_bslots = sb && !b_early_on ? (ngroups + gps - 1) / gps : 0;
    n_loads = nkb + n_bslots;
  };

  // epilogue state carried from the main-loop phase into the epilogue phase
  int cached_key = -1;
  uint32_t brow[kMaxRank / 2];
  float sw_pre = 0.0f;      // FP8: scale of this thread's weight row
  float alpha_pre = 1.0f;   // NVFP4: 1 / (g_x * g_w)

  auto load_brow = [&](int l, int mm) {
    const uint4* bsrc =
        reinterpret_cast<const uint4*>(p.B + (static_cast<size_t>(l) * p.N + n0 + mm) * p.r);
#pragma unroll
    for (int c = 0; c < kMaxRank / 8; ++c) {
      if (c < p.r / 8) {
        const uint4 v = ldg_nc_v4_now(bsrc + c);
        brow[4 * c + 0] = v.x;
        brow[4 * c + 1] = v.y;
        brow[4 * c + 2] = v.z;
        brow[4 * c + 3] = v.w;
      }
    }
    cached_key = l * kTileN + mm;
  };

  // ---------------------------------------------------------------- roles
  if (warp == 0) {
    // ===== TMA producer =====
    uint32_t issued_mask = (prologue >= 32) ? 0xffffffffu : ((1u << prologue) - 1u);
    uint32_t parity_mask = 0;
    bool stop = false;
    // one ring load: W/X stage (i < nkb) or the B slice of group i - nkb
    auto produce = [&](int i) {
      const int s = i % stages;
      const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
      if (*abort_flag) {
        stop = true;
        return;
      }
      if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, kWaitLimitNs)) {
        *abort_flag = 1;
        record_status(p.status, EPILORA_ERR_TIMEOUT);
        stop = true;
        return;
      }
      if (i < nkb) {
        issue_w(i, s);
        issue_x(i, s);
      } else {
        // groups [g0, g1) of this slot: rows [n0 + row_lo, + RR) of each
        // group's adapter, one box per 128 B of the row
        uint8_t* st = smem + static_cast<size_t>(s) * C::kStageBytes;
        const int g0 = (i - nkb) * gps;
        const int g1 = min(ngroups, g0 + gps);
        mbar_arrive_expect_tx(&full_bar[s], static_cast<uint32_t>((g1 - g0) * RR * p.b_box_bytes * p.b_atoms));
        for (int g = g0; g < g1; ++g) {
          const int y = g_adapter[g] * p.N + n0 + row_lo;
          for (int a = 0; a < p.b_atoms; ++a)
            tma_load_2d(st + (g - g0) * p.b_group_bytes + a * RR * p.b_box_bytes, &p.tmB, &full_bar[s],
                        a * p.b_box_bytes, y);
        }
      }
      issued_mask |= 1u << s;
      parity_mask = (parity_mask & ~(1u << s)) | (ph << s);
    };
    if (lane == 0)
      for (int i = prologue; i < nkb && !stop; ++i) produce(i);
    __syncwarp();
    // The B slices are freed by the epilogue warps, which first pass the
    // cluster barrier: arrive on its second phase before producing them.
    if (ks > 1) {
      cluster_wait();
      cluster_arrive();
    }
    if (lane == 0) {
      if (!stop && !mbar_wait_bounded(meta_bar, 0, kWaitLimitNs)) {
        *abort_flag = 1;
        record_status(p.status, EPILORA_ERR_TIMEOUT);
        stop = true;
      }
      if (!stop) set_groups();
      for (int i = (prologue > nkb ? prologue : nkb); i < n_loads && !stop; ++i) produce(i);
      if (*abort_flag) {
        // do not leave with copies in flight: wait for every issued fill
        for (int s = 0; s < stages; ++s)
          if (issued_mask & (1u << s)) (void)mbar_wait_bounded(&full_bar[s], (parity_mask >> s) & 1u, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===== MMA issuer =====
    for (int i = 0; i < nkb; ++i) {
      const int s = i % stages;
      const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
      // every lane observes the barrier itself (the NVFP4 re-layout reads
      // the TMA-written scale boxes with ordinary loads)
      const int ab = __shfl_sync(0xffffffffu, *abort_flag, 0);
      const bool ok = !ab && __all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[s], ph, kWaitLimitNs));
      if (!ok) {
        if (lane == 0) {
          *abort_flag = 1;
          record_status(p.status, EPILORA_ERR_TIMEOUT);
        }
        break;
      }
      uint8_t* st = smem + static_cast<size_t>(s) * C::kStageBytes;
      const uint32_t w_addr = smem_u32(st);
      const uint32_t x_addr = smem_u32(st + C::kWBytes);
      uint8_t* sfa = st + C::kWBytes + C::kXBytes;
      uint8_t* sfb = sfa + C::kSfABytes;
      if (C::kFP4) {
        // Re-lay the canonical [rows][16*KA scale bytes] TMA boxes into one
        // 512-B atom per K=64 step: line r0 (16 B) = the 4 scale bytes of
        // rows r0, r0+32, r0+64, r0+96.
        const uint8_t* raw_w = sfb + C::kSfBBytes;
        const uint8_t* raw_x = raw_w + C::kSfWRaw;
#pragma unroll
        for (int a = 0; a < KA; ++a) {
          uint4 v[4];
#pragma unroll
          for (int r1 = 0; r1 < 4; ++r1)
            v[r1] = *reinterpret_cast<const uint4*>(raw_w + (lane + 32 * r1) * C::kSfRow + 16 * a);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            uint4 o;
            o.x = (&v[0].x)[kk];
            o.y = (&v[1].x)[kk];
            o.z = (&v[2].x)[kk];
            o.w = (&v[3].x)[kk];
            *reinterpret_cast<uint4*>(sfa + (a * 4 + kk) * 512 + lane * 16) = o;
          }
#pragma unroll
          for (int b = 0; b < C::kSfAtomsB; ++b) {
#pragma unroll
            for (int r1 = 0; r1 < 4; ++r1) {
              const int row = 128 * b + 32 * r1 + lane;
              v[r1] = row < BT ? *reinterpret_cast<const uint4*>(raw_x + row * C::kSfRow + 16 * a)
                               : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              uint4 o;
              o.x = (&v[0].x)[kk];
              o.y = (&v[1].x)[kk];
              o.z = (&v[2].x)[kk];
              o.w = (&v[3].x)[kk];
              *reinterpret_cast<uint4*>(sfb + ((a * 4 + kk) * C::kSfAtomsB + b) * 512 + lane * 16) = o;
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t slot_col = static_cast<uint32_t>(BT + (i & 1) * C::kSfSlotCols);
#pragma unroll
        for (int a = 0; a < KA; ++a) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int j = a * 4 + kk;                       // K step within the stage
            const uint64_t adesc = make_smem_desc(w_addr + a * C::kWAtom + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bdesc = make_smem_desc(x_addr + a * C::kXAtom + kk * 32, 16, 1024, kSwizzle128B);
            const uint32_t accum = (i > 0 || j > 0) ? 1u : 0u;
            if (C::kFP4) {
              const uint32_t sfa_addr = smem_u32(sfa) + j * 512;
              const uint32_t sfb_addr = smem_u32(sfb) + j * C::kSfAtomsB * 512;
              const uint32_t sfa_col = slot_col + j * 4;
              const uint32_t sfb_col = slot_col + C::kSfColsA + j * 4 * C::kSfAtomsB;
              tc_cp_32x128b_warpx4(tmem_base + sfa_col, make_smem_desc(sfa_addr, 16, 128, kSwizzleNone));
#pragma unroll
              for (int b = 0; b < C::kSfAtomsB; ++b)
                tc_cp_32x128b_warpx4(tmem_base + sfb_col + 4 * b,
                                     make_smem_desc(sfb_addr + b * 512, 16, 128, kSwizzleNone));
              mma_mxf4nvf4(tmem_base, adesc, bdesc, C::kIdesc, tmem_base + sfa_col, tmem_base + sfb_col, accum);
            } else {
              mma_f8f6f4(tmem_base, adesc, bdesc, C::kIdesc, accum);
            }
          }
        }
        tc_commit(&empty_bar[s]);   // frees the stage once these MMAs have read it
      }
      __syncwarp();
    }
    if (lane == 0) tc_commit(acc_bar);   // accumulator complete (or drained after an abort)
    __syncwarp();
    if (ks > 1) {
      cluster_wait();      // first phase (armed after setup)
      cluster_arrive();    // second phase: nothing of this warp is still to land in a peer
    }
  } else {
    // ===== epilogue warps, main-loop phase =====
    if (p.fused || p.pdl) {
      // the primary grid (in the fused call the shrink grid: quantized
      // activations, scales, S) has completed; token metadata is read after
      pdl_wait_primary();
      build_meta();
    }
    set_groups();
    if (et == 0) mbar_arrive(meta_bar);   // the producer may now stream B slices
    if (b_early_on && et == 0) {
      // a one-group tile's B slice goes to its own buffer now (the ring is
      // busy with weight stages), so the epilogue finds it there
      mbar_arrive_expect_tx(b_bar, static_cast<uint32_t>(RR * p.b_box_bytes * p.b_atoms));
      const int y = g_adapter[0] * p.N + n0 + row_lo;
      for (int a = 0; a < p.b_atoms; ++a)
        tma_load_2d(b_early_buf + a * RR * p.b_box_bytes, &p.tmB, b_bar, a * p.b_box_bytes, y);
    }
    if (p.S != nullptr && !sb) {
      // L2 prefetch of the tile's B slices, first B row into registers
      const int rows = min(row_hi, p.N - n0) - row_lo;
      int first_l = -1;
      int prev = -1;
      for (int i = 0; i < BT; ++i) {
        const int l = meta_idx[i];
        if (l >= 0 && first_l < 0) first_l = l;
        if (et == 0 && rows > 0 && l >= 0 && l != prev) {
          prefetch_l2_bulk(p.B + (static_cast<size_t>(l) * p.N + n0 + row_lo) * p.r,
                           static_cast<uint32_t>(rows * p.r * 2));
          prev = l;
        }
      }
      const int mm = ks == 1 ? ((warp & 3) * 32 + lane) : row_lo + (R > 0 ? et % R : 0);
      if (first_l >= 0 && n0 + mm < p.N && mm < row_hi) load_brow(first_l, mm);
    }
    // The shrink's completion (normally well before the main loop ends): from
    // here on S is visible. Also orders this grid after the whole primary grid.
    pdl_wait_primary();
    if (C::kDecode && p.S != nullptr) {
      // S rows of this tile's tokens into shared memory (partials of a split
      // shrink added in part order)
      const size_t part = static_cast<size_t>(p.M) * p.s_row / 4;
      const int n4 = p.r / 4;
      float4* dst = reinterpret_cast<float4*>(s_stage);
      for (int i = et; i < tv * n4; i += 128) {
        const int tl = i / n4;
        const float4* src =
            reinterpret_cast<const float4*>(S_t + static_cast<size_t>(t0 + tl) * p.s_row) + (i - tl * n4);
        float4 v = __ldcg(src);
        for (int q = 1; q < p.s_parts; ++q) {
          const float4 w = __ldcg(src + q * part);
          v.x += w.x;
          v.y += w.y;
          v.z += w.z;
          v.w += w.w;
        }
        dst[i] = v;
      }
    }
    // this thread's weight-row scale and the NVFP4 dequantization factor,
    // loaded while the main loop runs
    if (!C::kFP4) {
      const int mrow = ks == 1 ? (warp & 3) * 32 + lane : row_lo + (R > 0 ? et % R : 0);
      sw_pre = n0 + mrow < p.N ? ldg_nc_f32_now(p.w_scale + n0 + mrow) : 0.0f;
    } else {
      alpha_pre = 1.0f / (*p.x_gs * *p.w_gs);
    }
    asm volatile("bar.sync %0, 128;" ::"r"(kEpiBarrier) : "memory");
    const bool ok = mbar_wait_bounded(acc_bar, 0, kWaitLimitNs);
    if (!ok) {
      *abort_flag = 1;
      record_status(p.status, EPILORA_ERR_TIMEOUT);
    }
    tc_fence_after();
    if (ks > 1) {
      // every CTA of the cluster has started (the phase armed after setup)
      cluster_wait();
      if (ok) {
        // scatter this CTA's fp32 partial rows into their owners' buffers:
        // owner d, slot [rank][token][row - row_lo(d)]
        const int q = warp & 3;
        const int m = q * 32 + lane;
        const int d = m / RR;
        const uint32_t dst = map_to_cta(smem_u32(red_buf), static_cast<uint32_t>(d)) +
                             static_cast<uint32_t>(((rank * BT) * RR + (m - d * RR)) * 4);
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
        for (int c = 0; c < BT / 16; ++c) {
          if (c * 16 >= tv) break;
          uint32_t v[16];
          tmem_ld_32x32b_x16(lane_base + c * 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c * 16 + j < tv) st_dsmem_f32(dst + static_cast<uint32_t>((c * 16 + j) * RR * 4), __uint_as_float(v[j]));
        }
      }
    }
    const bool all_ok = !epi_bar_any(!ok);    // uniform over the four warps (a barrier follows)
    if (!C::kDecode && p.stage_s && all_ok) {
      // every stage has been consumed: the ring now holds the S rows of this
      // tile's tokens (one read of each from L2 instead of one per element)
      const int n4 = p.r / 4;
      const size_t part = static_cast<size_t>(p.M) * p.s_row / 4;   // partial sums of a split shrink, in part order
      for (int k = et; k < tv * n4; k += 128) {
        const int tl = k / n4;
        const float4* src =
            reinterpret_cast<const float4*>(S_t + static_cast<size_t>(meta_tok[tl]) * p.s_row) + (k - tl * n4);
        float4 v = __ldcg(src);
        for (int q = 1; q < p.s_parts; ++q) {
          const float4 w = __ldcg(src + q * part);
          v.x += w.x;
          v.y += w.y;
          v.z += w.z;
          v.w += w.w;
        }
        reinterpret_cast<float4*>(s_big + tl * s_ld)[k - tl * n4] = v;
      }
      asm volatile("bar.sync %0, 128;" ::"r"(kEpiBarrier) : "memory");
    }
  }

  // The main loop is done: the next kernel on the stream (the next layer
  // call's shrink grid) may become resident now; it waits for this grid's
  // completion before it reads anything this grid writes.
  pdl_allow_dependents();

  // ---------------------------------------------------------------- epilogue
  const float alpha = alpha_pre;
  // base value of element (tile row mm, token column tl) from its fp32 sum
  auto base_value = [&](int mm, int tl, float acc, float sw) {
    return C::kFP4 ? acc * alpha : (acc * meta_sx[tl]) * sw;
  };
  // y = base + [token has an adapter] * S[t] . B[l, n]  (B row cached in
  // registers while consecutive elements share (row, adapter))
  auto finish = [&](int mm, int tl, float acc, float sw) {
    const int n = n0 + mm;
    const int t = t0 + tl;
    if (n >= p.N || t >= p.M) return;
    float y = base_value(mm, tl, acc, sw);
    const int l = meta_idx[tl];
    if (l >= 0 && p.yadd != nullptr) {
      y += __ldcg(p.yadd + static_cast<size_t>(t) * p.N + n);     // the expand pass's term
    } else if (l >= 0) {
      if (l * kTileN + mm != cached_key) load_brow(l, mm);
      const bool s_smem = C::kDecode || p.stage_s;
      const float4* srow =
          C::kDecode ? reinterpret_cast<const float4*>(s_stage + tl * p.r)
          : p.stage_s ? reinterpret_cast<const float4*>(s_big + tl * s_ld)
                      : reinterpret_cast<const float4*>(S_t + static_cast<size_t>(meta_tok[tl]) * p.s_row);
      y += dot_srow_brow(srow, brow, p.r, s_smem);
    }
    p.Y[static_cast<size_t>(meta_tok[tl]) * p.ldy + n] = __float2bfloat16_rn(y);
  };

  // wide tiles: 16 token columns of this warp's 32 output rows go through a
  // staging block in the (consumed) ring, [16 tokens][40] bf16 (rows padded
  // against bank conflicts), and leave as 16-byte row segments, 8 token rows
  // per store instruction instead of one
  constexpr int kYsLd = 40;
  auto y_stage_block = [&]() {
    return reinterpret_cast<__nv_bfloat16*>(smem + p.y_stage) + (warp & 3) * 16 * kYsLd;
  };
  auto flush16 = [&](int c) {
    const int q = warp & 3;
    const __nv_bfloat16* ys = y_stage_block();
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = h * 8 + (lane >> 2);
      const int tl = c * 16 + row;
      const int n = n0 + q * 32 + (lane & 3) * 8;
      if (tl < tv && n < p.N) {
        const __nv_bfloat16* src = ys + row * kYsLd + (lane & 3) * 8;
        __nv_bfloat16* dst = p.Y + static_cast<size_t>(meta_tok[tl]) * p.ldy + n;
        if (n + 8 <= p.N) {
          *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
        } else {
          for (int e = 0; e < p.N - n; ++e) dst[e] = src[e];
        }
      }
    }
    __syncwarp();     // the block is free for the next chunk
  };
  auto emit16 = [&](int c, const float* yv) {
    __nv_bfloat16* ys = y_stage_block();
#pragma unroll
    for (int j = 0; j < 16; ++j) ys[j * kYsLd + lane] = __float2bfloat16_rn(yv[j]);
    flush16(c);
  };

  if (ks > 1 && warp >= 2) {
    // all partial rows have landed in their owners' shared memory (the
    // producer and MMA warps arrived on this phase already)
    cluster_arrive();
    cluster_wait();
  }
  // the 4 epilogue warps agree on whether to produce output (the sections
  // below contain their named barrier, which all four must reach)
  if (warp >= 2 && !epi_bar_any(*abort_flag != 0)) {
    const float* red = reinterpret_cast<const float*>(red_buf);
    if (sb) {
      // ---- streamed-B epilogue (decode tile with >= 2 adapter groups) ----
      // 1) base values into the shared output tile y_tile[token][row]
      if (ks == 1) {
        const int q = warp & 3;
        const int m = q * 32 + lane;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        const float sw = sw_pre;
#pragma unroll 1
        for (int c = 0; c < BT / 16; ++c) {
          if (c * 16 >= tv) break;
          uint32_t v[16];
          tmem_ld_32x32b_x16(lane_base + c * 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c * 16 + j < tv) y_tile[(c * 16 + j) * RR + m] = base_value(m, c * 16 + j, __uint_as_float(v[j]), sw);
        }
      } else {
        for (int e = et; e < R * tv; e += 128) {
          const int i = e % R, tl = e / R;
          float acc = 0.0f;
#pragma unroll
          for (int s = 0; s < kMaxSplit; ++s)
            if (s < ks) acc += red[(s * BT + tl) * RR + i];     // rank order: deterministic
          const int mm = row_lo + i;
          y_tile[tl * RR + i] = base_value(mm, tl, acc, sw_pre);   // i == et % R: this thread's row
        }
      }
      asm volatile("bar.sync %0, 128;" ::"r"(kEpiBarrier) : "memory");
      // 2) ring slots of B slices (several adapter groups each): thread ->
      //    row i, the slot's tokens strided by 128 / R (R divides 128)
      const int i = et % R;
      const int tstep = 128 / R;
      const int tsl = et / R;
      const int sw_span = p.b_box_bytes;                   // 32, 64 or 128: swizzle span
      const int sw_mask = sw_span / 16 - 1;
      const int sw_shift = sw_span == 128 ? 0 : sw_span == 64 ? 1 : 2;   // row >> shift = (row * span) / 128
      const int cpa_log = 3 - sw_shift;                    // log2 of the 16-byte chunks per atom
      const bool bq = p.b_scale != nullptr;                // stored FP8 B rows (r bytes each)
      const int atom_stride = RR * sw_span;                // bytes between a group's atoms
      if (b_early_on) {
        // the only group's slice is in its own buffer
        const bool late = !mbar_wait_bounded(b_bar, 0, kWaitLimitNs);
        if (!epi_bar_any(late)) {
          const int xr = (i >> sw_shift) & sw_mask;
          for (int k = g_start[0] + tsl; k < g_start[1]; k += tstep) {
            const int tl = g_order[k];
            const uint8_t* gb = b_early_buf + i * sw_span;
            const float4* srow = reinterpret_cast<const float4*>(s_stage + tl * p.r);
            float d = dot_b_row_any(gb, atom_stride, cpa_log, sw_mask, xr, srow, p.r, bq);
            if (bq) d *= __ldg(p.b_scale + static_cast<size_t>(g_adapter[0]) * p.N + n0 + row_lo + i);
            y_tile[tl * RR + i] += d;
          }
          asm volatile("bar.sync %0, 128;" ::"r"(kEpiBarrier) : "memory");
        } else {
          *abort_flag = 1;
          record_status(p.status, EPILORA_ERR_TIMEOUT);
        }
      }
      for (int j = 0; j < n_bslots; ++j) {
        const int li = nkb + j;
        const int s = li % stages;
        const uint32_t ph = static_cast<uint32_t>(li / stages) & 1u;
        // every thread waits itself (TMA data visibility); the outcome is
        // made uniform over the 4 epilogue warps before anyone leaves
        const bool late = !mbar_wait_bounded(&full_bar[s], ph, kWaitLimitNs);
        if (epi_bar_any(late)) {
          *abort_flag = 1;
          record_status(p.status, EPILORA_ERR_TIMEOUT);
          break;
        }
        const uint8_t* st = smem + static_cast<size_t>(s) * C::kStageBytes;
        // y[t][i] += S[t] . B_g[row i], B's row read 16 bytes at a time from
        // the swizzled box (chunk c of row i lives at chunk c ^ f(i))
        const int xr = (i >> sw_shift) & sw_mask;
        const int g0 = j * gps;
        const int g1 = min(ngroups, g0 + gps);
        for (int k = g_start[g0] + tsl; k < g_start[g1]; k += tstep) {
          const int tl = g_order[k];
          const uint8_t* gb = st + (g_of[k] - g0) * p.b_group_bytes + i * sw_span;
          const float4* srow = reinterpret_cast<const float4*>(s_stage + tl * p.r);
          float d = dot_b_row_any(gb, atom_stride, cpa_log, sw_mask, xr, srow, p.r, bq);
          if (bq) d *= __ldg(p.b_scale + static_cast<size_t>(g_adapter[g_of[k]]) * p.N + n0 + row_lo + i);
          y_tile[tl * RR + i] += d;
        }
        asm volatile("bar.sync %0, 128;" ::"r"(kEpiBarrier) : "memory");
        if (et == 0) mbar_arrive(&empty_bar[s]);          // slot free for the producer
      }
      // 3) the output tile
      for (int e = et; e < R * tv; e += 128) {
        const int ii = e % R, tl = e / R;
        const int n = n0 + row_lo + ii;
        if (n < p.N) p.Y[static_cast<size_t>(meta_tok[tl]) * p.ldy + n] = __float2bfloat16_rn(y_tile[tl * RR + ii]);
      }
    } else if (ks == 1 && !C::kDecode && p.S != nullptr) {
      // wide tiles: the token columns in adapter-sorted chunks of 16. For
      // ranks <= 32 every chunk takes its adapter term from TF32 tensor-core
      // MMAs, one pass per adapter present in the chunk:
      //   D[row][token] = sum_k B_l[row][k] * S[token][k]
      // with the adapter rows (bf16, exact in TF32) as the A operand and S
      // split into two TF32 halves (hi + lo, together exact to about 2^-22)
      // as the B operand, fp32 accumulate. The m16n8 accumulator layout is
      // the one tcgen05.ld.16x256b returns the base sums in, so base and
      // adapter term meet in registers. Higher ranks go element by element
      // on CUDA cores: this thread's weight row m, its B row reloaded when
      // the adapter changes.
      const int q = warp & 3;
      const int m = q * 32 + lane;
      const int n = n0 + m;
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const float sw = sw_pre;
      const int g = lane >> 2, tq = lane & 3;     // MMA fragment coordinates
      // weight-row scales of this thread's fragment rows q*32 + mt*16 + g + 8h
      float swf[2][2];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = n0 + q * 32 + mt * 16 + g + 8 * h;
          swf[mt][h] = !C::kFP4 && row < p.N ? ldg_nc_f32_now(p.w_scale + row) : 0.0f;
        }
      // L2 prefetch of this warp's 32 B rows of the next adapter after column tl
      auto prefetch_next = [&](int l, int tl) {
        for (int base = tl + 1; base < tv; base += 32) {
          const int k = base + lane;
          const int lk = k < tv ? meta_idx[k] : -1;
          const uint32_t hit = __ballot_sync(0xffffffffu, lk >= 0 && lk != l);
          if (hit != 0u) {
            const int rows = min(32, p.N - (n0 + q * 32));
            if (lane == 0 && rows > 0)
              prefetch_l2_bulk(p.B + (static_cast<size_t>(meta_idx[base + __ffs(hit) - 1]) * p.N + n0 + q * 32) * p.r,
                               static_cast<uint32_t>(rows * p.r * 2));
            break;
          }
        }
      };
      auto run = [&](auto r4c) {
        constexpr int R4 = decltype(r4c)::value;     // float4 chunks of an S row
        constexpr bool kMma = R4 <= 8;               // tensor-core chunks: rank <= 32
        constexpr int KS = kMma ? R4 / 2 : 1;        // k-steps of 8
        int cur_l = -1;                              // adapter of brow
        int cur_la = -1;                             // adapter of the A fragments
        uint32_t af[2 * KS][4];                      // [mt * KS + ks]
        auto load_afrag = [&](int l) {
          const uint16_t* bl = reinterpret_cast<const uint16_t*>(p.B) + static_cast<size_t>(l) * p.N * p.r;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int row = n0 + q * 32 + mt * 16 + g + 8 * h;
#pragma unroll
              for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const uint32_t b = row < p.N ? __ldg(bl + static_cast<size_t>(row) * p.r + ks * 8 + tq + 4 * e) : 0u;
                  af[mt * KS + ks][h + 2 * e] = b << 16;     // bf16 -> fp32 (exact, also as TF32)
                }
            }
        };
#pragma unroll 1
        for (int c = 0; c < BT / 16; ++c) {
          if (c * 16 >= tv) break;
          // the chunk's adapters (the same for every thread): none, one, or several
          const int jl = c * 16 + (lane & 15);
          const int lj = jl < tv ? meta_idx[jl] : -1;
          const uint32_t actm = __ballot_sync(0xffffffffu, lj >= 0) & 0xffffu;
          if (kMma && p.stage_s && p.y_stage >= 0) {
            uint32_t va[2][8];
            tmem_ld_16x256b_x2(lane_base + c * 16, va[0]);
            tmem_ld_16x256b_x2(lane_base + (16u << 16) + c * 16, va[1]);
            float d[2][2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) d[mt][nt][i] = 0.0f;
            // one pass per adapter of the chunk, S of the other columns zeroed:
            // a column's sum is the same whichever chunk it falls in
            uint32_t rem = actm;
            while (rem != 0u) {
              const int l = meta_idx[c * 16 + __ffs(rem) - 1];
              const uint32_t cols = __ballot_sync(0xffffffffu, lj == l) & 0xffffu;
              rem &= ~cols;
              if (l != cur_la) {
                load_afrag(l);
                cur_la = l;
                prefetch_next(l, c * 16 + 31 - __clz(cols));
              }
#pragma unroll
              for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                  // S of token column c*16 + nt*8 + g, ranks ks*8 + tq and + 4
                  const bool on = (cols >> (nt * 8 + g)) & 1u;
                  const float* sp = s_big + (c * 16 + nt * 8 + g) * s_ld + ks * 8 + tq;
                  const float s0 = on ? sp[0] : 0.0f, s1 = on ? sp[4] : 0.0f;
                  const uint32_t h0 = f32_to_tf32(s0), h1 = f32_to_tf32(s1);
                  const uint32_t l0 = f32_to_tf32(s0 - __uint_as_float(h0));
                  const uint32_t l1 = f32_to_tf32(s1 - __uint_as_float(h1));
#pragma unroll
                  for (int mt = 0; mt < 2; ++mt) {
                    mma_tf32_m16n8k8(d[mt][nt], af[mt * KS + ks], l0, l1);
                    mma_tf32_m16n8k8(d[mt][nt], af[mt * KS + ks], h0, h1);
                  }
                }
            }
            tmem_ld_wait();
            // element (mt, nt, i): row q*32 + mt*16 + g + 8*(i/2), column
            // c*16 + nt*8 + 2*tq + i%2
            __nv_bfloat16* ys = y_stage_block();
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int col = nt * 8 + 2 * tq + (i & 1);
                  const float acc = __uint_as_float(va[mt][nt * 4 + i]);
                  const float b = C::kFP4 ? acc * alpha : (acc * meta_sx[c * 16 + col]) * swf[mt][i >> 1];
                  const float y = (actm >> col) & 1u ? b + d[mt][nt][i] : b;
                  ys[col * kYsLd + mt * 16 + g + 8 * (i >> 1)] = __float2bfloat16_rn(y);
                }
            flush16(c);
            continue;
          }
          uint32_t v[16];
          float yv[16] = {};
          tmem_ld_32x32b_x16(lane_base + c * 16, v);
          tmem_ld_wait();
          if (n < p.N) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int tl = c * 16 + j;
              if (tl < tv) {
                float y = base_value(m, tl, __uint_as_float(v[j]), sw);
                const int l = meta_idx[tl];
                if (l >= 0) {
                  if (l != cur_l) {
                    load_brow(l, m);
                    cur_l = l;
                  }
                  const float4* srow = p.stage_s ? reinterpret_cast<const float4*>(s_big + tl * s_ld)
                                                 : reinterpret_cast<const float4*>(
                                                       S_t + static_cast<size_t>(meta_tok[tl]) * p.s_row);
                  y += p.stage_s ? dot_srow_brow_n<R4, true>(srow, brow) : dot_srow_brow_n<R4, false>(srow, brow);
                }
                yv[j] = y;
              }
            }
          }
          if (p.y_stage >= 0) {
            emit16(c, yv);
          } else if (n < p.N) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c * 16 + j < tv) p.Y[static_cast<size_t>(meta_tok[c * 16 + j]) * p.ldy + n] = __float2bfloat16_rn(yv[j]);
          }
        }
      };
      if (p.yadd != nullptr) {
        // the adapter term comes from the expand pass: one fp32 per (sorted
        // row, output column), added to the base value as the CUDA-core term
        // below would be; the next chunk's values are requested before this
        // chunk is finished
        auto load_ya = [&](int c, float (&ya)[16]) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tl = c * 16 + j;
            ya[j] = tl < tv && n < p.N && meta_idx[tl] >= 0
                        ? __ldcg(p.yadd + static_cast<size_t>(t0 + tl) * p.N + n)
                        : 0.0f;
          }
        };
        float ya_next[16];
        load_ya(0, ya_next);
#pragma unroll 1
        for (int c = 0; c < BT / 16; ++c) {
          if (c * 16 >= tv) break;
          uint32_t v[16];
          float ya[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) ya[j] = ya_next[j];
          tmem_ld_32x32b_x16(lane_base + c * 16, v);
          if ((c + 1) * 16 < tv) load_ya(c + 1, ya_next);
          tmem_ld_wait();
          float yv[16] = {};
          if (n < p.N) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int tl = c * 16 + j;
              if (tl < tv) {
                float y = base_value(m, tl, __uint_as_float(v[j]), sw);
                if (meta_idx[tl] >= 0) y += ya[j];
                yv[j] = y;
              }
            }
          }
          if (p.y_stage >= 0) {
            emit16(c, yv);
          } else if (n < p.N) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c * 16 + j < tv) p.Y[static_cast<size_t>(meta_tok[c * 16 + j]) * p.ldy + n] = __float2bfloat16_rn(yv[j]);
          }
        }
      } else {
        switch (p.r) {
          case 16: run(std::integral_constant<int, 4>{}); break;
          case 32: run(std::integral_constant<int, 8>{}); break;
          case 64: run(std::integral_constant<int, 16>{}); break;
          default: run(std::integral_constant<int, 32>{}); break;
        }
      }
    } else if (ks == 1) {
      const int q = warp & 3;
      const int m = q * 32 + lane;
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const float sw = sw_pre;
#pragma unroll 1
      for (int c = 0; c < BT / 16; ++c) {
        if (c * 16 >= tv) break;
        uint32_t v[16];
        tmem_ld_32x32b_x16(lane_base + c * 16, v);
        tmem_ld_wait();
        if (C::kDecode) {
          // valid token columns to this thread's row of the output tile;
          // only they are finished below (a loop with a run-time bound, so
          // that no work is spent on the tile's empty columns)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c * 16 + j < tv) y_tile[(c * 16 + j) * RR + m] = __uint_as_float(v[j]);
        } else if (p.y_stage >= 0) {
          float yv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) yv[j] = base_value(m, c * 16 + j, __uint_as_float(v[j]), sw);
          emit16(c, yv);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) finish(m, c * 16 + j, __uint_as_float(v[j]), sw);
        }
      }
      if (C::kDecode) {
#pragma unroll 1
        for (int tl = 0; tl < tv; ++tl) finish(m, tl, y_tile[tl * RR + m], sw);
      }
    } else {
#pragma unroll 1
      for (int e = et; e < R * tv; e += 128) {
        const int i = e % R, tl = e / R;     // i == et % R: this thread's row
        const int mm = row_lo + i;
        float acc = 0.0f;
#pragma unroll
        for (int s = 0; s < kMaxSplit; ++s)
          if (s < ks) acc += red[(s * BT + tl) * RR + i];     // rank order: deterministic
        finish(mm, tl, acc, sw_pre);
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  if (b_early_on && et == 0 && *abort_flag) (void)mbar_wait_bounded(b_bar, 0, kWaitLimitNs);   // no copy in flight
  if (ks > 1 && warp < 2) cluster_wait();   // second phase, for the producer and MMA warps
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Host side ------------------------------------------------------------------
int gemm_smem_bytes(int stage_bytes, int stages, int red_bytes);

// CTAs per SM a decode grid larger than the GPU is sized for
constexpr int kResident = 2;

template <int FMT, int BT, int KA>
int launch_gemm_tiled(const GemmArgs& a) {
  using C = GemmCfg<FMT, BT, KA>;
  const bool fp4 = C::kFP4;
  const int kbytes = fp4 ? a.K / 2 : a.K;
  GemmParams p{};
  p.x_scale = a.x_scale;
  p.w_scale = a.w_scale;
  p.x_gs = a.x_global_scale;
  p.w_gs = a.w_global_scale;
  p.S = a.S;
  p.B = static_cast<const __nv_bfloat16*>(a.B);
  p.idx = a.idx;
  p.mask = a.mask;
  p.Y = static_cast<__nv_bfloat16*>(a.Y);
  p.status = a.status_dev;
  p.fused = a.fused;
  p.pdl = !a.fused && a.pdl_dependent ? 1 : 0;
  p.perm = a.perm;
  p.yadd = a.yadd;
  if (a.yadd != nullptr && (C::kDecode || a.S == nullptr)) return EPILORA_ERR_UNSUPPORTED;
  p.s_parts = a.s_parts < 1 ? 1 : a.s_parts;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.L = a.L;
  p.r = a.r;
  p.s_row = a.s_row > 0 ? a.s_row : a.r;
  p.n_slices = a.n_slices < 1 ? 1 : a.n_slices;
  for (int q = 0; q < 4; ++q) p.slice_end[q] = a.slice_end[q];
  p.ldy = a.ldy;
  p.num_kb = (kbytes + KA * kAtomBytes - 1) / (KA * kAtomBytes);
  p.rotate = 1;

  int rc = make_tma_2d_u8(&p.tmW, a.Wq, a.N, kbytes, kbytes, kTileN, kAtomBytes, true);
  if (rc != EPILORA_OK) return rc;
  rc = make_tma_2d_u8(&p.tmX, a.Xq, a.M, kbytes, kbytes, BT, kAtomBytes, true);
  if (rc != EPILORA_OK) return rc;
  if (fp4) {
    rc = make_tma_2d_u8(&p.tmSW, a.w_block_scale, a.N, a.K / 16, a.K / 16, kTileN, C::kSfRow, false);
    if (rc != EPILORA_OK) return rc;
    rc = make_tma_2d_u8(&p.tmSX, a.x_block_scale, a.M, a.K / 16, a.K / 16, BT, C::kSfRow, false);
    if (rc != EPILORA_OK) return rc;
  }

  // Decode grids: split K over clusters of 2/4/8 CTAs while the grid stays
  // resident (kResident CTAs per SM); a grid larger than the SM
  // count gets the shared memory of that many CTAs per SM.
  const int sms = num_sms();
  const int n_tiles = (a.N + kTileN - 1) / kTileN;
  const int t_tiles = (a.M + BT - 1) / BT;
  const long tiles = static_cast<long>(n_tiles) * t_tiles;
  int ks = 1;
  if (BT <= 64) {
    const int max_by_k = p.num_kb / 2 > 0 ? p.num_kb / 2 : 1;
    for (int cand = 2; cand <= kMaxSplit; cand *= 2)
      if (tiles * cand <= static_cast<long>(sms) * kResident && cand <= max_by_k) ks = cand;
  }
  p.ks = ks;
  const int RR = gemm_red_rows(ks);

  // streamed B (decode tiles): one TMA box of the tile's rows per adapter,
  // its inner extent the row of B (2r bytes, or r for stored FP8 rows, in
  // atoms of at most 128 B)
  p.b_scale = a.b_scale;
  const int brow_bytes = a.b_scale != nullptr ? a.r : 2 * a.r;
  p.b_box_bytes = brow_bytes >= 128 ? 128 : brow_bytes;
  p.b_atoms = brow_bytes > 128 ? brow_bytes / 128 : 1;
  p.stream_b = 0;
  p.b_group_bytes = (RR * brow_bytes + 1023) / 1024 * 1024;
  p.b_groups_per_slot = C::kStageBytes / p.b_group_bytes;
  if (p.b_groups_per_slot > BT) p.b_groups_per_slot = BT;
  if (C::kDecode && a.S != nullptr && p.b_groups_per_slot >= 1) {
    const uint64_t rows = static_cast<uint64_t>(a.L) * static_cast<uint64_t>(a.N);
    rc = make_tma_2d_swz(&p.tmB, a.B, rows, brow_bytes, brow_bytes, RR, p.b_box_bytes, p.b_box_bytes);
    if (rc != EPILORA_OK) return rc;
    p.stream_b = 1;
  }

  const long ctas = tiles * ks;
  // a grid larger than the GPU keeps kResident CTAs per SM: one
  // CTA's epilogue then runs while the other's main loop keeps the weight
  // stream (decode) or the tensor pipe (wide tiles) busy
  const int budget = ctas > sms ? (227 * 1024) / kResident - 2048 : 200 * 1024;
  const int red = gemm_red_bytes<BT>(ks);
  const int dec = gemm_decode_bytes(BT, a.r, ks);
  int stages = (budget - 1024 - red - kGemmMiscBytes - dec) / C::kStageBytes;
  if (stages > 16) stages = 16;
  const int per_cta = (p.num_kb + ks - 1) / ks;
  if (stages > per_cta && !p.stream_b) stages = per_cta;     // no deeper than the K loop needs
  if (stages < 2) p.stream_b = 0;        // B slots need a ring of two or more
  if (stages < 1) stages = 1;
  // one-group decode tiles: a buffer of its own for the B slice, if it fits
  // beside the ring without giving up a stage
  int early_bytes = 0;
  p.b_early = 0;
  if (p.stream_b) {
    early_bytes = p.b_group_bytes + 1024;      // + alignment of the swizzled box
    if (gemm_smem_bytes(C::kStageBytes, stages, red) + dec + early_bytes <= budget) p.b_early = 1;
    else early_bytes = 0;
  }
  // non-decode tiles stage S of their tokens in the ring once the main loop
  // is over (one fp32 row of r per token column); deepen the ring if needed
  p.stage_s = 0;
  if (!C::kDecode && a.S != nullptr && a.yadd == nullptr) {
    const int need = BT * (a.r + 4) * 4 + 5 * 1024;     // padded S rows + the output staging
    int st_need = (need + C::kStageBytes - 1) / C::kStageBytes;
    if (st_need < stages) st_need = stages;
    if (gemm_smem_bytes(C::kStageBytes, st_need, red) + dec <= budget) {
      stages = st_need;
      p.stage_s = 1;
    }
  }
  // wide tiles read a split shrink's partial sums only from the staged rows
  if (!C::kDecode && a.S != nullptr && a.yadd == nullptr && p.s_parts > 1 && !p.stage_s)
    return EPILORA_ERR_UNSUPPORTED;
  // stored FP8 B rows are read only by the streamed-B decode epilogue
  if (a.b_scale != nullptr && (!C::kDecode || !p.stream_b)) return EPILORA_ERR_UNSUPPORTED;
  p.stages = stages;
  // wide tiles without split K: output rows leave through a 5 KB staging
  // block placed after the staged S (16-byte stores need aligned rows)
  p.y_stage = -1;
  if (!C::kDecode && ks == 1 && (reinterpret_cast<uintptr_t>(a.Y) & 15) == 0 && a.ldy % 8 == 0) {
    const int off = p.stage_s ? (BT * (a.r + 4) * 4 + 127) / 128 * 128 : 0;
    if (off + 5 * 1024 <= stages * C::kStageBytes) p.y_stage = off;
  }
  // fused call: prefetch into L2 (while the shrink grid runs) up to about
  // kL2AheadBytes of weight stages beyond the ring, over the grid
  {
    const long budget_bytes = kL2AheadBytes;
    const long per_stage_grid = ctas * static_cast<long>(C::kWBytes + C::kSfWRaw);
    long ahead = per_stage_grid > 0 ? budget_bytes / per_stage_grid : 0;
    const long left = per_cta - stages;
    if (ahead > left) ahead = left;
    p.l2_ahead = a.fused && ahead > 0 ? static_cast<int>(ahead) : 0;
  }
  const int smem = gemm_smem_bytes(C::kStageBytes, stages, red) + dec + early_bytes;
  if (smem > 227 * 1024) return EPILORA_ERR_UNSUPPORTED;

  auto kern = gemm_lora_kernel<FMT, BT, KA>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return EPILORA_ERR_CUDA;
  if (attr_done[dev] < smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return EPILORA_ERR_CUDA;
    attr_done[dev] = smem;
  }

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(ks, t_tiles, n_tiles);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (ks > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = ks;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  if (a.pdl_dependent) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return EPILORA_ERR_CUDA;
  return EPILORA_OK;
}

}  // namespace epi

#include "gemm_wide.cuh"

namespace epi {

template <int FMT>
int launch_gemm_by_m(const GemmArgs& a) {
  if (a.b_scale != nullptr && a.M > kDecodeBT) return EPILORA_ERR_UNSUPPORTED;   // stored FP8 B: decode tiles only
  // decode tiles of 16 tokens: two 128-byte K atoms per stage (NVFP4 stages
  // also carry scale boxes: one atom keeps three or more stages in flight at
  // two CTAs per SM); 32-token decode tiles also keep output-tile and S
  // buffers: one atom per stage leaves room for three or more stages
  constexpr int KAD = FMT == EPILORA_FMT_NVFP4 ? 1 : 2;
  if (a.M <= 16) return launch_gemm_tiled<FMT, 16, KAD>(a);
  if (a.M <= 32) return launch_gemm_tiled<FMT, 32, 1>(a);
  if (a.M <= 64) return launch_gemm_tiled<FMT, 64, 2>(a);
  // wide token tiles: one atom per stage (a 256-token FP8 stage is then 48 KB
  // and the ring four deep); NVFP4 stages of 256 tokens carry scale boxes too
  // and at two CTAs per SM the ring would be one stage deep, so NVFP4 stays
  // at 128-token tiles
  if (a.M <= 128 || FMT == EPILORA_FMT_NVFP4) return launch_gemm_tiled<FMT, 128, 1>(a);
  if constexpr (FMT == EPILORA_FMT_FP8_E4M3) {
    const int rc = launch_gemm_wide<FMT>(a);     // persistent, two accumulators
    if (rc != EPILORA_ERR_UNSUPPORTED) return rc;
  }
  return launch_gemm_tiled<FMT, 256, 1>(a);
}

}  // namespace epi
