// Low-precision base GEMM with the multi-adapter LoRA epilogue ("K2"), on the
// 5th-generation tensor cores of sm_103a.
//
// EpiLoRA, "Fusing Many LoRA Adapters into Low-Precision GEMMs for Serving and
// RL":
//  * §Design › Multi-adapter kernels › K1 and K2 — the GEMM's epilogue applies
//    the weight and activation scales and then adds h_l B_l^T for the rows of
//    each adapter, reading only the tile's slice of B_l;
//  * › The decode path — the GEMM runs as the shrink's programmatic dependent:
//    it streams its weights while the shrink runs and waits for h only before
//    its epilogue; it prefetches B;
//  * › When the overlap hides the adapter — exposure grows when the GEMM has
//    more CTAs than SMs, so the decode grid is sized to one wave.
//
// GB300 design (not the pages' Triton kernel):
//  * swap-AB: weight rows are the MMA's M = 128 side (TMEM lanes), tokens the
//    MMA's N side (BT = 16..256 TMEM columns), so a decode batch of 1..32
//    tokens still issues full-height MMAs while W streams;
//  * one elected thread issues tcgen05.mma (kind::f8f6f4 for E4M3, or
//    kind::mxf4nvf4 block-scaled with UE4M3 scales for NVFP4) on 128-byte
//    swizzled K-major tiles that TMA writes into a multi-stage ring;
//    the accumulator lives in TMEM;
//  * few output tiles (decode): the K dimension is split over a thread-block
//    cluster of KS CTAs; each CTA's fp32 partial tile is reduced through
//    distributed shared memory in rank order (deterministic, no atomics),
//    each CTA finishing 128/KS rows;
//  * epilogue warps prefetch the tile's B_l slices into L2 at kernel start,
//    read TMEM after the main loop, then execute griddepcontrol.wait (the
//    shrink's completion) before reading S.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM allocator
// and MMA issuer (all 32 lanes re-lay NVFP4 scale factors), warps 2..5 =
// epilogue (warp w reads TMEM lane quadrant w % 4).
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace epi {

constexpr int kGemmThreads = 192;
constexpr int kTileN = 128;          // weight rows per tile (MMA M)
constexpr int kStageKBytes = 128;    // bytes of K per stage and row (one 128-B swizzle atom)
constexpr int kMaxRank = 128;

struct GemmParams {
  CUtensorMap tmW;    // uint8 [N, Kbytes], box 128 x 128 B, 128-B swizzle
  CUtensorMap tmX;    // uint8 [M, Kbytes], box BT x 128 B, 128-B swizzle
  CUtensorMap tmSW;   // NVFP4: uint8 [N, K/16], box 128 x 16 B
  CUtensorMap tmSX;   // NVFP4: uint8 [M, K/16], box BT x 16 B
  const float* x_scale;
  const float* w_scale;
  const float* x_gs;
  const float* w_gs;
  const float* S;
  const __nv_bfloat16* B;
  const int32_t* idx;
  const uint8_t* mask;
  __nv_bfloat16* Y;
  int* status;
  int M, N, K, L, r, ldy;
  int num_kb;         // stages of K in total
  int ks;             // cluster size along K (1 = no split)
  int stages;         // depth of the smem ring
};

template <int FMT, int BT>
struct GemmCfg {
  static constexpr bool kFP4 = (FMT == EPILORA_FMT_NVFP4);
  static constexpr int kWBytes = kTileN * kStageKBytes;           // 16 KB
  static constexpr int kXBytes = BT * kStageKBytes;               // multiple of 1 KB
  static constexpr int kSfAtomsB = (BT + 127) / 128;              // scale atoms per K=64 step for tokens
  static constexpr int kSfABytes = kFP4 ? 4 * 512 : 0;            // 4 K-steps x 512-B atom
  static constexpr int kSfBBytes = kFP4 ? 4 * 512 * kSfAtomsB : 0;
  static constexpr int kSfWRaw = kFP4 ? kTileN * 16 : 0;          // TMA box of W scales
  static constexpr int kSfXRaw = kFP4 ? BT * 16 : 0;              // TMA box of X scales
  static constexpr int kStageRaw = kWBytes + kXBytes + kSfABytes + kSfBBytes + kSfWRaw + kSfXRaw;
  static constexpr int kStageBytes = (kStageRaw + 1023) / 1024 * 1024;
  static constexpr int kStageTx = kWBytes + kXBytes + kSfWRaw + kSfXRaw;   // bytes TMA delivers per stage
  // TMEM: accumulator columns [0, BT); NVFP4 scale columns after it, two slots.
  static constexpr int kSfColsA = 16;                             // 4 K-steps x 4 columns
  static constexpr int kSfColsB = 16 * kSfAtomsB;
  static constexpr int kSfSlotCols = kSfColsA + kSfColsB;
  static constexpr int kTmemNeed = BT + (kFP4 ? 2 * kSfSlotCols : 0);
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
  static constexpr uint32_t kIdesc = kFP4 ? idesc_mxf4nvf4(kTileN, BT) : idesc_f8f6f4_e4m3(kTileN, BT);
  static_assert(BT % 16 == 0 && BT >= 16 && BT <= 256, "token tile");
  static_assert(kTmemNeed <= 512, "TMEM");
};

// bytes of dynamic shared memory beyond the stage ring
template <int BT>
__host__ __device__ constexpr int gemm_misc_bytes() { return 4096; }

template <int BT>
__host__ __device__ constexpr int gemm_red_bytes(int ks) { return ks > 1 ? kTileN * BT * 4 : 0; }

template <int FMT, int BT>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_lora_kernel(const __grid_constant__ GemmParams p) {
  using C = GemmCfg<FMT, BT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stages = p.stages;
  uint8_t* red_buf = smem + static_cast<size_t>(stages) * C::kStageBytes;
  uint8_t* misc = red_buf + gemm_red_bytes<BT>(p.ks);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(misc);
  uint64_t* empty_bar = full_bar + stages;
  uint64_t* acc_bar = empty_bar + stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* meta_sx = reinterpret_cast<float*>(tmem_slot + 4);
  int* meta_idx = reinterpret_cast<int*>(meta_sx + BT);       // adapter slot, -1 = none

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ks = p.ks;
  const int rank = ks > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int t0 = blockIdx.y * BT;
  const int n0 = blockIdx.z * kTileN;
  const int kb_begin = (p.num_kb * rank) / ks;
  const int kb_end = (p.num_kb * (rank + 1)) / ks;
  const int nkb = kb_end - kb_begin;

  // ---------------------------------------------------------------- setup
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(acc_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&p.tmW);
    tma_prefetch_desc(&p.tmX);
    if (C::kFP4) {
      tma_prefetch_desc(&p.tmSW);
      tma_prefetch_desc(&p.tmSX);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    const int et = threadIdx.x - 64;
    for (int i = et; i < BT; i += 128) {
      const int t = t0 + i;
      float sx = 0.0f;
      int l = -1;
      if (t < p.M) {
        if (!C::kFP4) sx = p.x_scale[t];
        if (p.S != nullptr) {
          const int li = p.idx[t];
          const bool on = li >= 0 && li < p.L && (p.mask == nullptr || p.mask[t] != 0);
          if (li >= p.L) record_status(p.status, EPILORA_ERR_INVALID_ARG);
          l = on ? li : -1;
        }
      }
      meta_sx[i] = sx;
      meta_idx[i] = l;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // ---------------------------------------------------------------- roles
  if (warp == 0) {
    // ===== TMA producer =====
    if (lane == 0) {
      uint32_t issued_mask = 0, parity_mask = 0;   // per stage: a fill was issued / its phase parity
      for (int i = 0; i < nkb; ++i) {
        const int s = i % stages;
        const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
        if (*abort_flag) break;
        if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, kWaitLimitNs)) {
          *abort_flag = 1;
          record_status(p.status, EPILORA_ERR_TIMEOUT);
          break;
        }
        uint8_t* st = smem + static_cast<size_t>(s) * C::kStageBytes;
        const int kb = kb_begin + i;
        mbar_arrive_expect_tx(&full_bar[s], C::kStageTx);
        tma_load_2d(st, &p.tmW, &full_bar[s], kb * kStageKBytes, n0);
        tma_load_2d(st + C::kWBytes, &p.tmX, &full_bar[s], kb * kStageKBytes, t0);
        if (C::kFP4) {
          uint8_t* raw = st + C::kWBytes + C::kXBytes + C::kSfABytes + C::kSfBBytes;
          tma_load_2d(raw, &p.tmSW, &full_bar[s], kb * 16, n0);
          tma_load_2d(raw + C::kSfWRaw, &p.tmSX, &full_bar[s], kb * 16, t0);
        }
        issued_mask |= 1u << s;
        parity_mask = (parity_mask & ~(1u << s)) | (ph << s);
      }
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
      if (C::kFP4) {
        // Re-lay the canonical [rows][16 scale bytes] TMA boxes into 512-B
        // atoms per K=64 step: line r0 (16 B) = the 4 scale bytes of rows
        // r0, r0+32, r0+64, r0+96 (4 bytes each).
        uint8_t* sfa = st + C::kWBytes + C::kXBytes;
        uint8_t* sfb = sfa + C::kSfABytes;
        const uint8_t* raw_w = sfb + C::kSfBBytes;
        const uint8_t* raw_x = raw_w + C::kSfWRaw;
        {
          uint4 v[4];
#pragma unroll
          for (int r1 = 0; r1 < 4; ++r1) v[r1] = *reinterpret_cast<const uint4*>(raw_w + (lane + 32 * r1) * 16);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            uint4 o;
            o.x = (&v[0].x)[kk];
            o.y = (&v[1].x)[kk];
            o.z = (&v[2].x)[kk];
            o.w = (&v[3].x)[kk];
            *reinterpret_cast<uint4*>(sfa + kk * 512 + lane * 16) = o;
          }
        }
#pragma unroll
        for (int a = 0; a < C::kSfAtomsB; ++a) {
          uint4 v[4];
#pragma unroll
          for (int r1 = 0; r1 < 4; ++r1) {
            const int row = 128 * a + 32 * r1 + lane;
            v[r1] = row < BT ? *reinterpret_cast<const uint4*>(raw_x + row * 16) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            uint4 o;
            o.x = (&v[0].x)[kk];
            o.y = (&v[1].x)[kk];
            o.z = (&v[2].x)[kk];
            o.w = (&v[3].x)[kk];
            *reinterpret_cast<uint4*>(sfb + (kk * C::kSfAtomsB + a) * 512 + lane * 16) = o;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t slot_col = static_cast<uint32_t>(BT + (i & 1) * C::kSfSlotCols);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t adesc = make_smem_desc(w_addr + kk * 32, 16, 1024, kSwizzle128B);
          const uint64_t bdesc = make_smem_desc(x_addr + kk * 32, 16, 1024, kSwizzle128B);
          const uint32_t accum = (i > 0 || kk > 0) ? 1u : 0u;
          if (C::kFP4) {
            const uint32_t sfa_addr = smem_u32(st + C::kWBytes + C::kXBytes) + kk * 512;
            const uint32_t sfb_addr = smem_u32(st + C::kWBytes + C::kXBytes + C::kSfABytes) + kk * C::kSfAtomsB * 512;
            const uint32_t sfa_col = slot_col + kk * 4;
            const uint32_t sfb_col = slot_col + C::kSfColsA + kk * 4 * C::kSfAtomsB;
            tc_cp_32x128b_warpx4(tmem_base + sfa_col, make_smem_desc(sfa_addr, 16, 128, kSwizzleNone));
#pragma unroll
            for (int a = 0; a < C::kSfAtomsB; ++a)
              tc_cp_32x128b_warpx4(tmem_base + sfb_col + 4 * a,
                                   make_smem_desc(sfb_addr + a * 512, 16, 128, kSwizzleNone));
            mma_mxf4nvf4(tmem_base, adesc, bdesc, C::kIdesc, tmem_base + sfa_col, tmem_base + sfb_col, accum);
          } else {
            mma_f8f6f4(tmem_base, adesc, bdesc, C::kIdesc, accum);
          }
        }
        tc_commit(&empty_bar[s]);   // frees the stage once these MMAs have read it
      }
      __syncwarp();
    }
    if (lane == 0) tc_commit(acc_bar);   // accumulator complete (or drained after an abort)
    __syncwarp();
  } else {
    // ===== epilogue warps: prefetch B slices, then wait for the accumulator =====
    const int et = threadIdx.x - 64;   // 0..127
    const int q = warp & 3;            // TMEM lane quadrant of this warp
    const int m = q * 32 + lane;       // tile row owned in the unsplit case
    const int row_lo = (kTileN * rank) / ks, row_hi = (kTileN * (rank + 1)) / ks;
    if (et == 0 && p.S != nullptr) {
      const int rows = min(row_hi, p.N - n0) - row_lo;
      if (rows > 0) {
        int prev = -1;
        for (int i = 0; i < BT; ++i) {
          const int l = meta_idx[i];
          if (l >= 0 && l != prev) {
            prefetch_l2_bulk(p.B + (static_cast<size_t>(l) * p.N + n0 + row_lo) * p.r,
                             static_cast<uint32_t>(rows * p.r * 2));
            prev = l;
          }
        }
      }
    }
    bool ok = mbar_wait_bounded(acc_bar, 0, kWaitLimitNs);
    if (!ok) {
      *abort_flag = 1;
      record_status(p.status, EPILORA_ERR_TIMEOUT);
    }
    tc_fence_after();
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    if (ks > 1 && ok) {
      // stage this CTA's fp32 partial tile for the cluster reduction: red[t][m]
      float* red = reinterpret_cast<float*>(red_buf);
#pragma unroll 1
      for (int c = 0; c < BT / 16; ++c) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(lane_base + c * 16, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) red[(c * 16 + j) * kTileN + m] = __uint_as_float(v[j]);
      }
    }
  }

  // ---------------------------------------------------------------- epilogue
  // Per element (tile row mm, token column tl) with its fp32 accumulator:
  //   y = acc * scales + [token has an adapter] * sum_j S[t, j] * B[l, n, j]
  // B rows are cached in registers while consecutive tokens share an adapter.
  auto finish = [&](int mm, int tl, float acc, int& cached_key, uint32_t (&brow)[kMaxRank / 2], float alpha,
                    float sw) {
    const int n = n0 + mm;
    const int t = t0 + tl;
    if (n >= p.N || t >= p.M) return;
    float y = C::kFP4 ? acc * alpha : (acc * meta_sx[tl]) * sw;
    const int l = meta_idx[tl];
    if (l >= 0) {
      const int key = l * kTileN + mm;
      if (key != cached_key) {
        const uint4* bsrc = reinterpret_cast<const uint4*>(p.B + (static_cast<size_t>(l) * p.N + n) * p.r);
#pragma unroll
        for (int c = 0; c < kMaxRank / 8; ++c) {
          if (c < p.r / 8) {
            const uint4 v = __ldg(bsrc + c);
            brow[4 * c + 0] = v.x;
            brow[4 * c + 1] = v.y;
            brow[4 * c + 2] = v.z;
            brow[4 * c + 3] = v.w;
          }
        }
        cached_key = key;
      }
      const float4* srow = reinterpret_cast<const float4*>(p.S + static_cast<size_t>(t) * p.r);
      float d = 0.0f;
#pragma unroll
      for (int c = 0; c < kMaxRank / 4; ++c) {
        if (c < p.r / 4) {
          const float4 s4 = __ldcg(srow + c);
          d = fmaf(s4.x, bf16_lo(brow[2 * c]), d);
          d = fmaf(s4.y, bf16_hi(brow[2 * c]), d);
          d = fmaf(s4.z, bf16_lo(brow[2 * c + 1]), d);
          d = fmaf(s4.w, bf16_hi(brow[2 * c + 1]), d);
        }
      }
      y += d;
    }
    p.Y[static_cast<size_t>(t) * p.ldy + n] = __float2bfloat16_rn(y);
  };

  const int aborted = __shfl_sync(0xffffffffu, *abort_flag, 0);   // warp-uniform
  if (ks == 1) {
    if (warp >= 2 && !aborted) {
      const int q = warp & 3;
      const int m = q * 32 + lane;
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const float alpha = C::kFP4 ? 1.0f / (*p.x_gs * *p.w_gs) : 1.0f;
      const float sw = (!C::kFP4 && n0 + m < p.N) ? p.w_scale[n0 + m] : 0.0f;
      if (p.S != nullptr) pdl_wait_primary();   // the shrink has completed: S is visible
      int cached_key = -1;
      uint32_t brow[kMaxRank / 2];
#pragma unroll 1
      for (int c = 0; c < BT / 16; ++c) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(lane_base + c * 16, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) finish(m, c * 16 + j, __uint_as_float(v[j]), cached_key, brow, alpha, sw);
      }
    }
  } else {
    // partials of every CTA of the cluster are in their shared memory
    cluster_arrive();
    cluster_wait();
    if (warp >= 2 && !__shfl_sync(0xffffffffu, *abort_flag, 0)) {
      const int et = threadIdx.x - 64;
      const int row_lo = (kTileN * rank) / ks, row_hi = (kTileN * (rank + 1)) / ks;
      const int R = row_hi - row_lo;
      const float alpha = C::kFP4 ? 1.0f / (*p.x_gs * *p.w_gs) : 1.0f;
      const uint32_t red_addr = smem_u32(red_buf);
      if (p.S != nullptr) pdl_wait_primary();
      int cached_key = -1;
      uint32_t brow[kMaxRank / 2];
      int sw_row = -1;
      float sw = 0.0f;
#pragma unroll 1
      for (int e = et; e < R * BT; e += 128) {
        const int mm = row_lo + e % R;
        const int tl = e / R;
        const uint32_t off = static_cast<uint32_t>((tl * kTileN + mm) * 4);
        float acc = 0.0f;
        for (int s = 0; s < ks; ++s) acc += ld_dsmem_f32(map_to_cta(red_addr + off, static_cast<uint32_t>(s)));
        if (!C::kFP4 && mm != sw_row) {
          sw = (n0 + mm < p.N) ? p.w_scale[n0 + mm] : 0.0f;
          sw_row = mm;
        }
        finish(mm, tl, acc, cached_key, brow, alpha, sw);
      }
    }
    // peers may still be reading this CTA's partials
    cluster_arrive();
    cluster_wait();
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Host side ------------------------------------------------------------------
int gemm_smem_bytes(int stage_bytes, int stages, int red_bytes);

template <int FMT, int BT>
int launch_gemm_tiled(const GemmArgs& a) {
  using C = GemmCfg<FMT, BT>;
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
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.L = a.L;
  p.r = a.r;
  p.ldy = a.ldy;
  p.num_kb = (kbytes + kStageKBytes - 1) / kStageKBytes;

  int rc = make_tma_2d_u8(&p.tmW, a.Wq, a.N, kbytes, kbytes, kTileN, kStageKBytes, true);
  if (rc != EPILORA_OK) return rc;
  rc = make_tma_2d_u8(&p.tmX, a.Xq, a.M, kbytes, kbytes, BT, kStageKBytes, true);
  if (rc != EPILORA_OK) return rc;
  if (fp4) {
    rc = make_tma_2d_u8(&p.tmSW, a.w_block_scale, a.N, a.K / 16, a.K / 16, kTileN, 16, false);
    if (rc != EPILORA_OK) return rc;
    rc = make_tma_2d_u8(&p.tmSX, a.x_block_scale, a.M, a.K / 16, a.K / 16, BT, 16, false);
    if (rc != EPILORA_OK) return rc;
  }

  const int n_tiles = (a.N + kTileN - 1) / kTileN;
  const int t_tiles = (a.M + BT - 1) / BT;
  const long tiles = static_cast<long>(n_tiles) * t_tiles;
  int ks = 1;
  if (BT <= 64) {
    const long fit = num_sms() / tiles;
    ks = static_cast<int>(fit < 1 ? 1 : fit > 8 ? 8 : fit);
    const int max_by_k = p.num_kb / 2 > 0 ? p.num_kb / 2 : 1;
    if (ks > max_by_k) ks = max_by_k;
  }
  p.ks = ks;
  const int red = gemm_red_bytes<BT>(ks);
  const int budget = 200 * 1024;
  int stages = (budget - 1024 - red - gemm_misc_bytes<BT>()) / C::kStageBytes;
  if (stages > 16) stages = 16;
  if (stages > p.num_kb / ks + 1) stages = p.num_kb / ks + 1;   // no deeper than the K loop needs
  if (stages < 2) stages = 2;
  p.stages = stages;
  const int smem = gemm_smem_bytes(C::kStageBytes, stages, red) ;

  auto kern = gemm_lora_kernel<FMT, BT>;
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

template <int FMT>
int launch_gemm_by_m(const GemmArgs& a) {
  if (a.M <= 16) return launch_gemm_tiled<FMT, 16>(a);
  if (a.M <= 32) return launch_gemm_tiled<FMT, 32>(a);
  if (a.M <= 64) return launch_gemm_tiled<FMT, 64>(a);
  if (a.M <= 128) return launch_gemm_tiled<FMT, 128>(a);
  return launch_gemm_tiled<FMT, 256>(a);
}

}  // namespace epi
