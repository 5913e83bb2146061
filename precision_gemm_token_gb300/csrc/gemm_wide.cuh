// Persistent wide-tile FP8 GEMM with the LoRA epilogue (token tiles of 256,
// one CTA per SM, two TMEM accumulators).
//
// The same layer as gemm_lora_kernel (Y = bf16(sx * sw * sum_k xq wq +
// [active] S[t] . B[idx_t][n])) for batches whose 256-token tiles outnumber
// the SMs. Each CTA walks tiles blockIdx.x, + gridDim.x, ... (token tile
// fastest, so that the CTAs in flight share weight tiles in L2). Roles:
//   warp 0      TMA producer: W and X stages of every tile through one ring
//   warp 1      MMA issuer: tile j accumulates into TMEM buffer j % 2
//   warps 2..5  epilogue: tile j's token metadata and S rows are staged
//               while its MMAs run; then base + adapter term leave buffer
//               j % 2 while the MMAs of tile j + 1 fill the other buffer.
// The adapter term comes from TF32 mma.sync passes in the accumulator layout
// of tcgen05.ld.16x256b (one pass per adapter present in a 16-column chunk,
// S split hi + lo, the adapter rows exact in TF32), or, when the expand pass
// has computed it (KS = -1), from its fp32 buffer.
//
// Every wait is bounded: on a timeout the CTA records EPILORA_ERR_TIMEOUT,
// stops issuing, waits (bounded) for its copies and MMAs in flight and frees
// its TMEM.
#pragma once

namespace epi {

constexpr int kWideBT = 256;
constexpr int kWideTmemCols = 512;         // two 256-column accumulators

// KS: k-steps of 8 in the adapter rank (r = 8 KS); 0: no adapters; -1: the
// adapter term is read from p.yadd
template <int KS>
__device__ __forceinline__ void wide_load_afrag(uint32_t (&af)[2 * (KS > 0 ? KS : 1)][4], const GemmParams& p,
                                                int l, int rbase, int g, int tq) {
  const uint16_t* bl = reinterpret_cast<const uint16_t*>(p.B) + static_cast<size_t>(l) * p.N * p.r;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = rbase + mt * 16 + g + 8 * h;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t b = row < p.N ? __ldg(bl + static_cast<size_t>(row) * p.r + ks * 8 + tq + 4 * e) : 0u;
          af[mt * KS + ks][h + 2 * e] = b << 16;     // bf16 -> fp32 (exact, also as TF32)
        }
    }
}

template <int KS>
__device__ __forceinline__ void wide_epilogue_tile(const GemmParams& p, uint32_t tmem_acc, const float* meta_sx,
                                                   const int* meta_idx, const int* meta_tok, const float* s_big,
                                                   int s_ld, __nv_bfloat16* ys, int t0, int n0, int tv, int warp,
                                                   int lane) {
  constexpr int kYsLd = 40;
  const int q = warp & 3;
  const int g = lane >> 2, tq = lane & 3;
  const uint32_t lane_base = tmem_acc + (static_cast<uint32_t>(q * 32) << 16);
  float swf[2][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = n0 + q * 32 + mt * 16 + g + 8 * h;
      swf[mt][h] = row < p.N ? ldg_nc_f32_now(p.w_scale + row) : 0.0f;
    }
  uint32_t af[2 * (KS > 0 ? KS : 1)][4];
  int cur_la = -1;
#pragma unroll 1
  for (int c = 0; c < kWideBT / 16; ++c) {
    if (c * 16 >= tv) break;
    const int jl = c * 16 + (lane & 15);
    const int lj = KS != 0 && jl < tv ? meta_idx[jl] : -1;
    const uint32_t actm = __ballot_sync(0xffffffffu, lj >= 0) & 0xffffu;
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
    if constexpr (KS > 0) {
      // one pass per adapter of the chunk, S of the other columns zeroed: a
      // column's sum is the same whichever chunk it falls in
      uint32_t rem = actm;
      while (rem != 0u) {
        const int l = meta_idx[c * 16 + __ffs(rem) - 1];
        const uint32_t cols = __ballot_sync(0xffffffffu, lj == l) & 0xffffu;
        rem &= ~cols;
        if (l != cur_la) {
          wide_load_afrag<KS>(af, p, l, n0 + q * 32, g, tq);
          cur_la = l;
        }
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
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
    } else if constexpr (KS < 0) {
      // the expand pass's term of element (mt, nt, i) (layout below)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int col = nt * 8 + 2 * tq + (i & 1);
            const int row = n0 + q * 32 + mt * 16 + g + 8 * (i >> 1);
            if (((actm >> col) & 1u) && row < p.N)
              d[mt][nt][i] = __ldcg(p.yadd + static_cast<size_t>(t0 + c * 16 + col) * p.N + row);
          }
    }
    tmem_ld_wait();
    // element (mt, nt, i): row q*32 + mt*16 + g + 8*(i/2), column
    // c*16 + nt*8 + 2*tq + i%2
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int col = nt * 8 + 2 * tq + (i & 1);
          const float acc = __uint_as_float(va[mt][nt * 4 + i]);
          const float b = (acc * meta_sx[c * 16 + col]) * swf[mt][i >> 1];
          const float y = (actm >> col) & 1u ? b + d[mt][nt][i] : b;
          ys[col * kYsLd + mt * 16 + g + 8 * (i >> 1)] = __float2bfloat16_rn(y);
        }
    __syncwarp();
    // 16-byte row segments, 8 token rows per store instruction
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
    __syncwarp();
  }
}

template <int KS>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_wide_kernel(const __grid_constant__ GemmParams p) {
  using C = GemmCfg<EPILORA_FMT_FP8_E4M3, kWideBT, 1>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stages = p.stages;
  // [ring][S rows (KS > 0)][output staging][barriers, metadata]
  float* s_big = reinterpret_cast<float*>(smem + static_cast<size_t>(stages) * C::kStageBytes);
  const int s_ld = p.r + 4;
  __nv_bfloat16* ystage = reinterpret_cast<__nv_bfloat16*>(smem + p.y_stage);
  uint8_t* misc = smem + p.y_stage + 4 * 16 * 40 * 2;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(misc);
  uint64_t* empty_bar = full_bar + stages;
  uint64_t* accf_bar = empty_bar + stages;     // [2] accumulator b complete
  uint64_t* acce_bar = accf_bar + 2;           // [2] accumulator b read out
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* meta_sx = reinterpret_cast<float*>(tmem_slot + 4);
  int* meta_idx = reinterpret_cast<int*>(meta_sx + kWideBT);
  int* meta_tok = meta_idx + kWideBT;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int et = threadIdx.x - 64;
  const int t_tiles = p.t_tiles;
  const int tiles = t_tiles * p.n_tiles;
  const int nkb = p.num_kb;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], 1);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&p.tmW);
    tma_prefetch_desc(&p.tmX);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kWideTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ===== TMA producer =====
    if (lane == 0) {
      uint32_t issued_mask = 0, parity_mask = 0;
      bool stop = false;
      long it = 0;
      bool waited = !p.fused;
      for (int tile = blockIdx.x; tile < tiles && !stop; tile += gridDim.x) {
        const int t0 = (tile % t_tiles) * kWideBT;
        const int n0 = (tile / t_tiles) * kTileN;
        const int rot = static_cast<int>(((tile / t_tiles) * 5u) % static_cast<unsigned>(nkb));
        // fused call, first tile: the weights of the first ring's worth of
        // stages before griddepcontrol.wait, their activations after it
        const int pre = waited ? 0 : min(nkb, stages);
        for (int i = 0; i < nkb && !stop; ++i) {
          const int s = static_cast<int>(it % stages);
          const uint32_t ph = static_cast<uint32_t>(it / stages) & 1u;
          if (*abort_flag || !mbar_wait_bounded(&empty_bar[s], ph ^ 1u, kWaitLimitNs)) {
            *abort_flag = 1;
            record_status(p.status, EPILORA_ERR_TIMEOUT);
            stop = true;
            break;
          }
          int kb = i + rot;
          if (kb >= nkb) kb -= nkb;
          uint8_t* st = smem + static_cast<size_t>(s) * C::kStageBytes;
          mbar_arrive_expect_tx(&full_bar[s], C::kStageTx);
          tma_load_2d(st, &p.tmW, &full_bar[s], kb * kAtomBytes, n0);
          if (i >= pre) tma_load_2d(st + C::kWBytes, &p.tmX, &full_bar[s], kb * kAtomBytes, t0);
          issued_mask |= 1u << s;
          parity_mask = (parity_mask & ~(1u << s)) | (ph << s);
          ++it;
          if (!waited && i == pre - 1) {
            // the shrink grid quantizes the activations: its completion
            // makes them visible
            pdl_wait_primary();
            fence_proxy_async_global();
            waited = true;
            for (int i2 = 0; i2 < pre; ++i2) {
              int kb2 = i2 + rot;
              if (kb2 >= nkb) kb2 -= nkb;
              const int s2 = static_cast<int>((it - pre + i2) % stages);
              tma_load_2d(smem + static_cast<size_t>(s2) * C::kStageBytes + C::kWBytes, &p.tmX, &full_bar[s2],
                          kb2 * kAtomBytes, t0);
            }
          }
        }
      }
      if (*abort_flag) {
        // no copy in flight at exit
        for (int s = 0; s < stages && s < 32; ++s)
          if (issued_mask & (1u << s)) (void)mbar_wait_bounded(&full_bar[s], (parity_mask >> s) & 1u, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===== MMA issuer =====
    long it = 0;
    int j = 0;
    bool stop = false;
    for (int tile = blockIdx.x; tile < tiles && !stop; tile += gridDim.x, ++j) {
      const int b = j & 1;
      // the epilogue has read this accumulator's previous tile
      const bool oke = __all_sync(0xffffffffu, mbar_wait_bounded(&acce_bar[b], ((j >> 1) & 1) ^ 1u, kWaitLimitNs));
      if (!oke || *abort_flag) {
        if (lane == 0) {
          *abort_flag = 1;
          record_status(p.status, EPILORA_ERR_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * kWideBT);
      for (int i = 0; i < nkb; ++i) {
        const int s = static_cast<int>(it % stages);
        const uint32_t ph = static_cast<uint32_t>(it / stages) & 1u;
        const int ab = __shfl_sync(0xffffffffu, *abort_flag, 0);
        const bool ok = !ab && __all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[s], ph, kWaitLimitNs));
        if (!ok) {
          if (lane == 0) {
            *abort_flag = 1;
            record_status(p.status, EPILORA_ERR_TIMEOUT);
          }
          stop = true;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t w_addr = smem_u32(smem + static_cast<size_t>(s) * C::kStageBytes);
          const uint32_t x_addr = w_addr + C::kWBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = make_smem_desc(w_addr + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bdesc = make_smem_desc(x_addr + kk * 32, 16, 1024, kSwizzle128B);
            mma_f8f6f4(d_tmem, adesc, bdesc, C::kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&empty_bar[s]);   // frees the stage once these MMAs have read it
        }
        __syncwarp();
        ++it;
      }
      if (lane == 0) tc_commit(&accf_bar[b]);   // accumulator complete (or drained after an abort)
      __syncwarp();
    }
    if (lane == 0) {
      // nothing of this warp still in flight at exit: the last commit covers
      // every MMA issued before it
      const int nt = j;     // tiles started (the last one may be partial)
      if (nt > 0) {
        const int bl = (nt - 1) & 1;
        (void)mbar_wait_bounded(&accf_bar[bl], ((nt - 1) >> 1) & 1u, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else {
    // ===== epilogue warps =====
    // the primary grid: in the fused call the shrink grid (quantized
    // activations, scales, S, perm); in a standalone dependent launch the
    // kernel that writes S, idx or mask
    if (p.fused || p.pdl) pdl_wait_primary();
    __nv_bfloat16* ys = ystage + (warp & 3) * 16 * 40;
    int j = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++j) {
      const int t0 = (tile % t_tiles) * kWideBT;
      const int n0 = (tile / t_tiles) * kTileN;
      const int tv = min(kWideBT, p.M - t0);
      const int b = j & 1;
      // token metadata and S rows of the tile, while its MMAs run
      asm volatile("bar.sync %0, 128;" ::"r"(kEpiBarrier) : "memory");   // the previous tile is written out
      for (int i = et; i < kWideBT; i += 128) {
        const int row = t0 + i;
        float sx = 0.0f;
        int l = -1;
        int tok = row;
        if (row < p.M) {
          if (p.perm != nullptr) tok = p.perm[row];
          sx = p.x_scale[row];
          if (KS != 0) {
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
      if (KS > 0) {
        const int n4 = p.r / 4;
        const size_t part = static_cast<size_t>(p.M) * p.s_row / 4;   // partial sums of a split shrink, in part order
        const float* S_t = p.S + s_slice_offset(p, n0);               // this tile's slice of S rows
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
      const bool ok = mbar_wait_bounded(&accf_bar[b], (j >> 1) & 1u, kWaitLimitNs);
      if (!ok) {
        *abort_flag = 1;
        record_status(p.status, EPILORA_ERR_TIMEOUT);
      }
      if (epi_bar_any(*abort_flag != 0)) break;
      tc_fence_after();
      wide_epilogue_tile<KS>(p, tmem_base + static_cast<uint32_t>(b * kWideBT), meta_sx, meta_idx, meta_tok, s_big,
                             s_ld, ys, t0, n0, tv, warp, lane);
      // accumulator b may take the next tile
      tc_fence_before();
      asm volatile("bar.sync %0, 128;" ::"r"(kEpiBarrier) : "memory");
      if (et == 0) mbar_arrive(&acce_bar[b]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kWideTmemCols);
  }
}

}  // namespace epi

namespace epi {

// Host side: the persistent wide-tile launch, or EPILORA_ERR_UNSUPPORTED for
// shapes it does not take (the caller then uses the two-CTAs-per-SM kernel).
// tiles per SM below which the two-CTAs-per-SM kernel is used instead
constexpr int kWideMinTilesPerSm = 4;

template <int KS>
int launch_gemm_wide_ks(GemmParams& p, const GemmArgs& a, int tiles, int sms) {
  using C = GemmCfg<EPILORA_FMT_FP8_E4M3, kWideBT, 1>;
  const int s_bytes = KS > 0 ? (kWideBT * (a.r + 4) * 4 + 127) / 128 * 128 : 0;
  constexpr int kYBytes = 4 * 16 * 40 * 2;
  constexpr int kMisc = 4096;
  int stages = (227 * 1024 - 1024 - s_bytes - kYBytes - kMisc) / C::kStageBytes;
  if (stages > 8) stages = 8;
  if (stages < 2) return EPILORA_ERR_UNSUPPORTED;
  p.stages = stages;
  p.y_stage = stages * C::kStageBytes + s_bytes;
  const int smem = 1024 + p.y_stage + kYBytes + kMisc;
  auto kern = gemm_wide_kernel<KS>;
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
  cfg.gridDim = dim3(tiles < sms ? tiles : sms, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attrs[1];
  int na = 0;
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
int launch_gemm_wide(const GemmArgs& a) {
  if (FMT != EPILORA_FMT_FP8_E4M3 || a.M <= 128) return EPILORA_ERR_UNSUPPORTED;
  const bool lora = a.S != nullptr && a.r > 0;
  if (lora && a.yadd == nullptr && (a.r != 16 && a.r != 32 && a.r != 64)) return EPILORA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(a.Y) & 15) != 0 || a.ldy % 8 != 0) return EPILORA_ERR_UNSUPPORTED;
  const int sms = num_sms();
  const int n_tiles = (a.N + kTileN - 1) / kTileN;
  const int t_tiles = (a.M + kWideBT - 1) / kWideBT;
  const long tiles = static_cast<long>(n_tiles) * t_tiles;
  // a tile or two per SM: nothing to overlap
  if (tiles <= static_cast<long>(sms) * kWideMinTilesPerSm || tiles <= sms || tiles > (1L << 30))
    return EPILORA_ERR_UNSUPPORTED;

  GemmParams p{};
  p.x_scale = a.x_scale;
  p.w_scale = a.w_scale;
  p.S = lora ? a.S : nullptr;
  p.B = static_cast<const __nv_bfloat16*>(a.B);
  p.idx = a.idx;
  p.mask = a.mask;
  p.Y = static_cast<__nv_bfloat16*>(a.Y);
  p.status = a.status_dev;
  p.fused = a.fused;
  p.pdl = !a.fused && a.pdl_dependent ? 1 : 0;
  p.perm = a.perm;
  p.yadd = lora ? a.yadd : nullptr;
  p.s_parts = a.s_parts < 1 ? 1 : a.s_parts;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.L = a.L;
  p.r = lora ? a.r : 0;
  p.s_row = a.s_row > 0 ? a.s_row : p.r;
  p.n_slices = a.n_slices < 1 ? 1 : a.n_slices;
  for (int q = 0; q < 4; ++q) p.slice_end[q] = a.slice_end[q];
  p.ldy = a.ldy;
  p.num_kb = (a.K + kAtomBytes - 1) / kAtomBytes;
  p.ks = 1;
  p.t_tiles = t_tiles;
  p.n_tiles = n_tiles;
  int rc = make_tma_2d_u8(&p.tmW, a.Wq, a.N, a.K, a.K, kTileN, kAtomBytes, true);
  if (rc != EPILORA_OK) return rc;
  rc = make_tma_2d_u8(&p.tmX, a.Xq, a.M, a.K, a.K, kWideBT, kAtomBytes, true);
  if (rc != EPILORA_OK) return rc;
  if (p.yadd != nullptr) return launch_gemm_wide_ks<-1>(p, a, static_cast<int>(tiles), sms);
  switch (p.r) {
    case 0: return launch_gemm_wide_ks<0>(p, a, static_cast<int>(tiles), sms);
    case 16: return launch_gemm_wide_ks<2>(p, a, static_cast<int>(tiles), sms);
    case 32: return launch_gemm_wide_ks<4>(p, a, static_cast<int>(tiles), sms);
    default: return launch_gemm_wide_ks<8>(p, a, static_cast<int>(tiles), sms);
  }
}

}  // namespace epi
