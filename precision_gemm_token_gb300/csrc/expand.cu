// Adapter term of a batch of more than 32 tokens as a pass of its own:
//   Yadd[row][n] = S[perm[row]] . B[l][n]   for every sorted row whose token
//                                            carries an adapter l (mask on)
// in fp32, read back by the GEMM's epilogue (Y = bf16(base + Yadd)).
//
// EpiLoRA, "Fusing Many LoRA Adapters into Low-Precision GEMMs for Serving and
// RL": §Design › Timed dispatch (above the decode batch sizes the adapter term
// is added by EpiLoRA's own adapter kernels after the base GEMM) and the
// appendix "Why EpiLoRA's adapter kernels win on these projections" (the
// expand-add tiles the concatenated output, each tile inside one slice, with
// the slice boundaries passed as kernel arguments). Here the term is not
// added to a bf16 output in place but handed to the GEMM in fp32, so that the
// output is rounded once, exactly as when the epilogue computes the term.
//
// Work item: one weight tile of 128 output columns and a range of at most 256
// adapter-sorted rows. The item's adapter per row is staged once and cut into
// segments (runs of one adapter, also cut every 64 rows (32 at rank 128),
// where a round of S rows is staged in shared memory). Each of the 8 warps owns 16 output
// columns: the 16 B rows of every adapter run that they use stream through
// the warp's own ring in shared memory with 16-byte asynchronous copies
// issued one to three runs ahead (no CTA-wide barrier per run). Per run the
// warp loads the A fragments of its B rows once, then per 8 tokens of the
// segment runs one bf16 m16n8k16 MMA per k-step of 16 and per part of S, S
// being split into three bf16 parts (hi + mid + lo == S exactly): every
// product is exact and the sum is accumulated in fp32, the precision the
// epilogue's own term has.
#include "common.cuh"
#include "ptx.cuh"

namespace epi {

namespace {

constexpr int kExpandThreads = 256;   // 8 warps of 16 output columns
constexpr int kExpandMinRows = 16;    // smallest row range of a work item
constexpr int kExpandItemRows = 256;  // largest row range of a work item
constexpr int kExpandItemCost = 16;   // set-up of a work item, in rows' worth of time

// Rings of B rows in shared memory, one per warp (the 16 rows of one
// adapter's B slice that the warp's columns use, per slot), filled by the
// warp's own 16-byte asynchronous copies kDepth - 1 adapter runs ahead, so
// that a warp waits for nothing but its own copies; 16-byte unit u of row n
// sits at unit u ^ (n & kSwMask) of its row, so that the rows a fragment load
// reads fall into different banks.
template <int R4>
struct ExpandCfg {
  static constexpr int kRowBytes = 8 * R4;                  // r = 4 R4 bf16 values
  static constexpr int kUnits = kRowBytes / 16;
  static constexpr int kSwMask = kUnits - 1 < 7 ? kUnits - 1 : 7;
  static constexpr int kSlotBytes = 16 * kRowBytes;        // one warp's rows of a slice
  static constexpr int kDepth = R4 >= 16 ? 2 : 4;
  static constexpr int kCtas = R4 >= 32 ? 2 : 3;            // resident CTAs per SM
  static constexpr int kRingBytes = 8 * kDepth * kSlotBytes;   // 8 warps
  // sorted rows whose S is staged per round (rank 128: 32, so that the
  // static shared memory stays within 48 KB)
  static constexpr int kRows = R4 >= 32 ? 32 : 64;
  // S rows of a round as three bf16 planes (hi, mid, lo), rows padded by 16
  // bytes so that the 8 token rows of an MMA fragment fall into different banks
  static constexpr int kSRowBytes = kRowBytes + 16;
  static constexpr int kSPlaneBytes = kRows * kSRowBytes;
};

struct ExpandParams {
  const float* S;        // [s_parts][M][s_row], rows by token
  const uint8_t* B;      // bf16 [L][N][r]
  const int32_t* perm;   // sorted row -> token (null: identity)
  const int32_t* idx;
  const uint8_t* mask;
  float* yadd;           // [M][N], rows in sorted order
  int* status;
  int M, N, L, r;
  int s_row, s_parts, n_slices;
  int slice_end[4];
  int n_tiles, row_groups, rows_per_group;
};

__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// fp32 -> three bf16 parts with x == hi + mid + lo exactly (8 + 8 + 8
// significant bits; each residual is exact in fp32)
__device__ __forceinline__ void split3_bf16(float x, uint16_t& hi, uint16_t& mid, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h);
  const __nv_bfloat16 m = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(m);
  const __nv_bfloat16 l = __float2bfloat16_rn(r2);
  hi = __bfloat16_as_ushort(h);
  mid = __bfloat16_as_ushort(m);
  lo = __bfloat16_as_ushort(l);
}

template <int R4>
__global__ void __launch_bounds__(kExpandThreads, ExpandCfg<R4>::kCtas)
    expand_kernel(const __grid_constant__ ExpandParams p) {
  using C = ExpandCfg<R4>;
  extern __shared__ __align__(16) uint8_t ring[];
  __shared__ __align__(16) uint8_t s_planes[3 * C::kSPlaneBytes];   // S of the round: hi, mid, lo
  __shared__ int meta_l[kExpandItemRows];
  __shared__ int meta_tok[kExpandItemRows];
  __shared__ int seg_start[kExpandItemRows + 1];
  __shared__ int seg_load[kExpandItemRows];     // B slice (load) a segment uses, -1: none
  __shared__ int load_l[kExpandItemRows];       // adapter of each load, in order
  __shared__ int nseg_s, nload_s;
  // the GEMM that reads Yadd may become resident at once (it streams its
  // weights and waits for this grid before its epilogue); S, perm and the
  // token metadata are read only once the shrink grid has completed
  pdl_allow_dependents();
  pdl_wait_primary();
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;    // output columns 16 warp .. 16 warp + 15 of the tile
  const int g = lane >> 2, tq = lane & 3;   // MMA fragment coordinates
  const int items = p.n_tiles * p.row_groups;
  const size_t part = static_cast<size_t>(p.M) * p.s_row / 4;   // float4s per partial array of S
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int nt = item / p.row_groups;
    const int rg = item - nt * p.row_groups;
    const int n0 = nt * 128;
    const int r0 = rg * p.rows_per_group;
    const int nrows = min(p.M, r0 + p.rows_per_group) - r0;
    // rank-r block of the S rows that this weight tile's slice reads
    int soff = 0;
    for (int q = 0; q + 1 < p.n_slices && q < 4; ++q)
      if (n0 >= p.slice_end[q]) soff += p.r;
    __syncthreads();   // the previous item's tables and ring slots are consumed
    // adapter of every row of the item (-1: none), and its token
    for (int i = tid; i < nrows; i += kExpandThreads) {
      const int row = r0 + i;
      const int tok = p.perm != nullptr ? p.perm[row] : row;
      const int li = p.idx[tok];
      const bool on = li >= 0 && li < p.L && (p.mask == nullptr || p.mask[tok] != 0);
      if (li >= p.L) record_status(p.status, EPILORA_ERR_INVALID_ARG);
      meta_l[i] = on ? li : -1;
      meta_tok[i] = tok;
    }
    __syncthreads();
    // segments: runs of one adapter (or of none), also cut where a round of
    // kRows rows starts; one B slice load per run with an adapter
    if (tid < 32) {
      int ns = 0, nl = 0;
      for (int base = 0; base < nrows; base += 32) {
        const int i = base + lane;
        const int l = i < nrows ? meta_l[i] : -1;
        const bool run = i < nrows && (i == 0 || meta_l[i - 1] != l);
        const bool st = run || (i < nrows && i % C::kRows == 0);
        const bool ld = run && l >= 0;
        const unsigned below = (1u << lane) - 1u;
        const unsigned smsk = __ballot_sync(0xffffffffu, st);
        const unsigned lmsk = __ballot_sync(0xffffffffu, ld);
        const int loads_to_here = nl + __popc(lmsk & below) + (ld ? 1 : 0);   // loads started at rows <= i
        if (st) {
          const int k = ns + __popc(smsk & below);
          seg_start[k] = i;
          seg_load[k] = l >= 0 ? loads_to_here - 1 : -1;
        }
        if (ld) load_l[nl + __popc(lmsk & below)] = l;
        ns += __popc(smsk);
        nl += __popc(lmsk);
      }
      if (lane == 0) {
        seg_start[ns] = nrows;
        nseg_s = ns;
        nload_s = nl;
      }
    }
    __syncthreads();
    const int nseg = nseg_s;
    const int nload = nload_s;
    // this warp's 16 rows of B slice j into its ring slot j % kDepth (rows
    // past N zero-filled); one commit group per call, empty past the last load
    uint8_t* wring = ring + warp * C::kDepth * C::kSlotBytes;
    auto issue_load = [&](int j) {
      if (j < nload) {
        uint8_t* slot = wring + (j % C::kDepth) * C::kSlotBytes;
        const int nw = n0 + warp * 16;
        const uint8_t* src = p.B + (static_cast<size_t>(load_l[j]) * p.N + nw) * C::kRowBytes;
        for (int e = lane; e < 16 * C::kUnits; e += 32) {
          const int row = e / C::kUnits;
          const int u = e - row * C::kUnits;
          const bool ok = nw + row < p.N;
          cp_async_16(slot + row * C::kRowBytes + ((u ^ (row & C::kSwMask)) << 4),
                      ok ? src + row * C::kRowBytes + (u << 4) : p.B, ok ? 16 : 0);
        }
      }
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < C::kDepth - 1; ++j) issue_load(j);
    constexpr int kKSteps = R4 / 4;   // k-steps of 16 in the rank
    uint32_t af[kKSteps][4];          // A fragments of the current adapter run
    int cur_j = -1;
    int k = 0;
    for (int c0 = 0; c0 < nrows; c0 += C::kRows) {
      const int nr = min(C::kRows, nrows - c0);
      __syncthreads();   // the previous round's rows are consumed
      // S rows of the round's active tokens (partial sums added in part
      // order), split into the three bf16 planes
      for (int e = tid; e < nr * R4; e += kExpandThreads) {
        const int i = e / R4;
        const int c = e - i * R4;
        if (meta_l[c0 + i] < 0) continue;
        const float4* src =
            reinterpret_cast<const float4*>(p.S + static_cast<size_t>(meta_tok[c0 + i]) * p.s_row + soff) + c;
        float4 v = __ldcg(src);
        for (int q = 1; q < p.s_parts; ++q) {
          const float4 w = __ldcg(src + q * part);
          v.x += w.x;
          v.y += w.y;
          v.z += w.z;
          v.w += w.w;
        }
        uint16_t hx, hy, hz, hw, mx, my, mz, mw, lx, ly, lz, lw;
        split3_bf16(v.x, hx, mx, lx);
        split3_bf16(v.y, hy, my, ly);
        split3_bf16(v.z, hz, mz, lz);
        split3_bf16(v.w, hw, mw, lw);
        uint8_t* d = s_planes + i * C::kSRowBytes + c * 8;
        *reinterpret_cast<uint2*>(d) = make_uint2(hx | (uint32_t(hy) << 16), hz | (uint32_t(hw) << 16));
        *reinterpret_cast<uint2*>(d + C::kSPlaneBytes) =
            make_uint2(mx | (uint32_t(my) << 16), mz | (uint32_t(mw) << 16));
        *reinterpret_cast<uint2*>(d + 2 * C::kSPlaneBytes) =
            make_uint2(lx | (uint32_t(ly) << 16), lz | (uint32_t(lw) << 16));
      }
      __syncthreads();
      for (; k < nseg && seg_start[k] < c0 + nr; ++k) {
        const int j = seg_load[k];
        if (j < 0) continue;
        if (j != cur_j) {
          // a new adapter run: every lane of the warp has read slot
          // (j - 1) % kDepth, so it may take load j + kDepth - 1; then the
          // warp's copies of load j are awaited and made visible to its lanes
          __syncwarp();
          issue_load(j + C::kDepth - 1);
          cp_async_wait<C::kDepth - 1>();
          __syncwarp();
          // A fragments of this warp's 16 B rows (rows g and g + 8, ranks
          // 2 tq, 2 tq + 1 and + 8 of each k-step of 16)
          const uint8_t* slot = wring + (j % C::kDepth) * C::kSlotBytes;
#pragma unroll
          for (int ks = 0; ks < kKSteps; ++ks)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int row = g + 8 * (e & 1);
              const int unit = 2 * ks + (e >> 1);
              af[ks][e] = *reinterpret_cast<const uint32_t*>(slot + row * C::kRowBytes +
                                                             ((unit ^ (row & C::kSwMask)) << 4) + 4 * tq);
            }
          cur_j = j;
        }
        const int i = seg_start[k] - c0;
        const int jr = seg_start[k + 1] - c0;
        // Yadd[token t][column n] = sum over the rank of B[n][k] S[t][k]: one
        // m16n8k16 MMA per 8 tokens, k-step and S part (lo, mid, hi). A token
        // column of the MMA depends on that token's S row alone: the columns
        // past the segment (other rows of the round, or none) are computed
        // but not stored.
        for (int t0 = i; t0 < jr; t0 += 8) {
          const int t = min(t0 + g, C::kRows - 1);
          float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int ks = 0; ks < kKSteps; ++ks)
#pragma unroll
            for (int part = 2; part >= 0; --part) {
              const uint8_t* sp = s_planes + part * C::kSPlaneBytes + t * C::kSRowBytes + (16 * ks + 2 * tq) * 2;
              const uint32_t b0 = *reinterpret_cast<const uint32_t*>(sp);
              const uint32_t b1 = *reinterpret_cast<const uint32_t*>(sp + 16);
              mma_bf16_m16n8k16(acc, af[ks], b0, b1);
            }
          // c0: (column g, token 2 tq), c1: (g, 2 tq + 1), c2/c3: column g + 8
          const int ta = t0 + 2 * tq;
          const int na = n0 + warp * 16 + g;
          float* out = p.yadd + static_cast<size_t>(r0 + c0) * p.N;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int te = ta + (e & 1);
            const int ne = na + 8 * (e >> 1);
            if (te < jr && ne < p.N) out[static_cast<size_t>(te) * p.N + ne] = acc[e];
          }
        }
      }
    }
    cp_async_wait<0>();   // no copy of this item outlives it
  }
}

template <int R4>
cudaError_t launch_expand_r(const ExpandParams& p, cudaLaunchConfig_t cfg) {
  using C = ExpandCfg<R4>;
  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    const cudaError_t rc =
        cudaFuncSetAttribute(expand_kernel<R4>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kRingBytes);
    if (rc != cudaSuccess) return rc;
    attr_done[dev] = 1;
  }
  const long items = static_cast<long>(p.n_tiles) * p.row_groups;
  const long slots = static_cast<long>(num_sms()) * C::kCtas;
  cfg.gridDim = dim3(static_cast<unsigned>(items < slots ? items : slots), 1, 1);
  cfg.dynamicSmemBytes = C::kRingBytes;
  return cudaLaunchKernelEx(&cfg, expand_kernel<R4>, p);
}

}  // namespace

size_t expand_yadd_bytes(int M, int N) {
  return M > 0 && N > 0 ? (static_cast<size_t>(M) * N * 4 + 255) / 256 * 256 : 0;
}

int launch_expand(const ExpandArgs& a) {
  if (a.M <= 0 || a.N <= 0) return EPILORA_OK;
  if (a.S == nullptr || a.B == nullptr || a.idx == nullptr || a.yadd == nullptr) return EPILORA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a.S) & 15) != 0 || (reinterpret_cast<uintptr_t>(a.B) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(a.yadd) & 3) != 0 || a.s_row % 4 != 0)
    return EPILORA_ERR_INVALID_ARG;
  if (a.r != 16 && a.r != 32 && a.r != 64 && a.r != 128) return EPILORA_ERR_INVALID_ARG;
  ExpandParams p{};
  p.S = a.S;
  p.B = static_cast<const uint8_t*>(a.B);
  p.perm = a.perm;
  p.idx = a.idx;
  p.mask = a.mask;
  p.yadd = a.yadd;
  p.status = a.status_dev;
  p.M = a.M;
  p.N = a.N;
  p.L = a.L;
  p.r = a.r;
  p.s_row = a.s_row > 0 ? a.s_row : a.r;
  p.s_parts = a.s_parts < 1 ? 1 : a.s_parts;
  p.n_slices = a.n_slices < 1 ? 1 : a.n_slices;
  for (int q = 0; q < 4; ++q) p.slice_end[q] = a.slice_end[q];
  p.n_tiles = (a.N + 127) / 128;
  // row groups per weight tile, items of kExpandMinRows to kExpandItemRows
  // rows: the count that minimises (waves of items over the grid's CTA
  // slots) x (rows per item + a fixed cost per item, counted in rows), fewer
  // items on a tie (each item reads its runs' B slices once)
  const int ctas = a.r >= 128 ? ExpandCfg<32>::kCtas
                   : a.r >= 64 ? ExpandCfg<16>::kCtas
                   : a.r >= 32 ? ExpandCfg<8>::kCtas
                               : ExpandCfg<4>::kCtas;
  const long slots = static_cast<long>(num_sms()) * ctas;
  int max_groups = (a.M + kExpandMinRows - 1) / kExpandMinRows;
  int min_groups = (a.M + kExpandItemRows - 1) / kExpandItemRows;
  if (min_groups < 1) min_groups = 1;
  if (max_groups < min_groups) max_groups = min_groups;
  int groups = min_groups;
  long best = -1;
  for (int g = min_groups; g <= max_groups; ++g) {
    const long rows = (a.M + g - 1) / g;
    const long items = static_cast<long>(p.n_tiles) * ((a.M + rows - 1) / rows);
    const long cost = (items + slots - 1) / slots * (rows + kExpandItemCost);
    if (best < 0 || cost < best) {
      best = cost;
      groups = g;
    }
  }
  p.rows_per_group = (a.M + groups - 1) / groups;
  p.row_groups = (a.M + p.rows_per_group - 1) / p.rows_per_group;

  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kExpandThreads, 1, 1);
  cfg.stream = a.stream;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = a.pdl_dependent ? 1 : 0;
  cudaError_t rc;
  switch (a.r) {
    case 16: rc = launch_expand_r<4>(p, cfg); break;
    case 32: rc = launch_expand_r<8>(p, cfg); break;
    case 64: rc = launch_expand_r<16>(p, cfg); break;
    default: rc = launch_expand_r<32>(p, cfg); break;
  }
  return rc == cudaSuccess ? EPILORA_OK : EPILORA_ERR_CUDA;
}

}  // namespace epi
