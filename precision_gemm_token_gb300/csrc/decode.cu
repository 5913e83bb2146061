// Single-kernel decode path: the whole multi-tenant LoRA layer of a few decode
// tokens in ONE launch per projection.
//
// EpiLoRA, "Fusing Many LoRA Adapters into Low-Precision GEMMs for Serving and
// RL":
//  * §Design › Multi-adapter kernels › K1 and K2 — activations quantized once
//    per token, h = x A^T from the bf16 activations, the GEMM epilogue applies
//    the weight and activation scales and adds h B^T before Y is written once;
//  * › The decode path — the GEMM streams its weights while the
//    down-projection runs and needs h only before its epilogue; the page does
//    this with two launches chained by programmatic dependent launch and
//    counts the second launch and its hand-off in "exposed + launch"
//    (§Evaluation › Kernels, Table 13); here both are one kernel.
//
// GB300 design: one persistent CTA per SM (about 113 KB of shared memory, so
// the next projection's CTA fits beside it and streams its weights while this
// one finishes). The weight matrix is cut into units (128 rows x 256 bytes of
// K, 32 KB of codes) in tile-major order and every CTA takes an equal
// contiguous run of units (stream-K), so no SM streams more than its share.
// Roles (192 threads):
//   warp 0      TMA producer: the CTA's weight units (and NVFP4 weight scale
//               boxes) through a ring, started before the dependency wait
//               (weights are never written by the preceding kernel), L2
//               hints (activations first, adapter rows behind the first
//               units);
//   warp 1      MMA issuer: tcgen05.mma (kind::f8f6f4, or kind::mxf4nvf4 with
//               scales copied into TMEM) into one of two TMEM accumulators
//               (one per segment of the run that falls in one weight tile),
//               the activations read in place from the compact quantized
//               copy (a no-swizzle operand whose core matrices are M x 16
//               bytes apart along K);
//   warps 2..5  helpers: the dependency wait (griddepcontrol.wait), one
//               bulk copy of the bf16 activation rows into the last ring
//               slots, quantization of every token into shared memory (each
//               CTA for itself: FP8 divisions by Markstein's correction of
//               the reciprocal product; each CTA encodes the K range of its
//               own units),
//               shrink work items (token x 4 ranks x K slice, the arithmetic
//               of the standalone shrink; CTA c takes items c, c + G, ...),
//               then the epilogue of each segment.
// A weight tile split over several CTAs is finished by the CTA that holds its
// first K unit (it reaches that tile last): the others store their fp32
// partial rows, and the shrink items their partial sums of S, each value in a
// 64-bit word with this launch's tag; the finisher reads them until the tags
// match (all of a row's words requested at once), adds the partial rows in
// CTA order and S's slices in part order (deterministic), applies the scales,
// adds the adapter term and writes Y. The tag comes from a launch counter in
// the workspace to which every launch adds 256 in all as its CTAs exit (one
// reduction each, nothing waited for), so a launch reads 256 j plus less
// than 256 and takes j as its epoch. Every wait is bounded (an error status,
// then an orderly exit) and waits only on work of running CTAs. The next
// kernel on the stream is released as soon as every CTA has started: it
// streams its first weight units while this one works and waits for this
// grid's completion before it reads anything else.
#include "quant_row.cuh"

namespace epi {

namespace {

constexpr int kDecThreads = 192;
constexpr int kDecMaxTokens = 8;
constexpr int kDecMaxCtas = 256;
constexpr int kDecXcBytes = 16384;         // compact quantized activations per CTA
constexpr int kDecRanksPerItem = 4;
constexpr int kDecHelperBar = 1;           // named barrier of the 4 helper warps
constexpr int kDecAtomW = 128 * 128;       // weight codes of one 128-byte K atom of a tile (bytes)
constexpr int kDecSmemBudget = 113 * 1024;
constexpr int kDecMaxStages = 8;
constexpr int kMaxRankBrow = 64;           // 32-bit words of a rank-128 bf16 B row

// sync block at the start of the workspace: words [4, 6) hold the 64-bit
// launch counter; then the tagged region (partial rows, then S)
constexpr int kDecSyncWords = 64;
constexpr int kDecCounterWord = 4;
constexpr int kDecSParts = 8;              // K slices of the shrink at most
constexpr int kDecMaxSRow = 512;           // rank 128 x 4 slices

struct DecParams {
  CUtensorMap tmW;     // uint8 [N, Kb], box 128 rows x 128 B, 128-B swizzle
  CUtensorMap tmSW;    // NVFP4: uint8 [N, K/16], box 128 rows x 16 B
  const __nv_bfloat16* X;
  const __nv_bfloat16* A;
  const __nv_bfloat16* B;
  // stored FP8 adapters: A and B hold E4M3 codes ([L, s_row, K] and [L, N, r]
  // bytes) with one fp32 scale per row; null: bf16 tables
  const float* a_scale;
  const float* b_scale;
  const int32_t* idx;
  const uint8_t* mask;
  const float* w_scale;
  const float* w_gs;
  const float* x_gs;
  __nv_bfloat16* Y;
  int* status;
  unsigned long long* counter;   // launch counter (256 per launch)
  // Published values carry the launch epoch in the same 64-bit word (value
  // bits low, epoch high): a reader retries until the tag is this launch's,
  // so no flag or counter has to be polled before the data.
  uint2* S;            // [parts][M][s_row] partial sums of the shrink
  uint2* accp;         // [G][M][128] partial rows of split weight tiles
  uint8_t* xq_out;     // the quantized activations also go here (each code by one CTA)
  float* xs_out;       // FP8 scales
  uint8_t* xsb_out;    // NVFP4 block scales
  long long U;         // units in total
  int G, nkb, n_tiles, stages;
  int M, N, K, ldx, ldy, L, r, s_row, n_slices;
  int slice_end[4];
  int adapters, parts, kslice, n_items;
  int drop_s;          // test hook: the shrink items publish nothing (finishers time out)
  int kb_pad;          // code bytes of one token's row, padded to whole units
  int xslots;          // last ring slots that first hold the bf16 activation rows
};

// A unit is KA 128-byte K atoms of one 128-row weight tile (16 KB each).
template <int FMT, int KA>
struct DecCfg {
  static constexpr bool kFP4 = FMT == EPILORA_FMT_NVFP4;
  static constexpr int kKSteps = 4 * KA;                    // MMAs per unit (32 bytes of K each)
  static constexpr int kUnitW = KA * kDecAtomW;
  static constexpr int kSfA = kFP4 ? kKSteps * 512 : 0;     // weight scales re-laid for tcgen05.cp
  static constexpr int kSfWRaw = kFP4 ? 128 * 16 * KA : 0;  // TMA box of weight scales [128][16 KA]
  static constexpr int kStageRaw = kUnitW + kSfA + kSfWRaw;
  static constexpr int kStage = (kStageRaw + 1023) / 1024 * 1024;
  static constexpr int kStageTx = kUnitW + kSfWRaw;         // bytes TMA delivers per stage
  static constexpr int kSfCols = 4 * kKSteps;               // TMEM columns of one scale slot (A or B)
  static constexpr int kSfSlot = 2 * kSfCols;
  static constexpr int kTmemNeed = 32 + (kFP4 ? 2 * kSfSlot : 0);   // 2 accumulators of 16 (+ 2 scale slots)
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128 : 256;
  static constexpr uint32_t kIdesc = kFP4 ? idesc_mxf4nvf4(128, 16) : idesc_f8f6f4_e4m3(128, 16);
};

__device__ __forceinline__ void helper_sync() {
  asm volatile("bar.sync %0, 128;" ::"r"(kDecHelperBar) : "memory");
}

// OR of a flag over the 4 helper warps (also a barrier among them)
__device__ __forceinline__ bool helper_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(kDecHelperBar)
      : "memory");
  return r != 0;
}

// Tag of the launch with epoch e: odd (never the zero of fresh memory) and
// distinct for epochs less than 2^31 apart.
__device__ __forceinline__ unsigned launch_tag(unsigned long long e) {
  return (static_cast<unsigned>(e) << 1) | 1u;
}

// One tagged 64-bit value, read again until its tag is `epoch` (1 s limit;
// on timeout the last word read, whose tag is then another). `w` holds a
// first read already made.
// n <= N tagged values p[0], p[stride], ... whose first reads are in w:
// the late ones are read again, all of them in each round (one round trip
// per round however many are late), until every tag is this launch's or
// the wait limit has passed. The values go to v[0..n); false on a timeout.
template <int N>
__device__ __forceinline__ bool check_tagged_n(const uint2* p, size_t stride, int n, unsigned epoch, uint2 (&w)[N],
                                               float (&v)[N]) {
  auto all_here = [&]() {
    bool ok = true;
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (i < n && w[i].y != epoch) ok = false;
    return ok;
  };
  bool ok = all_here();
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      __nanosleep(32);
#pragma unroll
      for (int i = 0; i < N; ++i)
        if (i < n && w[i].y != epoch) w[i] = __ldcg(p + i * stride);
      ok = all_here();
      if (ok || globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  }
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (i < n) v[i] = __uint_as_float(w[i].x);
  return ok;
}

// First reads of n <= N tagged values p[0], p[stride], ..., all issued before
// any is used (one round trip when they are all there).
template <int N>
__device__ __forceinline__ void load_tagged_n(const uint2* p, size_t stride, int n, uint2 (&w)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (i < n) w[i] = __ldcg(p + i * stride);
}

// |x| max of a 16-byte chunk of 8 bf16 values as a bf16 pair (the max of
// bf16 magnitudes is one of them: exact).
__device__ __forceinline__ __nv_bfloat162 absmax8_bf16(const uint4& v) {
  const __nv_bfloat162 a = __hmax2(__habs2(*reinterpret_cast<const __nv_bfloat162*>(&v.x)),
                                   __habs2(*reinterpret_cast<const __nv_bfloat162*>(&v.y)));
  const __nv_bfloat162 b = __hmax2(__habs2(*reinterpret_cast<const __nv_bfloat162*>(&v.z)),
                                   __habs2(*reinterpret_cast<const __nv_bfloat162*>(&v.w)));
  return __hmax2(a, b);
}

__device__ __forceinline__ float dec_dot8(const uint4& xv, const uint4& av, float acc) {
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

// x / s rounded to nearest float, from rs = 1/s rounded to nearest: P.
// Markstein's correction of the reciprocal product ("Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990; also Muller et al., Handbook of Floating-Point Arithmetic, the
// theorem on division by FMA): q0 = RN(x rs) is within one ulp of x / s, the
// residual x - q0 s is then exact in one fma, and RN(q0 + residual rs) is the
// correctly rounded quotient, provided the residual does not underflow.
// Callers keep |x / s| <= 448 and s >= 2^-100, so the residual is a normal
// number or x / s is far below the smallest E4M3 subnormal.
__device__ __forceinline__ float div_rn_by_recip(float x, float s, float rs) {
  const float q0 = __fmul_rn(x, rs);
  const float e = __fmaf_rn(-q0, s, x);
  return __fmaf_rn(e, rs, q0);
}

// E4M3 codes of 8 bf16 values divided by the row scale s (rs = 1/s rounded
// to nearest); for scales of at least 2^-100 (callers take the IEEE division
// below that).
__device__ __forceinline__ uint2 quant8_e4m3_rs(const uint4& v, float s, float rs) {
  float x[8];
  unpack8(v, x);
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    q[i] = cvt_e4m3x2(div_rn_by_recip(x[2 * i], s, rs), div_rn_by_recip(x[2 * i + 1], s, rs));
  return make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

// S[v] . B[l, n] with the B row in registers (R4 float4 chunks of S from
// shared memory; two accumulators)
// Two E4M3 codes (the low 16 bits of c, low byte first) as floats.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t c) {
  uint32_t h2;
  const uint16_t c16 = static_cast<uint16_t>(c & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c16));
  __half2_raw hr;
  hr.x = static_cast<unsigned short>(h2 & 0xFFFFu);
  hr.y = static_cast<unsigned short>(h2 >> 16);
  return __half22float2(__half2(hr));
}

// x (8 bf16) . a (8 E4M3 codes), accumulated into acc in element order
__device__ __forceinline__ float dec_dot8_e4m3(const uint4& xv, const uint2& av, float acc) {
  const float2 a01 = e4m3x2_to_f32x2(av.x), a23 = e4m3x2_to_f32x2(av.x >> 16);
  const float2 a45 = e4m3x2_to_f32x2(av.y), a67 = e4m3x2_to_f32x2(av.y >> 16);
  acc = fmaf(bf16_lo(xv.x), a01.x, acc);
  acc = fmaf(bf16_hi(xv.x), a01.y, acc);
  acc = fmaf(bf16_lo(xv.y), a23.x, acc);
  acc = fmaf(bf16_hi(xv.y), a23.y, acc);
  acc = fmaf(bf16_lo(xv.z), a45.x, acc);
  acc = fmaf(bf16_hi(xv.z), a45.y, acc);
  acc = fmaf(bf16_lo(xv.w), a67.x, acc);
  acc = fmaf(bf16_hi(xv.w), a67.y, acc);
  return acc;
}

// S[v] . codes of an E4M3 B row held 4 per 32-bit word (R4 float4 chunks)
template <int R4>
__device__ __forceinline__ float dec_dot_row_e4m3(const float4* srow, const uint32_t* brow) {
  float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
  for (int c = 0; c < R4; ++c) {
    const float4 s4 = srow[c];
    const float2 lo = e4m3x2_to_f32x2(brow[c]), hi = e4m3x2_to_f32x2(brow[c] >> 16);
    float& d = (c & 1) ? d1 : d0;
    d = fmaf(s4.x, lo.x, d);
    d = fmaf(s4.y, lo.y, d);
    d = fmaf(s4.z, hi.x, d);
    d = fmaf(s4.w, hi.y, d);
  }
  return d0 + d1;
}

template <int R4>
__device__ __forceinline__ float dec_dot_row(const float4* srow, const uint32_t* brow) {
  float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
  for (int c = 0; c < R4; ++c) {
    const float4 s4 = srow[c];
    float& d = (c & 1) ? d1 : d0;
    d = fmaf(s4.x, bf16_lo(brow[2 * c]), d);
    d = fmaf(s4.y, bf16_hi(brow[2 * c]), d);
    d = fmaf(s4.z, bf16_lo(brow[2 * c + 1]), d);
    d = fmaf(s4.w, bf16_hi(brow[2 * c + 1]), d);
  }
  return d0 + d1;
}

// Run of units of CTA c: [U c / G, U (c + 1) / G), walked as segments that
// each lie in one weight tile.
struct SegWalk {
  long long u, u1;
  int nkb;
  __device__ SegWalk(const DecParams& p, int c)
      : u((p.U * c) / p.G), u1((p.U * (c + 1)) / p.G), nkb(p.nkb) {}
  __device__ bool next(int& T, int& kb0, int& kb1) {
    if (u >= u1) return false;
    T = static_cast<int>(u / nkb);
    kb0 = static_cast<int>(u - static_cast<long long>(T) * nkb);
    const long long left = u1 - u;
    kb1 = left < nkb - kb0 ? kb0 + static_cast<int>(left) : nkb;
    u += kb1 - kb0;
    return true;
  }
};

// CTA whose run holds unit u
__device__ __forceinline__ int cta_of_unit(const DecParams& p, long long u) {
  return static_cast<int>(((u + 1) * p.G + p.U - 1) / p.U) - 1;
}

__device__ __forceinline__ int dec_slice_offset(const DecParams& p, int n0) {
  int off = 0;
  for (int q = 0; q + 1 < p.n_slices && q < 4; ++q)
    if (n0 >= p.slice_end[q]) off += p.r;
  return off;
}

template <int FMT, int KA>
__global__ void __launch_bounds__(kDecThreads, 2) fused_decode_kernel(const __grid_constant__ DecParams p) {
  using C = DecCfg<FMT, KA>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stages = p.stages;
  const int M = p.M;
  // Quantized activations, chunk-major: 16-byte K chunk j of token t at
  // (j * M + t) * 16. The MMA reads them in place as its B operand (K-major,
  // no swizzle, core matrices M * 16 bytes apart along K: rows t < M are the
  // tokens, the other rows of a core matrix fall on the next chunk and only
  // feed output columns that are never read), + 128 bytes of slack.
  uint8_t* xc = smem + static_cast<size_t>(stages) * C::kStage;
  // NVFP4 token block scales, one 16-byte line per (MMA k-step s, token t) at
  // (s * M + t) * 16 holding the token's 4 scales of that k-step: read in
  // place by tcgen05.cp, + 512 bytes of slack
  uint8_t* xsf = xc + M * p.kb_pad + 128;
  const int xsf_bytes = C::kFP4 ? (M * (p.kb_pad / 32) * 16 + 512 + 127) / 128 * 128 : 0;
  float* s_stage = reinterpret_cast<float*>(xsf + xsf_bytes);
  float* yacc = s_stage + (M * p.s_row + 31) / 32 * 32;             // [M][128] a finisher's row sums
  uint8_t* misc = reinterpret_cast<uint8_t*>(yacc + M * 128);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(misc);
  uint64_t* empty_bar = full_bar + kDecMaxStages;
  uint64_t* accf_bar = empty_bar + kDecMaxStages;    // [2] accumulator complete
  uint64_t* acce_bar = accf_bar + 2;                 // [2] accumulator read out
  uint64_t* xrdy_bar = acce_bar + 2;                 // compact activations written
  uint64_t* xst_bar = xrdy_bar + 1;                  // the bf16 activation rows have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xst_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);               // [4 warps][8]
  int* meta_idx = reinterpret_cast<int*>(red + 32);                   // [kDecMaxTokens] adapter or -1
  float* meta_sx = reinterpret_cast<float*>(meta_idx + kDecMaxTokens);   // FP8 activation scales
  float* meta_rs = meta_sx + kDecMaxTokens;                           // their reciprocals

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], 1);
    }
    mbar_init(xrdy_bar, 1);
    mbar_init(xst_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&p.tmW);
    if (C::kFP4) tma_prefetch_desc(&p.tmSW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // every CTA of this grid is running: the next kernel on the stream may
  // start its CTAs (they stream weights, never written here, and wait for
  // this grid's completion before they read anything else)
  if (threadIdx.x == 0) pdl_allow_dependents();

  if (warp == 0) {
    // ===== TMA producer: the run's weight units, in order =====
    if (lane == 0) {
      // the activation rows go to L2 first (a hint: the preceding kernel may
      // still be writing them)
      for (int t = 0; t < M; ++t)
        prefetch_l2_bulk(p.X + static_cast<size_t>(t) * p.ldx, static_cast<uint32_t>(p.K * 2));
      uint32_t issued_mask = 0, parity_mask = 0;
      long long it = 0;
      // every weight byte is read once per call: streamed with the first
      // eviction priority, so that the activations, the adapter rows and the
      // exchanged partial sums stay in L2 beside the stream
      const uint64_t wpol = l2_policy_evict_first();
      const long long u_begin = (p.U * c) / p.G, u_end = (p.U * (c + 1)) / p.G;
      for (long long u = u_begin; u < u_end; ++u, ++it) {
        const int s = static_cast<int>(it % stages);
        const uint32_t ph = static_cast<uint32_t>(it / stages) & 1u;
        if (*abort_flag || !mbar_wait_bounded(&empty_bar[s], ph ^ 1u, kWaitLimitNs)) {
          *abort_flag = 1;
          record_status(p.status, EPILORA_ERR_TIMEOUT);
          break;
        }
        // the last xslots slots hold the activation rows until the quantized
        // copy is published; meanwhile, with the first units requested, this
        // CTA's share of the adapters' A rows and the B slices of the tiles
        // it finishes go to L2 (the index read here may still change: hints)
        if (it == stages - p.xslots && p.adapters) {
          const size_t abytes = static_cast<size_t>(p.s_row) * p.K * (p.a_scale != nullptr ? 1 : 2);
          const size_t share = ((abytes + p.G - 1) / p.G + 255) / 256 * 256;
          const size_t lo = share * c;
          int prev = -1;
          for (int t = 0; t < M; ++t) {
            int l;
            asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(l) : "l"(p.idx + t));
            if (l < 0 || l >= p.L || l == prev) continue;
            prev = l;
            if (lo < abytes)
              prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(p.A) + static_cast<size_t>(l) * abytes + lo,
                               static_cast<uint32_t>(min(share, abytes - lo)));
            SegWalk w2(p, c);
            int T2, kb0, kb1;
            while (w2.next(T2, kb0, kb1)) {
              if (kb0 != 0) continue;
              const int rows = min(128, p.N - T2 * 128);
              const int bb = p.a_scale != nullptr ? p.r : 2 * p.r;   // bytes of one B row
              prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(p.B) + (static_cast<size_t>(l) * p.N + T2 * 128) * bb,
                               static_cast<uint32_t>(rows * bb));
            }
          }
        }
        if (it == stages - p.xslots && !mbar_wait_bounded(xrdy_bar, 0, kWaitLimitNs)) {
          *abort_flag = 1;
          record_status(p.status, EPILORA_ERR_TIMEOUT);
          break;
        }
        const int T = static_cast<int>(u / p.nkb);
        const int kb = static_cast<int>(u - static_cast<long long>(T) * p.nkb);
        uint8_t* st = smem + static_cast<size_t>(s) * C::kStage;
        mbar_arrive_expect_tx(&full_bar[s], C::kStageTx);
#pragma unroll
        for (int a = 0; a < KA; ++a)
          tma_load_2d_hint(st + a * kDecAtomW, &p.tmW, &full_bar[s], (kb * KA + a) * 128, T * 128, wpol);
        if (C::kFP4) tma_load_2d_hint(st + C::kUnitW + C::kSfA, &p.tmSW, &full_bar[s], kb * 16 * KA, T * 128, wpol);
        issued_mask |= 1u << s;
        parity_mask = (parity_mask & ~(1u << s)) | (ph << s);
      }
      if (*abort_flag) {
        for (int s = 0; s < stages; ++s)
          if (issued_mask & (1u << s)) (void)mbar_wait_bounded(&full_bar[s], (parity_mask >> s) & 1u, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===== MMA issuer =====
    const uint32_t xc_addr = smem_u32(xc);
    const uint32_t xsf_addr = smem_u32(xsf);
    const uint32_t x_lbo = static_cast<uint32_t>(16 * M);
    SegWalk walk(p, c);
    int T, kb0, kb1, j = 0;
    long long it = 0;
    bool have = walk.next(T, kb0, kb1);           // (the first segment before the wait)
    const bool xok = __all_sync(0xffffffffu, mbar_wait_bounded(xrdy_bar, 0, kWaitLimitNs));
    if (!xok && lane == 0) {
      *abort_flag = 1;
      record_status(p.status, EPILORA_ERR_TIMEOUT);
    }
    bool stop = !xok;
    for (; !stop && have; have = walk.next(T, kb0, kb1)) {
      const int b = j & 1;
      // the helpers have read this accumulator's previous segment
      const bool oke = __all_sync(0xffffffffu, mbar_wait_bounded(&acce_bar[b], ((j >> 1) & 1) ^ 1u, kWaitLimitNs));
      if (!oke || *abort_flag) {
        if (lane == 0) {
          *abort_flag = 1;
          record_status(p.status, EPILORA_ERR_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * 16);
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
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
        uint8_t* st = smem + static_cast<size_t>(s) * C::kStage;
        uint8_t* sfa = st + C::kUnitW;
        if (C::kFP4) {
          // weight scales: canonical [128 rows][16 KA bytes] box -> one 512-B
          // atom per K = 64 step (line r0 = 4 bytes of rows r0, r0+32, r0+64,
          // r0+96), the layout tcgen05.cp .32x128b.warpx4 takes
          const uint8_t* raw_w = sfa + C::kSfA;
#pragma unroll
          for (int a = 0; a < KA; ++a) {
            uint4 v[4];
#pragma unroll
            for (int r1 = 0; r1 < 4; ++r1)
              v[r1] = *reinterpret_cast<const uint4*>(raw_w + (lane + 32 * r1) * (16 * KA) + 16 * a);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              uint4 o;
              o.x = (&v[0].x)[kk];
              o.y = (&v[1].x)[kk];
              o.z = (&v[2].x)[kk];
              o.w = (&v[3].x)[kk];
              *reinterpret_cast<uint4*>(sfa + (a * 4 + kk) * 512 + lane * 16) = o;
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t w_addr = smem_u32(st);
#pragma unroll
          for (int a = 0; a < KA; ++a) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const int jj = a * 4 + kk;                               // k-step within the unit
              const int chunk = (kb * KA + a) * 8 + kk * 2;              // first 16-byte K chunk
              const uint64_t adesc = make_smem_desc(w_addr + a * kDecAtomW + kk * 32, 16, 1024, kSwizzle128B);
              const uint64_t bdesc = make_smem_desc(xc_addr + chunk * x_lbo, x_lbo, 0, kSwizzleNone);
              const uint32_t accum = (kb > kb0 || jj > 0) ? 1u : 0u;
              if (C::kFP4) {
                const uint32_t slot = 32u + static_cast<uint32_t>(it & 1) * C::kSfSlot;
                const uint32_t sfa_col = slot + jj * 4;
                const uint32_t sfb_col = slot + C::kSfCols + jj * 4;
                if (jj == 0) {
                  // the unit's scale copies first (weight atoms and token lines
                  // of its k-steps), then its MMAs
#pragma unroll
                  for (int j2 = 0; j2 < 4 * KA; ++j2) {
                    tc_cp_32x128b_warpx4(tmem_base + slot + j2 * 4,
                                         make_smem_desc(smem_u32(sfa) + j2 * 512, 16, 128, kSwizzleNone));
                    tc_cp_32x128b_warpx4(tmem_base + slot + C::kSfCols + j2 * 4,
                                         make_smem_desc(xsf_addr + (kb * KA * 4 + j2) * x_lbo, 16, 128, kSwizzleNone));
                  }
                }
                mma_mxf4nvf4(d_tmem, adesc, bdesc, C::kIdesc, tmem_base + sfa_col, tmem_base + sfb_col, accum);
              } else {
                mma_f8f6f4(d_tmem, adesc, bdesc, C::kIdesc, accum);
              }
            }
          }
          tc_commit(&empty_bar[s]);   // frees the stage once these MMAs have read it
        }
        __syncwarp();
      }
      if (lane == 0) tc_commit(&accf_bar[b]);   // this segment's accumulator (or a drain after an abort)
      __syncwarp();
      ++j;
    }
    if (lane == 0 && j > 0) {
      // nothing of this warp in flight at exit
      const int bl = (j - 1) & 1;
      (void)mbar_wait_bounded(&accf_bar[bl], ((j - 1) >> 1) & 1u, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ===== helpers =====
    const int et = threadIdx.x - 64;
    const int hw = warp - 2;                      // helper warp 0..3
    // (launch parameters only: worked out while the preceding kernel runs)
    const int nch = p.K / 8;                      // 16-byte bf16 chunks per row
    // Quantization steps (FP8: 8-element chunks; NVFP4: 16-element blocks;
    // 16 KA of either per weight unit) that this CTA's MMAs read: those of
    // the K atoms its units cover, [lo, hi] or, wrapping around a tile end,
    // [lo, end) and [0, hi]; the whole row when it covers a tile.
    const int nsteps = C::kFP4 ? p.K / kNvfp4Block : nch;
    int rb0, re0, rb1 = 0, re1 = 0;
    // the K units of tile 0 in this CTA's run [own_lo, own_hi): the codes of
    // those steps go to the workspace copy from this CTA only (one writer each)
    int own_lo, own_hi;
    {
      const long long ub = (p.U * c) / p.G, ue = (p.U * (c + 1)) / p.G;
      own_lo = static_cast<int>(min(ub, static_cast<long long>(p.nkb)));
      own_hi = static_cast<int>(min(ue, static_cast<long long>(p.nkb)));
      const int lo = static_cast<int>(ub % p.nkb) * 16 * KA;
      const int hi = min(nsteps, (static_cast<int>((ue - 1) % p.nkb) + 1) * 16 * KA);
      rb0 = ue - ub >= p.nkb ? 0 : lo;
      re0 = ue - ub >= p.nkb || lo >= hi ? nsteps : hi;
      if (ue - ub < p.nkb && lo >= hi) re1 = hi;
    }
    // the preceding kernel on the stream has completed: X, idx, mask and the
    // workspace are valid from here on
    pdl_wait_primary();
    // The activation rows come in one bulk copy into the last ring slots
    // (one round trip for any K), and the quantizers read them from there:
    // on this two-die GPU a dependent round trip to L2 costs about a
    // microsecond, so loads that do not depend on each other are issued
    // together.
    const __nv_bfloat16* xs = reinterpret_cast<const __nv_bfloat16*>(smem + static_cast<size_t>(stages - p.xslots) *
                                                                     C::kStage);
    if (et == 0) {
      fence_proxy_async_global();       // the preceding kernel's writes of X, for the copy engine
      mbar_arrive_expect_tx(xst_bar, static_cast<uint32_t>(M * p.K * 2));
      for (int t = 0; t < M; ++t)
        bulk_copy_g2s(const_cast<__nv_bfloat16*>(xs) + static_cast<size_t>(t) * p.K,
                      p.X + static_cast<size_t>(t) * p.ldx, static_cast<uint32_t>(p.K * 2), xst_bar);
    }
    int li = -1, mk = 1;
    if (et < M && p.adapters) {
      li = p.idx[et];
      if (p.mask != nullptr) mk = p.mask[et];
    }
    // this launch's tag: earlier launches on this workspace have added 256
    // each to the counter, CTAs of this one that already exited less than 256
    const unsigned epoch = launch_tag(__ldcg(p.counter) >> 8);
    float alpha = 1.0f;
    if (et < M) {
      if (li >= p.L) record_status(p.status, EPILORA_ERR_INVALID_ARG);
      meta_idx[et] = (li >= 0 && li < p.L && mk != 0) ? li : -1;
    }
    if (!mbar_wait_bounded(xst_bar, 0, kWaitLimitNs)) {
      *abort_flag = 1;
      record_status(p.status, EPILORA_ERR_TIMEOUT);
    }
    const uint4* xs4 = reinterpret_cast<const uint4*>(xs);   // chunk q of the M x nch chunks
    // ---- activation quantization into the compact copy ----
    if (!C::kFP4) {
      // per-token amax over the whole row, on bf16 pairs
#pragma unroll 1
      for (int t = 0; t < M; ++t) {
        const uint4* row = xs4 + static_cast<size_t>(t) * nch;
        __nv_bfloat162 m2 = __float2bfloat162_rn(0.0f);
#pragma unroll 4
        for (int q = et; q < nch; q += 128) m2 = __hmax2(m2, absmax8_bf16(row[q]));
        float mx = fmaxf(__low2float(m2), __high2float(m2));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) red[hw * kDecMaxTokens + t] = mx;
      }
      helper_sync();
      if (et < M) {
        const float mx = fmaxf(fmaxf(red[et], red[kDecMaxTokens + et]),
                               fmaxf(red[2 * kDecMaxTokens + et], red[3 * kDecMaxTokens + et]));
        const float sc = __fdiv_rn(fmaxf(mx, kAmaxFloor), kE4M3Max);
        meta_sx[et] = sc;
        meta_rs[et] = __frcp_rn(sc);
        if (c == 0) p.xs_out[et] = sc;
      }
      helper_sync();
      // the codes of this CTA's steps, also stored to the workspace copy:
      // four independent chunks per thread and round (the division by the
      // reciprocal product; the IEEE division for rows whose scale is below
      // 2^-100)
      bool tiny = false;
      for (int t = 0; t < M; ++t) tiny = tiny || !(meta_sx[t] >= 0x1p-100f);
      const int kown0 = own_lo * 128 * KA, kown1 = own_hi * 128 * KA;
      auto put = [&](int t, int k0, uint2 code) {
        *reinterpret_cast<uint2*>(xc + ((k0 >> 4) * M + t) * 16 + ((k0 >> 3) & 1) * 8) = code;
        if (k0 >= kown0 && k0 < kown1) *reinterpret_cast<uint2*>(p.xq_out + static_cast<size_t>(t) * p.K + k0) = code;
      };
#pragma unroll 1
      for (int g = 0; g < 2; ++g) {
        const int rbg = g == 0 ? rb0 : rb1;
        const int n = (g == 0 ? re0 : re1) - rbg;
        if (!tiny) {
#pragma unroll 1
          for (int q0 = et; q0 < M * n; q0 += 4 * 128) {
            int t4[4], k4[4];
            uint4 v4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int q = q0 + u * 128;
              t4[u] = q / n;
              k4[u] = (rbg + q - t4[u] * n) * 8;
              if (q < M * n) v4[u] = xs4[static_cast<size_t>(t4[u]) * nch + k4[u] / 8];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (q0 + u * 128 < M * n)
                put(t4[u], k4[u], quant8_e4m3_rs(v4[u], meta_sx[t4[u]], meta_rs[t4[u]]));
          }
        } else {
#pragma unroll 1
          for (int q = et; q < M * n; q += 128) {
            const int t = q / n;
            const int k0 = (rbg + q - t * n) * 8;
            const float sc = meta_sx[t];
            const uint4 v = xs4[static_cast<size_t>(t) * nch + k0 / 8];
            put(t, k0, sc >= 0x1p-100f ? quant8_e4m3_rs(v, sc, meta_rs[t]) : quant8_e4m3(v, sc));
          }
        }
      }
      // zero codes past K up to the unit boundary (finite values against the
      // weight box's zero fill)
      for (int q = et; q < M * (p.kb_pad - p.K) / 8; q += 128) {
        const int per = (p.kb_pad - p.K) / 8;
        const int t = q / per;
        const int k0 = p.K + (q - t * per) * 8;
        *reinterpret_cast<uint2*>(xc + ((k0 >> 4) * M + t) * 16 + ((k0 >> 3) & 1) * 8) = make_uint2(0, 0);
      }
    } else {
      // NVFP4: per 16-element block, its scale and codes (block-local), for
      // this CTA's blocks
      const float g = *p.x_gs;
      const bool g_ok = (g > 0.0f) && isfinite(g);
      if (!g_ok && et == 0) record_status(p.status, EPILORA_ERR_INVALID_ARG);
      alpha = 1.0f / (g * *p.w_gs);
      const int nb = nsteps;
#pragma unroll 1
      for (int gi = 0; gi < 2; ++gi) {
        const int rbg = gi == 0 ? rb0 : rb1;
        const int n = (gi == 0 ? re0 : re1) - rbg;
#pragma unroll 2
        for (int q = et; q < M * n; q += 128) {
          const int t = q / n;
          const int b = rbg + q - t * n;
          const uint4* row = xs4 + static_cast<size_t>(t) * nch;
          float x[16];
          {
            float a0[8], a1[8];
            unpack8(row[2 * b], a0);
            unpack8(row[2 * b + 1], a1);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              x[i] = a0[i];
              x[8 + i] = a1[i];
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
          // block b is bytes [8 b, 8 b + 8) of the packed row: 16-byte chunk
          // b / 2, half b % 2; its scale is byte b % 4 of the line of k-step b / 4
          *reinterpret_cast<uint2*>(xc + ((b >> 1) * M + t) * 16 + (b & 1) * 8) = make_uint2(lo, hi);
          xsf[((b >> 2) * M + t) * 16 + (b & 3)] = static_cast<uint8_t>(sb);
          if (b >= own_lo * 16 * KA && b < own_hi * 16 * KA) {
            *reinterpret_cast<uint2*>(p.xq_out + static_cast<size_t>(t) * (p.K / 2) + b * 8) = make_uint2(lo, hi);
            p.xsb_out[static_cast<size_t>(t) * nb + b] = static_cast<uint8_t>(sb);
          }
        }
      }
    }
    if (C::kFP4) {
      // codes and scales past K up to the unit boundary are zero (E4M3 scale
      // bytes could otherwise read as NaN against the zero-filled weights)
      const int nb = p.K / kNvfp4Block, nb_pad = 2 * p.kb_pad / kNvfp4Block;
      for (int q = et; q < M * (nb_pad - nb); q += 128) {
        const int t = q / (nb_pad - nb);
        const int b = nb + (q - t * (nb_pad - nb));
        *reinterpret_cast<uint2*>(xc + ((b >> 1) * M + t) * 16 + (b & 1) * 8) = make_uint2(0, 0);
        xsf[((b >> 2) * M + t) * 16 + (b & 3)] = 0;
      }
    }
    // the MMA reads the compact copy through the async proxy
    fence_proxy_async_smem();
    helper_sync();
    if (et == 0) mbar_arrive(xrdy_bar);           // the MMA warp may start
    // ---- epilogue of one segment (T, kb0, kb1), the j-th of this CTA ----
    const int q4 = warp & 3;                      // TMEM lane quadrant of this warp
    const int m = q4 * 32 + lane;                 // weight row within the tile
    bool s_ready = false;
    uint32_t brow[kMaxRankBrow];
    long long brow_key = -1;
    const bool qa = p.a_scale != nullptr;         // stored FP8 adapters
    const int brow_bytes = qa ? p.r : 2 * p.r;
    auto load_brow = [&](int l, int T, int n) {
      const uint4* bsrc = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.B) +
                                                         (static_cast<size_t>(l) * p.N + n) * brow_bytes);
#pragma unroll
      for (int cc = 0; cc < kMaxRankBrow / 4; ++cc)
        if (cc < brow_bytes / 16) {
          const uint4 bv = ldg_nc_v4_now(bsrc + cc);
          brow[4 * cc] = bv.x;
          brow[4 * cc + 1] = bv.y;
          brow[4 * cc + 2] = bv.z;
          brow[4 * cc + 3] = bv.w;
        }
      brow_key = static_cast<long long>(l) * p.n_tiles + T;
    };
    auto fail = [&]() {
      if (et == 0) {
        *abort_flag = 1;
        record_status(p.status, EPILORA_ERR_TIMEOUT);
      }
      return false;
    };
    auto epilogue_segment = [&](int T, int kb0, int kb1, int j) -> bool {
      const int b = j & 1;
      const int n = T * 128 + m;
      const bool finisher = kb0 == 0;
      float sw = 0.0f;
      if (finisher && n < p.N) {
        // loads of this row's scale and B row go out before the accumulator
        // is ready (the B row of the first token that carries an adapter)
        if (!C::kFP4) sw = ldg_nc_f32_now(p.w_scale + n);
        if (p.adapters) {
          for (int t = 0; t < M; ++t) {
            const int l = meta_idx[t];
            if (l < 0) continue;
            if (static_cast<long long>(l) * p.n_tiles + T != brow_key) load_brow(l, T, n);
            break;
          }
        }
      }
      const bool ok = mbar_wait_bounded(&accf_bar[b], (j >> 1) & 1u, kWaitLimitNs);
      if (helper_any(!ok || *abort_flag)) return fail();
      tc_fence_after();
      uint32_t v[16];
      tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(b * 16), v);
      tmem_ld_wait();
      tc_fence_before();
      helper_sync();
      if (et == 0) mbar_arrive(&acce_bar[b]);     // the accumulator may take the next segment
      float acc[kDecMaxTokens];
#pragma unroll
      for (int t = 0; t < kDecMaxTokens; ++t) acc[t] = __uint_as_float(v[t]);
      if (!finisher) {
        // publish this CTA's partial rows of tile T: slot c, [token][row],
        // each value tagged with the launch epoch
        uint2* dst = p.accp + static_cast<size_t>(c) * M * 128;
#pragma unroll
        for (int t = 0; t < kDecMaxTokens; ++t)
          if (t < M) __stcg(dst + t * 128 + m, make_uint2(__float_as_uint(acc[t]), epoch));
        return true;
      }
      // finisher: the partial rows of the CTAs holding the rest of tile T
      // (added in CTA order) and, the first time, S (its K-slice partial sums
      // added in part order), each value read until it carries this launch's
      // epoch (bounded)
      const int c_last = kb1 < p.nkb ? cta_of_unit(p, static_cast<long long>(T) * p.nkb + p.nkb - 1) : c;
      const bool need_s = p.adapters && !s_ready;
      bool late = false;
      // first round, all in flight together: up to 8 partial-row values of
      // this thread's row (the other CTAs' rows in CTA order, tokens
      // innermost: one run with a stride of 128 words) and the S parts of
      // this thread's first S element
      const int np = (c_last - c) * M;
      const uint2* pp = p.accp + static_cast<size_t>(c + 1) * M * 128 + m;
      const size_t part_stride = static_cast<size_t>(M) * p.s_row;
      uint2 wp[8], wsp[kDecSParts];
      load_tagged_n<8>(pp, 128, min(8, np), wp);
      if (need_s && et < M * p.s_row && meta_idx[et / p.s_row] >= 0)
        load_tagged_n<kDecSParts>(p.S + et, part_stride, p.parts, wsp);
      if (need_s) {
        for (int e = et; e < M * p.s_row; e += 128) {
          const int t = e / p.s_row;
          float sum = 0.0f;
          if (meta_idx[t] >= 0 && !late) {
            if (e != et) load_tagged_n<kDecSParts>(p.S + e, part_stride, p.parts, wsp);
            float v[kDecSParts];
            if (check_tagged_n<kDecSParts>(p.S + e, part_stride, p.parts, epoch, wsp, v)) {
              sum = v[0];
#pragma unroll
              for (int q = 1; q < kDecSParts; ++q)
                if (q < p.parts) sum += v[q];
            } else {
              late = true;
            }
          }
          s_stage[e] = sum;
        }
      }
      for (int i0 = 0; i0 < np && !late; i0 += 8) {
        if (i0 > 0) load_tagged_n<8>(pp + static_cast<size_t>(i0) * 128, 128, min(8, np - i0), wp);
        float v[8];
        if (!check_tagged_n<8>(pp + static_cast<size_t>(i0) * 128, 128, min(8, np - i0), epoch, wp, v)) {
          late = true;
          break;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i0 + i < np) {
            const int t = (i0 + i) % M;
#pragma unroll
            for (int tt = 0; tt < kDecMaxTokens; ++tt)
              if (tt == t) acc[tt] += v[i];
          }
      }
      if (helper_any(late)) return fail();        // (also: S staged for every thread)
      s_ready = s_ready || need_s;
      if (n < p.N) {
        const int soff = p.adapters ? dec_slice_offset(p, T * 128) : 0;
        // a rolled loop over the tokens (this thread's sums through shared
        // memory): one copy of the adapter dot in the code
#pragma unroll
        for (int t = 0; t < kDecMaxTokens; ++t)
          if (t < M) yacc[t * 128 + m] = acc[t];
#pragma unroll 1
        for (int t = 0; t < M; ++t) {
          float y = C::kFP4 ? yacc[t * 128 + m] * alpha : (yacc[t * 128 + m] * meta_sx[t]) * sw;
          const int l = meta_idx[t];
          if (l >= 0) {
            if (static_cast<long long>(l) * p.n_tiles + T != brow_key) load_brow(l, T, n);
            const float4* srow = reinterpret_cast<const float4*>(s_stage + t * p.s_row + soff);
            if (qa) {
              float d;
              switch (p.r) {
                case 16: d = dec_dot_row_e4m3<4>(srow, brow); break;
                case 32: d = dec_dot_row_e4m3<8>(srow, brow); break;
                case 64: d = dec_dot_row_e4m3<16>(srow, brow); break;
                default: d = dec_dot_row_e4m3<32>(srow, brow); break;
              }
              y += d * __ldg(p.b_scale + static_cast<size_t>(l) * p.N + n);
            } else {
              switch (p.r) {
                case 16: y += dec_dot_row<4>(srow, brow); break;
                case 32: y += dec_dot_row<8>(srow, brow); break;
                case 64: y += dec_dot_row<16>(srow, brow); break;
                default: y += dec_dot_row<32>(srow, brow); break;
              }
            }
          }
          p.Y[static_cast<size_t>(t) * p.ldy + n] = __float2bfloat16_rn(y);
        }
      }
      return true;
    };
    // ---- shrink items: (token, 4 ranks, K slice); CTA c takes items c,
    // c + G, c + 2 G, ... ----
    const int groups = p.s_row / kDecRanksPerItem;
    auto do_item = [&](int item) {
      const int t = item / (groups * p.parts);
      const int rem = item - t * groups * p.parts;
      const int part = rem / groups;
      const int j0 = (rem - part * groups) * kDecRanksPerItem;
      const int l = meta_idx[t];
      if (l >= 0) {
        const int c0 = part * p.kslice / 8;
        const int c1 = min(p.K, (part + 1) * p.kslice) / 8;
        const uint4* xr = reinterpret_cast<const uint4*>(p.X + static_cast<size_t>(t) * p.ldx);
        const size_t arow = (static_cast<size_t>(l) * p.s_row + j0) * static_cast<size_t>(p.K);   // first A row
        float accs[kDecRanksPerItem];
#pragma unroll
        for (int jr = 0; jr < kDecRanksPerItem; ++jr) accs[jr] = 0.0f;
        if (!qa) {
          const uint4* ar = reinterpret_cast<const uint4*>(p.A + arow);
#pragma unroll 2
          for (int ch = c0 + et; ch < c1; ch += 128) {
            const uint4 xw = __ldcg(xr + ch);
            uint4 av[kDecRanksPerItem];
#pragma unroll
            for (int jr = 0; jr < kDecRanksPerItem; ++jr) av[jr] = __ldg(ar + static_cast<size_t>(jr) * nch + ch);
#pragma unroll
            for (int jr = 0; jr < kDecRanksPerItem; ++jr) accs[jr] = dec_dot8(xw, av[jr], accs[jr]);
          }
        } else {
          // E4M3 rows: 8 codes (8 bytes) per 8 activations
          const uint2* ar = reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(p.A) + arow);
#pragma unroll 2
          for (int ch = c0 + et; ch < c1; ch += 128) {
            const uint4 xw = __ldcg(xr + ch);
            uint2 av[kDecRanksPerItem];
#pragma unroll
            for (int jr = 0; jr < kDecRanksPerItem; ++jr) av[jr] = __ldg(ar + static_cast<size_t>(jr) * nch + ch);
#pragma unroll
            for (int jr = 0; jr < kDecRanksPerItem; ++jr) accs[jr] = dec_dot8_e4m3(xw, av[jr], accs[jr]);
          }
        }
#pragma unroll
        for (int jr = 0; jr < kDecRanksPerItem; ++jr) {
          float sv = accs[jr];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
          if (lane == 0) red[hw * kDecRanksPerItem + jr] = sv;
        }
        helper_sync();
        if (et == 0) {
          float4 o;
          float* ov = &o.x;
#pragma unroll
          for (int jr = 0; jr < kDecRanksPerItem; ++jr) {
            float sum = 0.0f;
            for (int w = 0; w < 4; ++w) sum += red[w * kDecRanksPerItem + jr];
            // stored FP8 rows: the row's scale applied to the slice's sum
            ov[jr] = qa ? sum * __ldg(p.a_scale + static_cast<size_t>(l) * p.s_row + j0 + jr) : sum;
          }
          uint4* dst = reinterpret_cast<uint4*>(p.S + (static_cast<size_t>(part) * M + t) * p.s_row + j0);
          if (!p.drop_s) {
            __stcg(dst, make_uint4(__float_as_uint(o.x), epoch, __float_as_uint(o.y), epoch));
            __stcg(dst + 1, make_uint4(__float_as_uint(o.z), epoch, __float_as_uint(o.w), epoch));
          }
        }
      }
    };
    if (p.adapters && c < p.n_items) do_item(c);
    SegWalk walk(p, c);
    int T, kb0, kb1, j = 0;
    bool have = walk.next(T, kb0, kb1);
    bool alive = true;
    // a first segment that another CTA finishes: its partial rows next, so
    // that CTA does not wait on them
    if (have && kb0 > 0) {
      alive = epilogue_segment(T, kb0, kb1, j++);
      have = walk.next(T, kb0, kb1);
    }
    if (p.adapters && alive)
      for (int item = c + p.G; item < p.n_items; item += p.G) do_item(item);
    while (alive && have) {
      alive = epilogue_segment(T, kb0, kb1, j++);
      have = walk.next(T, kb0, kb1);
    }
  }

  // ---------------------------------------------------------------- exit
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 64) {
    // (a helper thread: it has read this launch's epoch) 256 in all per
    // launch: 1 per CTA, CTA 0 the rest; nothing waits for the reduction
    const unsigned long long add = c == 0 ? static_cast<unsigned long long>(kDecMaxCtas + 1 - p.G) : 1ull;
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p.counter), "l"(add) : "memory");
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace

// Whether the single-kernel decode path takes (fmt, M, K): a few tokens whose
// quantized rows fit the per-CTA compact copy (and, for FP8, the quantizer's
// registers).
// 128-byte K atoms per weight unit (a unit is KA atoms of one 128-row tile)
constexpr int kDecKA = 2;

namespace {

// Shared-memory plan of one call: ring stages, the slots that first hold the
// bf16 activation rows, and the bytes outside the ring.
struct DecPlan {
  int nkb, kb_pad, stages, xslots, fixed, stage_bytes;
};

template <int FMT, int KA>
bool decode_plan_t(int M, int K, int s_row, DecPlan* pl) {
  using C = DecCfg<FMT, KA>;
  const int kbytes = C::kFP4 ? K / 2 : K;
  pl->nkb = (kbytes + 128 * KA - 1) / (128 * KA);
  pl->kb_pad = pl->nkb * 128 * KA;
  pl->stage_bytes = C::kStage;
  // [ring][compact codes + 128][token scale lines + 512][S rows][row sums][barriers, metadata]
  const int xsf_bytes = C::kFP4 ? (M * (pl->kb_pad / 32) * 16 + 512 + 127) / 128 * 128 : 0;
  pl->fixed = 1024 + M * pl->kb_pad + 128 + xsf_bytes + (M * s_row + 31) / 32 * 128 + M * 512 + 1024;
  int stages = (kDecSmemBudget - pl->fixed) / C::kStage;
  if (stages > kDecMaxStages) stages = kDecMaxStages;
  pl->stages = stages;
  pl->xslots = (M * K * 2 + C::kStage - 1) / C::kStage;
  // at least one slot streams weights while the rows are quantized
  return stages >= 2 && pl->xslots <= stages - 1 && pl->fixed + stages * C::kStage <= 227 * 1024;
}

}  // namespace

// Whether the single-kernel decode path takes (fmt, M, K) with S rows of
// s_row floats (rank x slices, 0 without adapters): a few tokens whose
// quantized rows (padded to whole units) fit the per-CTA compact copy, whose
// bf16 rows fit the ring slots that stage them, and, for FP8, M * K <= 16384.
bool decode_path_eligible(int fmt, int M, int K, int s_row) {
  if (M < 1 || M > kDecMaxTokens || K < 32 || K % 32 != 0 || s_row < 0 || s_row > kDecMaxSRow) return false;
  DecPlan pl{};
  if (fmt == EPILORA_FMT_FP8_E4M3)
    return M * K <= 16384 && decode_plan_t<EPILORA_FMT_FP8_E4M3, kDecKA>(M, K, s_row, &pl) &&
           M * pl.kb_pad <= kDecXcBytes;
  if (fmt == EPILORA_FMT_NVFP4)
    return K % 256 == 0 && decode_plan_t<EPILORA_FMT_NVFP4, kDecKA>(M, K, s_row, &pl) &&
           M * pl.kb_pad <= kDecXcBytes;
  return false;
}

// The workspace head: the counters, then the tagged partial rows (every CTA,
// every token) and the tagged S partial sums, at fixed places that only this
// path writes, so that every tagged word there was written by an earlier
// launch (an older epoch) or is still zero.
size_t decode_sync_bytes() { return static_cast<size_t>(kDecSyncWords + kDecMaxCtas) * 4; }
size_t decode_partial_bytes() { return static_cast<size_t>(kDecMaxCtas) * kDecMaxTokens * 128 * 8; }
size_t decode_s_bytes() { return static_cast<size_t>(kDecSParts) * kDecMaxTokens * kDecMaxSRow * 8; }
static_assert((kDecSyncWords + kDecMaxCtas) * 4 + static_cast<size_t>(kDecMaxCtas) * kDecMaxTokens * 128 * 8 +
                      static_cast<size_t>(kDecSParts) * kDecMaxTokens * kDecMaxSRow * 8 ==
                  EPILORA_WORKSPACE_SYNC_BYTES,
              "workspace head size");

namespace {

template <int FMT, int KA>
int launch_fused_decode_t(DecParams& p, const DecodeArgs& a) {
  using C = DecCfg<FMT, KA>;
  DecPlan pl{};
  if (!decode_plan_t<FMT, KA>(a.M, a.K, a.s_row, &pl)) return EPILORA_ERR_UNSUPPORTED;
  const int kbytes = C::kFP4 ? a.K / 2 : a.K;
  p.nkb = pl.nkb;
  p.kb_pad = pl.kb_pad;
  p.stages = pl.stages;
  p.xslots = pl.xslots;
  p.n_tiles = (a.N + 127) / 128;
  p.U = static_cast<long long>(p.n_tiles) * p.nkb;
  int G = num_sms();
  if (G > kDecMaxCtas) G = kDecMaxCtas;
  if (p.U < G) G = static_cast<int>(p.U);
  p.G = G;
  int rc = make_tma_2d_u8(&p.tmW, a.Wq, a.N, kbytes, kbytes, 128, 128, true);
  if (rc != EPILORA_OK) return rc;
  if (C::kFP4) {
    rc = make_tma_2d_u8(&p.tmSW, a.w_block_scale, a.N, a.K / 16, a.K / 16, 128, 16 * KA, false);
    if (rc != EPILORA_OK) return rc;
  }
  const int smem = pl.fixed + pl.stages * C::kStage;

  auto kern = fused_decode_kernel<FMT, KA>;
  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EPILORA_ERR_CUDA;
  if (attr_done[dev] < smem) {
    // the largest shared-memory carveout: this CTA and the next projection's
    // fit on one SM together
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
            cudaSuccess)
      return EPILORA_ERR_CUDA;
    attr_done[dev] = smem;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(G, 1, 1);
  cfg.blockDim = dim3(kDecThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return EPILORA_ERR_CUDA;
  return EPILORA_OK;
}

}  // namespace

int launch_fused_decode(const DecodeArgs& a) {
  DecParams p{};
  p.X = static_cast<const __nv_bfloat16*>(a.X);
  p.A = static_cast<const __nv_bfloat16*>(a.A);
  p.B = static_cast<const __nv_bfloat16*>(a.B);
  p.a_scale = a.a_scale;
  p.b_scale = a.b_scale;
  p.idx = a.idx;
  p.mask = a.mask;
  p.w_scale = a.w_scale;
  p.w_gs = a.w_global_scale;
  p.x_gs = a.x_global_scale;
  p.Y = static_cast<__nv_bfloat16*>(a.Y);
  p.status = a.status_dev;
  p.counter = reinterpret_cast<unsigned long long*>(static_cast<unsigned*>(a.sync) + kDecCounterWord);
  p.S = reinterpret_cast<uint2*>(a.S);
  p.accp = reinterpret_cast<uint2*>(a.accp);
  p.xq_out = static_cast<uint8_t*>(a.Xq);
  p.xs_out = a.x_scale;
  p.xsb_out = a.x_block_scale;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.ldx = a.ldx;
  p.ldy = a.ldy;
  p.L = a.L;
  p.r = a.r;
  p.s_row = a.s_row;
  p.n_slices = a.n_slices;
  for (int q = 0; q < 4; ++q) p.slice_end[q] = a.slice_end[q];
  p.adapters = a.A != nullptr && a.B != nullptr ? 1 : 0;
  p.parts = a.parts;
  p.kslice = a.kslice;
  p.n_items = p.adapters ? a.M * (a.s_row / kDecRanksPerItem) * a.parts : 0;
  p.drop_s = a.drop_s;
  return a.fmt == EPILORA_FMT_NVFP4 ? launch_fused_decode_t<EPILORA_FMT_NVFP4, kDecKA>(p, a)
                                    : launch_fused_decode_t<EPILORA_FMT_FP8_E4M3, kDecKA>(p, a);
}

}  // namespace epi
