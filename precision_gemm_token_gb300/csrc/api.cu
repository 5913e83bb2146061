// C ABI of the multi-tenant LoRA layer: argument validation, workspace layout,
// TMA descriptor encoding and the fused decode-path launch sequence.
#include <atomic>
#include <cstring>

#include "common.cuh"

namespace epi {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static std::atomic<EncodeTiledFn> cached{nullptr};
  EncodeTiledFn fn = cached.load(std::memory_order_acquire);
  if (fn != nullptr) return fn;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || p == nullptr)
    return nullptr;
  fn = reinterpret_cast<EncodeTiledFn>(p);
  cached.store(fn, std::memory_order_release);
  return fn;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool fmt_ok(int fmt) { return fmt == EPILORA_FMT_FP8_E4M3 || fmt == EPILORA_FMT_NVFP4; }
inline bool rank_ok(int r) { return r == 16 || r == 32 || r == 64 || r == 128; }
inline bool k_ok(int K) { return K >= 32 && K % 32 == 0; }
inline size_t round256(size_t v) { return (v + 255) / 256 * 256; }

bool quant_args_ok(int fmt, const void* X, int M, int K, int ldx, const void* Xq, const float* x_scale,
                   const uint8_t* x_block_scale, const float* x_global_scale) {
  // FP8 rows need only whole 16-element groups (rank-16 rows of adapter tables)
  const bool kq = fmt == EPILORA_FMT_FP8_E4M3 ? (K >= 16 && K % 16 == 0) : k_ok(K);
  if (!fmt_ok(fmt) || M < 0 || !kq || ldx < K || ldx % 8 != 0) return false;
  if (M == 0) return true;
  if (X == nullptr || Xq == nullptr || !al16(X) || !al16(Xq)) return false;
  if (fmt == EPILORA_FMT_FP8_E4M3) return x_scale != nullptr && al4(x_scale);
  return x_block_scale != nullptr && al16(x_block_scale) && x_global_scale != nullptr && al4(x_global_scale);
}

bool shrink_args_ok(const void* X, int M, int K, int ldx, const void* A, int L, int r, const int32_t* idx,
                    const uint8_t* mask, const float* S) {
  if (M < 0 || !k_ok(K) || ldx < K || ldx % 8 != 0 || L < 1 || !rank_ok(r)) return false;
  if (M == 0) return true;
  if (X == nullptr || A == nullptr || idx == nullptr || S == nullptr) return false;
  if (!al16(X) || !al16(A) || !al16(S) || !al4(idx)) return false;
  (void)mask;
  return true;
}

}  // namespace

namespace {
std::atomic<int> g_test_drop_s{0};
std::atomic<int> g_decode_path{EPILORA_DECODE_PATH_AUTO};

// Whether the single-kernel decode path takes a call: eligible, and chosen by
// the policy (automatic: FP8 only; for NVFP4 the shrink grid and the GEMM
// are the faster pair on GB300 at one token, the 8B layer 73.5-74 against
// 77.5 us).
bool single_kernel_takes(int fmt, int M, int K, int r) {
  const int pol = g_decode_path.load(std::memory_order_relaxed);
  if (pol == EPILORA_DECODE_PATH_TWO) return false;
  if (pol == EPILORA_DECODE_PATH_AUTO && fmt != EPILORA_FMT_FP8_E4M3) return false;
  return decode_path_eligible(fmt, M, K, r);
}
}  // namespace

int decode_test_drop_s() { return g_test_drop_s.load(); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

int gemm_smem_bytes(int stage_bytes, int stages, int red_bytes) {
  return 1024 + stages * stage_bytes + red_bytes + 4096;
}

int make_tma_2d_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols_bytes, uint64_t pitch_bytes,
                   uint32_t box_rows, uint32_t box_cols, bool swizzle128) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return EPILORA_ERR_CUDA;
  if (rows == 0 || cols_bytes == 0 || pitch_bytes % 16 != 0 || !al16(base)) return EPILORA_ERR_INVALID_ARG;
  std::memset(map, 0, sizeof(*map));
  cuuint64_t dims[2] = {cols_bytes, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? EPILORA_OK : EPILORA_ERR_CUDA;
}

int make_tma_2d_swz(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols_bytes, uint64_t pitch_bytes,
                    uint32_t box_rows, uint32_t box_cols, int swizzle_span) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return EPILORA_ERR_CUDA;
  if (rows == 0 || cols_bytes == 0 || pitch_bytes % 16 != 0 || !al16(base) ||
      box_cols > static_cast<uint32_t>(swizzle_span))
    return EPILORA_ERR_INVALID_ARG;
  const CUtensorMapSwizzle swz = swizzle_span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : swizzle_span == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                 : swizzle_span == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  std::memset(map, 0, sizeof(*map));
  cuuint64_t dims[2] = {cols_bytes, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? EPILORA_OK : EPILORA_ERR_CUDA;
}

int prefer_max_shared(const void* func, int* done_flags) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EPILORA_ERR_CUDA;
  if (!done_flags[dev]) {
    if (cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
        cudaSuccess)
      return EPILORA_ERR_CUDA;
    done_flags[dev] = 1;
  }
  return EPILORA_OK;
}

static int gemm_validate(int fmt, int M, int N, int K, const void* Xq, const float* x_scale,
                         const uint8_t* x_block_scale, const float* x_global_scale, const void* Wq,
                         const float* w_scale, const uint8_t* w_block_scale, const float* w_global_scale,
                         const float* S, const void* B, int L, int r, const int32_t* idx, const void* Y, int ldy) {
  if (!fmt_ok(fmt) || M < 0 || N < 16 || N % 16 != 0 || !k_ok(K) || ldy < N || ldy % 8 != 0)
    return EPILORA_ERR_INVALID_ARG;
  if (fmt == EPILORA_FMT_NVFP4 && K % 256 != 0) return EPILORA_ERR_UNSUPPORTED;
  if (M == 0) return EPILORA_OK;
  if (Xq == nullptr || Wq == nullptr || Y == nullptr || !al16(Xq) || !al16(Wq) || !al16(Y))
    return EPILORA_ERR_INVALID_ARG;
  if (fmt == EPILORA_FMT_FP8_E4M3) {
    if (x_scale == nullptr || w_scale == nullptr || !al4(x_scale) || !al4(w_scale)) return EPILORA_ERR_INVALID_ARG;
  } else {
    if (x_block_scale == nullptr || w_block_scale == nullptr || x_global_scale == nullptr ||
        w_global_scale == nullptr || !al16(x_block_scale) || !al16(w_block_scale) || !al4(x_global_scale) ||
        !al4(w_global_scale))
      return EPILORA_ERR_INVALID_ARG;
  }
  if (S != nullptr) {
    if (B == nullptr || idx == nullptr || L < 1 || !rank_ok(r) || !al16(S) || !al16(B) || !al4(idx))
      return EPILORA_ERR_INVALID_ARG;
  }
  return EPILORA_OK;
}

}  // namespace epi

using namespace epi;

extern "C" {

EPILORA_API int epilora_abi_version(void) { return 1; }

EPILORA_API const char* epilora_status_string(int status) {
  switch (status) {
    case EPILORA_OK: return "EPILORA_OK";
    case EPILORA_ERR_INVALID_ARG: return "EPILORA_ERR_INVALID_ARG";
    case EPILORA_ERR_UNSUPPORTED: return "EPILORA_ERR_UNSUPPORTED";
    case EPILORA_ERR_CUDA: return "EPILORA_ERR_CUDA";
    case EPILORA_ERR_TIMEOUT: return "EPILORA_ERR_TIMEOUT";
    case EPILORA_ERR_WORKSPACE: return "EPILORA_ERR_WORKSPACE";
    default: return "EPILORA_UNKNOWN_STATUS";
  }
}

EPILORA_API int epilora_quant_act(int fmt, const void* X, int M, int K, int ldx, void* Xq, float* x_scale,
                                  uint8_t* x_block_scale, const float* x_global_scale, int* status_dev,
                                  void* stream) {
  if (!quant_args_ok(fmt, X, M, K, ldx, Xq, x_scale, x_block_scale, x_global_scale)) return EPILORA_ERR_INVALID_ARG;
  return launch_quant(fmt, X, M, K, ldx, Xq, x_scale, x_block_scale, x_global_scale, status_dev,
                      static_cast<cudaStream_t>(stream));
}

EPILORA_API int epilora_nvfp4_global_scale(const void* T, size_t n, float* g_out, void* stream) {
  if (T == nullptr || g_out == nullptr || n == 0 || !al16(T) || !al4(g_out)) return EPILORA_ERR_INVALID_ARG;
  return launch_global_scale(T, n, g_out, static_cast<cudaStream_t>(stream));
}

EPILORA_API int epilora_lora_shrink(const void* X, int M, int K, int ldx, const void* A, int L, int r,
                                    const int32_t* idx, const uint8_t* mask, float* S, int* status_dev,
                                    void* stream) {
  if (!shrink_args_ok(X, M, K, ldx, A, L, r, idx, mask, S)) return EPILORA_ERR_INVALID_ARG;
  return launch_shrink(X, M, K, ldx, A, L, r, idx, mask, S, status_dev, static_cast<cudaStream_t>(stream));
}

EPILORA_API int epilora_gemm_lora_epilogue(int fmt, int M, int N, int K, const void* Xq, const float* x_scale,
                                           const uint8_t* x_block_scale, const float* x_global_scale,
                                           const void* Wq, const float* w_scale, const uint8_t* w_block_scale,
                                           const float* w_global_scale, const float* S, const void* B, int L,
                                           int r, const int32_t* idx, const uint8_t* mask, void* Y, int ldy,
                                           int pdl_dependent, int* status_dev, void* stream) {
  int rc = gemm_validate(fmt, M, N, K, Xq, x_scale, x_block_scale, x_global_scale, Wq, w_scale, w_block_scale,
                         w_global_scale, S, B, L, r, idx, Y, ldy);
  if (rc != EPILORA_OK || M == 0) return rc;
  GemmArgs a{};
  a.fmt = fmt;
  a.M = M;
  a.N = N;
  a.K = K;
  a.Xq = Xq;
  a.x_scale = x_scale;
  a.x_block_scale = x_block_scale;
  a.x_global_scale = x_global_scale;
  a.Wq = Wq;
  a.w_scale = w_scale;
  a.w_block_scale = w_block_scale;
  a.w_global_scale = w_global_scale;
  a.S = S;
  a.B = B;
  a.L = S != nullptr ? L : 1;
  a.r = S != nullptr ? r : 16;
  a.idx = idx;
  a.mask = mask;
  a.Y = Y;
  a.ldy = ldy;
  a.pdl_dependent = pdl_dependent ? 1 : 0;
  a.status_dev = status_dev;
  a.stream = static_cast<cudaStream_t>(stream);
  return fmt == EPILORA_FMT_FP8_E4M3 ? launch_gemm_fp8(a) : launch_gemm_nvfp4(a);
}

EPILORA_API int epilora_layer_forward_kernels(int fmt, int M, int K, int r) {
  if (!fmt_ok(fmt) || M < 0 || !k_ok(K) || r < 0) return 0;
  if (M == 0) return 0;
  return single_kernel_takes(fmt, M, K, r) ? 1 : 2;
}

EPILORA_API int epilora_set_decode_path(int policy) {
  if (policy != EPILORA_DECODE_PATH_AUTO && policy != EPILORA_DECODE_PATH_SINGLE && policy != EPILORA_DECODE_PATH_TWO)
    return EPILORA_ERR_INVALID_ARG;
  return g_decode_path.exchange(policy);
}

EPILORA_API size_t epilora_workspace_bytes(int fmt, int M, int K, int r) {
  if (!fmt_ok(fmt) || M < 0 || K < 0 || r < 0) return 0;
  const size_t m = static_cast<size_t>(M), k = static_cast<size_t>(K);
  if (M == 0) return 0;
  // the head: counters and tagged exchange regions of the single-kernel
  // decode path, at a fixed place
  size_t bytes = EPILORA_WORKSPACE_SYNC_BYTES;
  if (fmt == EPILORA_FMT_FP8_E4M3) {
    bytes += round256(m * k);          // Xq
    bytes += round256(m * 4);          // x_scale
  } else {
    bytes += round256(m * k / 2);      // packed Xq
    bytes += round256(m * k / 16);     // block scales
  }
  // S, or the partial sums of a shrink split over K slices
  bytes += round256(m * static_cast<size_t>(r) * 4 * static_cast<size_t>(r > 0 ? shrink_parts_max(K) : 1));
  // more than one decode tile of tokens with adapters: the adapter-sorted row order
  if (r > 0 && M > 32) bytes += round256(m * 4);
  return bytes;
}

EPILORA_API size_t epilora_layer_workspace_bytes(int fmt, int M, int N, int K, int r) {
  const size_t base = epilora_workspace_bytes(fmt, M, K, r);
  if (base == 0 || N < 0) return 0;
  return r >= kExpandMinRank && M > 32 ? base + expand_yadd_bytes(M, N) : base;
}

}  // extern "C"

static int layer_forward_impl(int fmt, int M, int N, int K, const void* X, int ldx, const void* Wq,
                              const float* w_scale, const uint8_t* w_block_scale, const float* w_global_scale,
                              const float* x_global_scale, const void* A, const void* B, int L, int r,
                              const int32_t* idx, const uint8_t* mask, void* Y, int ldy, void* workspace,
                              size_t workspace_bytes, int* status_dev, void* stream, int n_slices,
                              const int* slice_end, const float* a_scale = nullptr, const float* b_scale = nullptr) {
  const bool adapters = A != nullptr && B != nullptr;
  // stored FP8 adapters (both scales given): decode batches of at most 32 tokens
  if ((a_scale == nullptr) != (b_scale == nullptr)) return EPILORA_ERR_INVALID_ARG;
  if (a_scale != nullptr) {
    if (!adapters || !al4(a_scale) || !al4(b_scale)) return EPILORA_ERR_INVALID_ARG;
    if (M > 32) return EPILORA_ERR_UNSUPPORTED;
  }
  // S rows: n_slices rank-r blocks (the shrink runs with rank r * n_slices)
  const int rs = r * n_slices;
  if (!fmt_ok(fmt) || M < 0 || !k_ok(K) || ldx < K || ldx % 8 != 0) return EPILORA_ERR_INVALID_ARG;
  if (adapters && (L < 1 || !rank_ok(r) || idx == nullptr)) return EPILORA_ERR_INVALID_ARG;
  if (fmt == EPILORA_FMT_NVFP4 && (x_global_scale == nullptr || K % 256 != 0))
    return x_global_scale == nullptr ? EPILORA_ERR_INVALID_ARG : EPILORA_ERR_UNSUPPORTED;
  if (M == 0) return EPILORA_OK;
  const int rr = adapters ? rs : 0;
  const size_t need = epilora_workspace_bytes(fmt, M, K, rr);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return EPILORA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t m = static_cast<size_t>(M), k = static_cast<size_t>(K);
  void* sync = ws;
  void* accp = ws + decode_sync_bytes();
  void* S_tagged = ws + decode_sync_bytes() + decode_partial_bytes();
  size_t off = EPILORA_WORKSPACE_SYNC_BYTES;
  void* Xq = ws + off;
  float* x_scale = nullptr;
  uint8_t* x_block_scale = nullptr;
  float* S = nullptr;
  if (fmt == EPILORA_FMT_FP8_E4M3) {
    off += round256(m * k);
    x_scale = reinterpret_cast<float*>(ws + off);
    off += round256(m * 4);
  } else {
    off += round256(m * k / 2);
    x_block_scale = ws + off;
    off += round256(m * k / 16);
  }
  int32_t* perm = nullptr;
  if (adapters) {
    S = reinterpret_cast<float*>(ws + off);
    off += round256(m * static_cast<size_t>(rs) * 4 * static_cast<size_t>(shrink_parts_max(K)));
    if (M > 32) {
      perm = reinterpret_cast<int32_t*>(ws + off);
      off += round256(m * 4);
    }
  }
  // more than 32 tokens with bf16 adapters of rank 32 or more and room for
  // the fp32 term: the expand pass computes the adapter term between the
  // shrink grid and the GEMM (rank 16 stays in the GEMM's epilogue, whose
  // tensor-core term costs little there, while the pass would add the fp32
  // term's round trip through memory)
  float* yadd = nullptr;
  if (adapters && M > 32 && r >= kExpandMinRank && a_scale == nullptr &&
      workspace_bytes >= off + expand_yadd_bytes(M, N))
    yadd = reinterpret_cast<float*>(ws + off);

  int rc = gemm_validate(fmt, M, N, K, Xq, x_scale, x_block_scale, x_global_scale, Wq, w_scale, w_block_scale,
                         w_global_scale, S, B, L, r, idx, Y, ldy);
  if (rc != EPILORA_OK) return rc;
  if (adapters && !shrink_args_ok(X, M, K, ldx, A, L, r, idx, mask, S)) return EPILORA_ERR_INVALID_ARG;
  if (!quant_args_ok(fmt, X, M, K, ldx, Xq, x_scale, x_block_scale, x_global_scale)) return EPILORA_ERR_INVALID_ARG;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (single_kernel_takes(fmt, M, K, rr)) {
    // a few tokens: quantizer, shrink and GEMM in one persistent launch
    DecodeArgs d{};
    d.fmt = fmt;
    d.M = M;
    d.N = N;
    d.K = K;
    d.ldx = ldx;
    d.ldy = ldy;
    d.L = adapters ? L : 1;
    d.r = adapters ? r : 16;
    d.s_row = adapters ? rs : 0;
    d.n_slices = n_slices;
    for (int q = 0; q < n_slices && q < 4; ++q) d.slice_end[q] = slice_end != nullptr ? slice_end[q] : N;
    int parts = shrink_parts_max(K);
    while (parts > 1 && shrink_kslice(K, parts) * (parts - 1) >= K) --parts;
    d.parts = parts;
    d.kslice = shrink_kslice(K, parts);
    d.X = X;
    d.Wq = Wq;
    d.w_scale = w_scale;
    d.w_block_scale = w_block_scale;
    d.w_global_scale = w_global_scale;
    d.x_global_scale = x_global_scale;
    d.A = adapters ? A : nullptr;
    d.B = adapters ? B : nullptr;
    d.a_scale = a_scale;
    d.b_scale = b_scale;
    d.idx = idx;
    d.mask = mask;
    d.Y = Y;
    d.status_dev = status_dev;
    d.stream = st;
    d.sync = sync;
    d.S = S_tagged;
    d.accp = accp;
    d.Xq = Xq;
    d.x_scale = x_scale;
    d.x_block_scale = x_block_scale;
    d.drop_s = decode_test_drop_s();
    return launch_fused_decode(d);
  }

  // The shrink grid (with the quantizer CTAs) is a programmatic dependent of
  // the previous kernel on the stream and releases the GEMM at once; the GEMM
  // streams W immediately and reads everything the shrink grid writes (and
  // the token metadata) only after that grid has completed.
  const int parts = adapters ? shrink_parts(M, K, rs) : shrink_parts(M, K, 0);
  rc = launch_shrink_quant(X, M, K, ldx, A, adapters ? L : 1, adapters ? rs : 0, idx, mask, S, parts, fmt, Xq,
                           x_scale, x_block_scale, x_global_scale, perm, status_dev, st, a_scale);
  if (rc != EPILORA_OK) return rc;
  if (yadd != nullptr) {
    ExpandArgs e{};
    e.M = M;
    e.N = N;
    e.L = L;
    e.r = r;
    e.s_row = rs;
    e.s_parts = parts;
    e.n_slices = n_slices;
    for (int q = 0; q < 4; ++q) e.slice_end[q] = q < n_slices && slice_end != nullptr ? slice_end[q] : N;
    e.S = S;
    e.B = B;
    e.perm = perm;
    e.idx = idx;
    e.mask = mask;
    e.yadd = yadd;
    e.status_dev = status_dev;
    e.stream = st;
    e.pdl_dependent = 1;
    rc = launch_expand(e);
    if (rc != EPILORA_OK) return rc;
  }
  GemmArgs a{};
  a.fmt = fmt;
  a.M = M;
  a.N = N;
  a.K = K;
  a.Xq = Xq;
  a.x_scale = x_scale;
  a.x_block_scale = x_block_scale;
  a.x_global_scale = x_global_scale;
  a.Wq = Wq;
  a.w_scale = w_scale;
  a.w_block_scale = w_block_scale;
  a.w_global_scale = w_global_scale;
  a.S = S;
  a.B = B;
  a.b_scale = b_scale;
  a.L = adapters ? L : 1;
  a.r = adapters ? r : 16;
  a.idx = idx;
  a.mask = mask;
  a.Y = Y;
  a.ldy = ldy;
  a.pdl_dependent = 1;
  a.status_dev = status_dev;
  a.stream = st;
  a.fused = 1;
  a.s_parts = parts;
  a.perm = perm;
  a.yadd = yadd;
  a.s_row = adapters ? rs : 0;
  a.n_slices = n_slices;
  for (int q = 0; q < n_slices && q < 4; ++q) a.slice_end[q] = slice_end != nullptr ? slice_end[q] : N;
  return fmt == EPILORA_FMT_FP8_E4M3 ? launch_gemm_fp8(a) : launch_gemm_nvfp4(a);
}

extern "C" {

EPILORA_API int epilora_layer_forward(int fmt, int M, int N, int K, const void* X, int ldx, const void* Wq,
                                      const float* w_scale, const uint8_t* w_block_scale,
                                      const float* w_global_scale, const float* x_global_scale, const void* A,
                                      const void* B, int L, int r, const int32_t* idx, const uint8_t* mask,
                                      void* Y, int ldy, void* workspace, size_t workspace_bytes, int* status_dev,
                                      void* stream) {
  return layer_forward_impl(fmt, M, N, K, X, ldx, Wq, w_scale, w_block_scale, w_global_scale, x_global_scale, A, B,
                            L, r, idx, mask, Y, ldy, workspace, workspace_bytes, status_dev, stream, 1, nullptr);
}

EPILORA_API int epilora_layer_forward_slices(int fmt, int M, int N, int K, const void* X, int ldx, const void* Wq,
                                             const float* w_scale, const uint8_t* w_block_scale,
                                             const float* w_global_scale, const float* x_global_scale,
                                             const void* A, const void* B, int L, int r, int n_slices,
                                             const int* slice_end, const int32_t* idx, const uint8_t* mask,
                                             void* Y, int ldy, void* workspace, size_t workspace_bytes,
                                             int* status_dev, void* stream) {
  if (A == nullptr || B == nullptr || n_slices < 1 || n_slices > 4 || slice_end == nullptr)
    return EPILORA_ERR_INVALID_ARG;
  int prev = 0;
  for (int q = 0; q < n_slices; ++q) {
    const int e = slice_end[q];
    if (e <= prev || e > N) return EPILORA_ERR_INVALID_ARG;
    if (q + 1 < n_slices && e % 128 != 0) return EPILORA_ERR_INVALID_ARG;   // a weight tile lies in one slice
    prev = e;
  }
  if (prev != N) return EPILORA_ERR_INVALID_ARG;
  return layer_forward_impl(fmt, M, N, K, X, ldx, Wq, w_scale, w_block_scale, w_global_scale, x_global_scale, A, B,
                            L, r, idx, mask, Y, ldy, workspace, workspace_bytes, status_dev, stream, n_slices,
                            slice_end);
}

EPILORA_API int epilora_test_drop_shrink_results(int on) {
  g_test_drop_s.store(on != 0 ? 1 : 0);
  return EPILORA_OK;
}

EPILORA_API int epilora_layer_forward_fp8_adapters(int fmt, int M, int N, int K, const void* X, int ldx,
                                                   const void* Wq, const float* w_scale, const uint8_t* w_block_scale,
                                                   const float* w_global_scale, const float* x_global_scale,
                                                   const uint8_t* Aq, const float* a_scale, const uint8_t* Bq,
                                                   const float* b_scale, int L, int r, const int32_t* idx,
                                                   const uint8_t* mask, void* Y, int ldy, void* workspace,
                                                   size_t workspace_bytes, int* status_dev, void* stream) {
  if (Aq == nullptr || Bq == nullptr || a_scale == nullptr || b_scale == nullptr) return EPILORA_ERR_INVALID_ARG;
  return layer_forward_impl(fmt, M, N, K, X, ldx, Wq, w_scale, w_block_scale, w_global_scale, x_global_scale, Aq,
                            Bq, L, r, idx, mask, Y, ldy, workspace, workspace_bytes, status_dev, stream, 1, nullptr,
                            a_scale, b_scale);
}

}  // extern "C"
