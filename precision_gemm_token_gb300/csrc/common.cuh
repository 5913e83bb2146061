// Shared definitions of the CUDA library (not part of the public ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/epilora.h"

namespace epi {

constexpr float kE4M3Max = 448.0f;
constexpr float kE2M1Max = 6.0f;
constexpr float kAmaxFloor = EPILORA_FP8_AMAX_FLOOR;
constexpr int kNvfp4Block = 16;
// Wall-clock limit of any spin-wait inside a kernel (legitimate waits last
// microseconds). After it runs out the kernel records EPILORA_ERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// First error wins (0 = OK).
__device__ __forceinline__ void record_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// host-side launch helpers shared by the translation units
// ---------------------------------------------------------------------------
struct GemmArgs {
  int fmt;
  int M, N, K;
  const void* Xq;
  const float* x_scale;
  const uint8_t* x_block_scale;
  const float* x_global_scale;
  const void* Wq;
  const float* w_scale;
  const uint8_t* w_block_scale;
  const float* w_global_scale;
  const float* S;
  const void* B;
  const float* b_scale = nullptr;   // stored FP8 B (E4M3 [L, N, r] bytes, fp32 scale per row [L, N])
  int L, r;
  const int32_t* idx;
  const uint8_t* mask;
  void* Y;
  int ldy;
  int pdl_dependent;
  int* status_dev;
  cudaStream_t stream;
  // fused layer call: Xq, its scales, idx and mask come from the primary
  // grid (launch_shrink_quant), S as s_parts partial arrays [s_parts][M][r]
  int fused = 0;
  int s_parts = 1;
  // fused call, more than one decode tile of tokens: rows of Xq / x_scale /
  // x_block_scale are in adapter-sorted order, perm[row] = token
  const int32_t* perm = nullptr;
  // multi-slice projection: S rows hold n_slices consecutive rank-r blocks
  // (s_row = n_slices * r floats); output columns [slice_end[s-1],
  // slice_end[s]) take block s. slice_end ascending, multiples of 128 but the
  // last (= N). s_row 0: r.
  int s_row = 0;
  int n_slices = 1;
  int slice_end[4] = {0, 0, 0, 0};
  // wide tiles (more than 32 tokens): the adapter term of every sorted row
  // with an adapter, computed by launch_expand, fp32 [M][N] (row = row of Xq);
  // the epilogue adds it instead of computing S[t] . B[l][n] itself. null:
  // the epilogue computes the term.
  const float* yadd = nullptr;
};

int launch_quant(int fmt, const void* X, int M, int K, int ldx, void* Xq, float* x_scale,
                 uint8_t* x_block_scale, const float* x_global_scale, int* status_dev, cudaStream_t stream);
int launch_global_scale(const void* T, size_t n, float* g_out, cudaStream_t stream);
int launch_shrink(const void* X, int M, int K, int ldx, const void* A, int L, int r, const int32_t* idx,
                  const uint8_t* mask, float* S, int* status_dev, cudaStream_t stream);
// Shrink grid with extra quantizer CTAs: Xq / scales as launch_quant, and S
// as `s_parts` partial arrays [s_parts][M][r] over consecutive K slices (their
// sum in part order is S; s_parts == 1 gives S itself). Launched as a
// programmatic dependent of the previous kernel on the stream: it releases its
// own dependent at once and waits for that kernel before reading anything.
// perm != nullptr (s_parts == 1 only): the quantized rows and their scales are
// written in adapter-sorted order (key idx[t] if the token carries an adapter,
// else L; ties by token), and perm[row] = token.
// a_scale != nullptr: A holds E4M3 codes [L, r, K] bytes with one fp32 scale
// per row [L, r] (stored FP8 adapters; at most 32 tokens).
int launch_shrink_quant(const void* X, int M, int K, int ldx, const void* A, int L, int r, const int32_t* idx,
                        const uint8_t* mask, float* S, int s_parts, int fmt, void* Xq, float* x_scale,
                        uint8_t* x_block_scale, const float* x_global_scale, int32_t* perm, int* status_dev,
                        cudaStream_t stream, const float* a_scale = nullptr);
// Number of K slices launch_shrink_quant uses for (M, K, r) (1 when M > 32),
// and the largest it can use for K (sizes the workspace).
int shrink_parts(int M, int K, int r);
int shrink_parts_max(int K);
// Single-kernel decode path (decode.cu): the whole fused layer call for a few
// tokens in one persistent launch.
struct DecodeArgs {
  int fmt;
  int M, N, K, ldx, ldy, L, r;
  int s_row;            // floats per S row (n_slices * r)
  int n_slices;
  int slice_end[4];
  int parts, kslice;    // K slices of the shrink items
  const void* X;
  const void* Wq;
  const float* w_scale;
  const uint8_t* w_block_scale;
  const float* w_global_scale;
  const float* x_global_scale;
  const void* A;        // NULL with B: no adapters
  const void* B;
  const float* a_scale; // stored FP8 adapters: row scales of A [L, s_row] and B [L, N]; NULL: bf16
  const float* b_scale;
  const int32_t* idx;
  const uint8_t* mask;
  void* Y;
  int* status_dev;
  cudaStream_t stream;
  // workspace regions (the head: counters, tagged partial rows, tagged S)
  void* sync;           // decode_sync_bytes()
  void* S;              // decode_s_bytes(): tagged [parts][M][s_row]
  void* accp;           // decode_partial_bytes(): tagged [CTA][M][128]
  void* Xq;             // the quantized activations as used (each CTA writes its K range)
  float* x_scale;
  uint8_t* x_block_scale;
  int drop_s = 0;       // test hook: the shrink items publish nothing
};
// test hook of the single-kernel path (epilora_test_drop_shrink_results)
int decode_test_drop_s();
bool decode_path_eligible(int fmt, int M, int K, int s_row);
size_t decode_sync_bytes();
size_t decode_partial_bytes();
size_t decode_s_bytes();
int launch_fused_decode(const DecodeArgs& a);
// K slice length of a shrink split into `parts` slices (multiple of 256)
int shrink_kslice(int K, int parts);

// Adapter term of a batch of more than 32 tokens as a pass of its own
// (expand.cu): yadd[row][n] = S[perm[row]] . B[l][n] for the sorted rows whose
// token carries an adapter l (mask on); other rows are not written. Launched
// as a programmatic dependent of the shrink grid when pdl_dependent is set; it
// releases its own dependent (the GEMM) at once and reads S, perm, idx and
// mask only after that grid has completed.
struct ExpandArgs {
  int M, N, L, r;
  int s_row, s_parts, n_slices;
  int slice_end[4];
  const float* S;          // [s_parts][M][s_row] fp32, rows by token
  const void* B;           // bf16 [L, N, r], 16-byte aligned
  const int32_t* perm;     // sorted row -> token, or null (identity)
  const int32_t* idx;
  const uint8_t* mask;
  float* yadd;             // fp32 [M][N]
  int* status_dev;
  cudaStream_t stream;
  int pdl_dependent;
};
int launch_expand(const ExpandArgs& a);
// smallest adapter rank (per slice) for which a layer call takes the expand pass
constexpr int kExpandMinRank = 32;
// bytes of the fp32 [M][N] buffer launch_expand writes (a multiple of 256)
size_t expand_yadd_bytes(int M, int N);

int launch_gemm_fp8(const GemmArgs& a);
int launch_gemm_nvfp4(const GemmArgs& a);

// Encodes a 2D tiled TMA descriptor for a row-major uint8 matrix
// [rows, cols_bytes] with row pitch `pitch_bytes`, box [box_rows, box_cols].
int make_tma_2d_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols_bytes, uint64_t pitch_bytes,
                   uint32_t box_rows, uint32_t box_cols, bool swizzle128);

// As make_tma_2d_u8 with the box's inner extent swizzled over `swizzle_span`
// bytes (32, 64 or 128; the inner box extent must not exceed it).
int make_tma_2d_swz(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols_bytes, uint64_t pitch_bytes,
                    uint32_t box_rows, uint32_t box_cols, int swizzle_span);

// Once per device: prefer the largest shared-memory carveout for a small
// kernel, so that the SMs it lands on keep room for the GEMM's CTAs beside it.
int prefer_max_shared(const void* func, int* done_flags);

int num_sms();

}  // namespace epi
