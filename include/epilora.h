/*
 * epilora.h — C ABI of the multi-tenant LoRA linear layer of an LLM decode step
 * on NVIDIA GB300 (sm_103a).
 *
 *   Y[t,:] = bf16( dequant( Q(X)[t,:] . Q(W)^T ) + mask[t] * (x_t . A[idx_t]^T) . B[idx_t]^T )
 *
 * The operation is the one defined on the EpiLoRA page ("Fusing Many LoRA
 * Adapters into Low-Precision GEMMs for Serving and RL"):
 *   - §Background and motivation › The cost of the separate adapter path:
 *     shrink h = x A^T, expand h B^T added to the projection's output;
 *   - §Design › Multi-adapter kernels › K1 and K2: per-token activation
 *     quantization for the low-precision base GEMM, h from the bf16
 *     activations, the GEMM epilogue applies the scales then adds h B^T;
 *   - §Design › Multi-adapter kernels › The decode path: the shrink is
 *     launched first, the GEMM as its programmatic dependent, waiting for h
 *     only before its epilogue;
 * and on the PreFT page ("PreFT: Prefill-only finetuning for efficient
 * inference", Core claim): the adapter applies to prefill tokens only, which
 * is the per-token mask.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every data pointer is a DEVICE pointer (cudaMalloc'd or equivalent) owned
 *    by the caller. The library allocates nothing and keeps no state between
 *    calls besides cached kernel attributes and the driver entry point used
 *    to encode TMA descriptors.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call
 *    only enqueues work; it never synchronizes.
 *  - Layouts are row-major with the innermost dimension contiguous:
 *      X   bf16  [M, ldx]     (K used)            activations
 *      Xq  FP8:  uint8 [M, K] E4M3 codes;  NVFP4: uint8 [M, K/2] packed E2M1
 *          (element 2i in the low nibble of byte i)
 *      x_scale        fp32 [M]                     FP8 per-token scale
 *      x_block_scale  uint8 [M, K/16] E4M3         NVFP4 per-16-block scale
 *      x_global_scale fp32 scalar (device)         NVFP4 encode multiplier g_x
 *      Wq  FP8: uint8 [N, K];  NVFP4: uint8 [N, K/2]
 *      w_scale        fp32 [N]                     FP8 per-output-channel scale
 *      w_block_scale  uint8 [N, K/16];  w_global_scale fp32 scalar (device)
 *      A   bf16 [L, r, K]   (h = x A_l^T)
 *      B   bf16 [L, N, r]   (delta = h B_l^T)
 *      idx int32 [M]   adapter slot of each token; idx < 0 = no adapter
 *      mask uint8 [M]  0 = adapter skipped for this token; NULL = all ones
 *      S   fp32 [M, r]  shrink output (workspace)
 *      Y   bf16 [M, ldy] (N used)
 *  - Constraints (checked on the host before any launch; violation returns
 *    EPILORA_ERR_INVALID_ARG and enqueues nothing): M >= 0 (M == 0 is a
 *    no-op), K % 32 == 0 and K >= 32, N % 16 == 0 and N >= 16,
 *    r in {16, 32, 64, 128}, L >= 1, ldx >= K and ldx % 8 == 0,
 *    for NVFP4 GEMMs K % 256 == 0 (the block-scale rows must be 16-byte
 *    multiples for the tensor-memory-accelerator copies),
 *    ldy >= N and ldy % 8 == 0, every data pointer 16-byte aligned, the
 *    NVFP4 global scales non-NULL.
 *  - Device-detected conditions are written to the optional `status_dev`
 *    (int32 on the device, caller-owned; the first error wins through an
 *    atomic compare-and-swap of 0): an adapter index idx >= L makes that
 *    token "no adapter" and records EPILORA_ERR_INVALID_ARG; a non-positive
 *    or non-finite NVFP4 global scale records EPILORA_ERR_INVALID_ARG; a
 *    bounded wait inside a kernel that ran out records EPILORA_ERR_TIMEOUT
 *    (the kernel then releases its resources and returns; its outputs are
 *    undefined). Kernels never trap.
 *  - Results are deterministic: every reduction is summed in a fixed order
 *    (no floating-point atomics), so the same inputs at the same M give
 *    bitwise-identical outputs.
 *  - Errors from the CUDA runtime at launch are returned as EPILORA_ERR_CUDA.
 */
#ifndef EPILORA_H_
#define EPILORA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define EPILORA_API __attribute__((visibility("default")))
#else
#define EPILORA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EPILORA_OK = 0,
  EPILORA_ERR_INVALID_ARG = -1,
  EPILORA_ERR_UNSUPPORTED = -2,
  EPILORA_ERR_CUDA = -3,
  EPILORA_ERR_TIMEOUT = -4,
  EPILORA_ERR_WORKSPACE = -5
} epilora_status;

typedef enum { EPILORA_FMT_FP8_E4M3 = 0, EPILORA_FMT_NVFP4 = 1 } epilora_format;

/* Smallest per-token amax used by the FP8 quantizer: an all-zero token gets
 * scale 1e-12f / 448 and all-zero codes. */
#define EPILORA_FP8_AMAX_FLOOR 1e-12f

/* Version of this ABI (bumped on any signature change). */
EPILORA_API int epilora_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
EPILORA_API const char* epilora_status_string(int status);

/*
 * Per-token activation quantizer (S1 / S1').
 * Defined by: EpiLoRA page, §Design › Multi-adapter kernels › K1 and K2
 * (activations are quantized one time per layer, with one scale per token,
 * for the low-precision base GEMM), and its Introduction / Related work for
 * the block-scaled 4-bit NVFP4 format.
 *
 * FP8:   s_t = fl32(max(amax_t, EPILORA_FP8_AMAX_FLOOR) / 448)  (IEEE division)
 *        Xq[t,k] = E4M3_rn_satfinite(fl32(X[t,k] / s_t));  x_scale[t] = s_t
 *        (x_block_scale, x_global_scale ignored; may be NULL)
 * NVFP4: per 16-element block b of token t, with g = *x_global_scale:
 *        sb = E4M3_rn_satfinite(fl32(fl32(amax_b / 6) * g));
 *        sb == 0 -> the block's codes are 0, else
 *        code = E2M1_rn_satfinite(fl32(X * fl32(g / sb)));
 *        x_block_scale[t,b] = sb (E4M3 byte)          (x_scale ignored)
 * Applied to a weight matrix (M := N rows) this also produces the FP8
 * per-output-channel weight scales and the NVFP4 weight codes, and applied to
 * the rows of adapter tables the stored FP8 adapters of
 * epilora_layer_forward_fp8_adapters (FP8 takes any K % 16 == 0, so rank-16
 * rows too). Codes and scales are bit-exact functions of the inputs.
 */
EPILORA_API int epilora_quant_act(int fmt, const void* X, int M, int K, int ldx,
                      void* Xq, float* x_scale, uint8_t* x_block_scale,
                      const float* x_global_scale, int* status_dev, void* stream);

/*
 * NVFP4 encode multiplier of a whole bf16 tensor of n elements:
 *   *g_out = fl32(448 * 6 / max(amax, EPILORA_FP8_AMAX_FLOOR)).
 * A load-time (weights) or calibration (activations) helper; the EpiLoRA
 * page only says NVFP4 has an fp32 global scale. g_out is a device float.
 */
EPILORA_API int epilora_nvfp4_global_scale(const void* T, size_t n, float* g_out, void* stream);

/*
 * Multi-adapter shrink (down-projection) (S2).
 * Defined by: EpiLoRA page, §Background and motivation › The cost of the
 * separate adapter path (h = x A^T) and §Design › Multi-adapter kernels ›
 * K1 and K2 (h from the bf16 activations); mask from the PreFT page.
 *   S[t, j] = sum_k X[t,k] * A[idx_t, j, k]   (fp32 accumulate, fixed order)
 * for tokens with idx_t in [0, L) and (mask == NULL or mask[t] != 0);
 * S[t, :] = 0 for every other token. Launched as an ordinary kernel (it
 * waits for X); it allows a dependent kernel to launch at once.
 */
EPILORA_API int epilora_lora_shrink(const void* X, int M, int K, int ldx,
                        const void* A, int L, int r,
                        const int32_t* idx, const uint8_t* mask,
                        float* S, int* status_dev, void* stream);

/*
 * Low-precision base GEMM with the multi-adapter LoRA epilogue (S3 + S5, S4).
 * Defined by: EpiLoRA page, §Design › Multi-adapter kernels › K1 and K2
 * (the epilogue applies the scales and adds h_l B_l^T for the rows of each
 * adapter) and › The decode path (launched as the shrink's dependent; waits
 * for h only before its epilogue).
 *   FP8:   Y[t,n] = bf16( (sum_k Xq[t,k] Wq[n,k]) * x_scale[t] * w_scale[n] + d[t,n] )
 *   NVFP4: Y[t,n] = bf16( (sum_k (Xq*sbx)[t,k] (Wq*sbw)[n,k]) / (g_x * g_w) + d[t,n] )
 *   d[t,n] = sum_j S[t,j] * B[idx_t, n, j] for active tokens (as in the
 *            shrink), else 0; with S == NULL there is no adapter term.
 * pdl_dependent = 1 launches the kernel with programmatic stream
 * serialization: it may start while the previous kernel on the stream (the
 * shrink) is still running, streams W and Xq at once, and executes the
 * grid-dependency wait before it reads x_scale, idx, mask or S.
 * pdl_dependent = 0 is an ordinary launch.
 * With pdl_dependent = 1, Xq and x_block_scale must already be complete when
 * the previous kernel on the stream started (e.g. written by
 * epilora_quant_act before the shrink); x_scale, S, idx and mask may be
 * written by that kernel.
 */
EPILORA_API int epilora_gemm_lora_epilogue(int fmt, int M, int N, int K,
                               const void* Xq, const float* x_scale,
                               const uint8_t* x_block_scale, const float* x_global_scale,
                               const void* Wq, const float* w_scale,
                               const uint8_t* w_block_scale, const float* w_global_scale,
                               const float* S, const void* B, int L, int r,
                               const int32_t* idx, const uint8_t* mask,
                               void* Y, int ldy, int pdl_dependent,
                               int* status_dev, void* stream);

/*
 * Bytes of device workspace epilora_layer_forward needs for (fmt, M, K, r):
 * a head of EPILORA_WORKSPACE_SYNC_BYTES (2.25 MiB: the single-kernel decode
 * path's launch counter and the regions where its thread blocks exchange
 * partial results, see epilora_layer_forward_kernels), then the quantized
 * activations, their scales, S (r = 0: no adapters; S is held as up to
 * ceil(K / 1024) partial sums over K slices, capped at 8) and, for more than
 * 32 tokens with adapters, a row-to-token map; each region 256-byte aligned.
 * Returns 0 for M == 0 or invalid arguments.
 */
#define EPILORA_WORKSPACE_SYNC_BYTES 2360576
EPILORA_API size_t epilora_workspace_bytes(int fmt, int M, int K, int r);

/*
 * Bytes of device workspace with which epilora_layer_forward (and _slices,
 * _noalloc) computes the adapter term of a batch of more than 32 tokens in a
 * pass of its own (the adapter kernels the EpiLoRA page runs after the base
 * GEMM above the decode batch sizes, §Design › Timed dispatch):
 * epilora_workspace_bytes(fmt, M, K, r) plus, for M > 32 and r >= 32, an
 * fp32 buffer of M x N (256-byte rounded) placed right after the regions
 * listed there. A call with more than 32 tokens and bf16 adapters of rank 32
 * or more (per slice) whose workspace_bytes reaches this size enqueues three
 * kernels instead of two: the shrink grid, the expand pass (S . B_l for
 * every sorted row with an adapter, 128 output columns per tile, each tile
 * inside one slice) as its programmatic dependent, and the GEMM as the
 * expand pass's programmatic dependent, whose epilogue adds the fp32 term to
 * the base value before the one rounding to bf16 (the term: bf16 tensor-core
 * MMAs of the B rows with S split exactly into three bf16 parts, fp32
 * accumulation). Otherwise (rank 16, or a smaller workspace) the GEMM's
 * epilogue computes the term itself; the two agree within the arithmetic
 * bound of the method. Other shapes: the same as epilora_workspace_bytes.
 * Returns 0 for M == 0 or invalid arguments.
 */
EPILORA_API size_t epilora_layer_workspace_bytes(int fmt, int M, int N, int K, int r);

/*
 * Number of kernels epilora_layer_forward (and _slices, _fp8_adapters,
 * _noalloc) enqueues for (fmt, M, K, r), r as for epilora_workspace_bytes
 * (rank times slices, 0 without adapters), under the current decode-path
 * policy (epilora_set_decode_path): 1 when the single-kernel decode path takes
 * the call, 2 otherwise (the shrink grid with its quantizer blocks, then the
 * GEMM as its programmatic dependent), for a workspace of
 * epilora_workspace_bytes; a workspace of epilora_layer_workspace_bytes adds
 * the expand pass (3) where that size exceeds epilora_workspace_bytes. The single kernel can take a few
 * tokens: M <= 8, FP8 with M * K <= 16384 (one token up to K = 16384, four at
 * K = 4096), NVFP4 with the bf16 rows within 40 KB (one token up to
 * K = 16384, two at K = 8192), as long as the shared memory of the call
 * leaves room for two weight stages (large M * r excludes it); the automatic
 * policy gives it the FP8 calls only. Returns 0 for invalid arguments.
 */
EPILORA_API int epilora_layer_forward_kernels(int fmt, int M, int K, int r);

/*
 * Decode-path policy for all later calls in the process (calls already
 * enqueued are not affected): which path epilora_layer_forward (and _slices,
 * _fp8_adapters, _noalloc) takes for calls the single kernel can run.
 *   EPILORA_DECODE_PATH_AUTO (the default): the single kernel for FP8 bases,
 *     the shrink grid and the GEMM for NVFP4 bases (on GB300 each is the
 *     faster of the two for its format at one token on the 8B layer);
 *   EPILORA_DECODE_PATH_SINGLE: the single kernel wherever it can run;
 *   EPILORA_DECODE_PATH_TWO: the shrink grid and the GEMM always.
 * Results agree between the paths within the arithmetic bound of the
 * method (the adapter term and the split-K sums are added in a different
 * order). Returns the previous policy, or EPILORA_ERR_INVALID_ARG (policy
 * unchanged) for another value.
 */
#define EPILORA_DECODE_PATH_AUTO 0
#define EPILORA_DECODE_PATH_SINGLE 1
#define EPILORA_DECODE_PATH_TWO 2
EPILORA_API int epilora_set_decode_path(int policy);

/*
 * Fused one-call layer (the decode path of the EpiLoRA page, §Design ›
 * Multi-adapter kernels › The decode path).
 *
 * A few tokens (epilora_layer_forward_kernels == 1) run as ONE persistent
 * kernel, a programmatic dependent of the previous kernel on the stream: it
 * streams Wq (and w_block_scale) at once, waits for that kernel, then every
 * thread block quantizes the activations (the arithmetic of
 * epilora_quant_act) over the K range of its own weight units, takes a fixed
 * share of the shrink work items (token, 4 ranks, K slice: the arithmetic of
 * epilora_lora_shrink split into partial sums), and finishes its share of
 * the output; the weight stream is split evenly over the SMs, a weight tile
 * split between thread blocks being summed in a fixed order. It lets the
 * next kernel on the stream launch as soon as all its thread blocks run.
 * Otherwise it enqueues two kernels,
 *   1. the shrink grid (the arithmetic of epilora_lora_shrink, split over K
 *      slices into partial sums; for more than 32 tokens, blocks of 16
 *      consecutive tokens carrying at most two adapters on the tensor
 *      cores) plus quantizer CTAs (the arithmetic of epilora_quant_act; for
 *      more than 32 tokens with adapters the rows of Xq are written in
 *      adapter-sorted order), launched as a programmatic dependent of the
 *      previous kernel on the stream: it lets the GEMM launch when its CTAs
 *      start (decode batches, or a grid that fits the GPU) or as they
 *      finish, and waits for that kernel's completion before reading
 *      anything, and
 *   2. the GEMM of epilora_gemm_lora_epilogue as its programmatic dependent:
 *      it starts streaming Wq (and w_block_scale) as soon as it is resident,
 *      and reads everything else only after the shrink grid has completed;
 * using `workspace` (>= epilora_workspace_bytes, 256-byte aligned) for the
 * head, Xq, scales, S and the row map; with more than 32 tokens, adapters and
 * a workspace of epilora_layer_workspace_bytes, the expand pass runs between
 * the two (see there). The head (the first
 * EPILORA_WORKSPACE_SYNC_BYTES) must be zero before the first call that uses
 * the workspace: zero-fill a workspace once after allocating it. Calls keep
 * the head valid for the next call (each adds 256 to a 64-bit launch
 * counter at bytes [16, 24) of the head, whose value at the start of a call
 * gives the tag of every value its thread blocks exchange, so older values
 * are never taken for new ones); nothing else needs an initial value. Y is the
 * same whatever the row order. Calls that share a workspace must be ordered
 * on one stream.
 * Because the GEMM may start while the kernel that precedes this call on the
 * stream is still running, that kernel must not write Wq or w_block_scale
 * (every other input, X included, may be its output).
 * A == NULL or B == NULL computes the base layer only. Graph-capturable: it
 * makes no allocation and no synchronizing call.
 */
EPILORA_API int epilora_layer_forward(int fmt, int M, int N, int K,
                          const void* X, int ldx,
                          const void* Wq, const float* w_scale,
                          const uint8_t* w_block_scale, const float* w_global_scale,
                          const float* x_global_scale,
                          const void* A, const void* B, int L, int r,
                          const int32_t* idx, const uint8_t* mask,
                          void* Y, int ldy,
                          void* workspace, size_t workspace_bytes,
                          int* status_dev, void* stream);

/*
 * Multi-slice projection (the EpiLoRA page, §Design › Multi-adapter kernels:
 * fused projections such as qkv or gate_up carry one adapter per slice):
 * epilora_layer_forward where output columns [slice_end[s-1], slice_end[s])
 * (slice_end[-1] = 0) take slice s's own rank-r adapter pair. A is bf16
 * [L, n_slices * r, K] (slice s's A rows at [s*r, (s+1)*r)), B stays
 * [L, N, r] (row n belongs to its column's slice). n_slices in 1..4;
 * slice_end (host memory, read during the call) ascending, every end but the
 * last a multiple of 128, the last == N. The workspace must hold
 * epilora_workspace_bytes(fmt, M, K, n_slices * r) bytes (with
 * epilora_layer_workspace_bytes(fmt, M, N, K, n_slices * r), batches of more
 * than 32 tokens take the expand pass). idx / mask select
 * one adapter slot per token for all slices. Other arguments and errors as
 * epilora_layer_forward (A and B are required).
 */
EPILORA_API int epilora_layer_forward_slices(int fmt, int M, int N, int K,
                          const void* X, int ldx,
                          const void* Wq, const float* w_scale,
                          const uint8_t* w_block_scale, const float* w_global_scale,
                          const float* x_global_scale,
                          const void* A, const void* B, int L, int r,
                          int n_slices, const int* slice_end,
                          const int32_t* idx, const uint8_t* mask,
                          void* Y, int ldy,
                          void* workspace, size_t workspace_bytes,
                          int* status_dev, void* stream);

/*
 * Stored FP8 adapters (EpiLoRA page, §Design › Multi-adapter kernels › K1
 * and K2: adapters may be kept in FP8 and are dequantized in registers):
 * epilora_layer_forward with the adapter tables as E4M3 codes and one fp32
 * scale per row,
 *   Aq uint8 [L, r, K], a_scale fp32 [L, r]   (rank j of adapter l over K)
 *   Bq uint8 [L, N, r], b_scale fp32 [L, N]   (output n of adapter l over r)
 *   S[t, j] = a_scale[l, j] * sum_k X[t, k] * E4M3(Aq[l, j, k])   (l = idx_t)
 *   d[t, n] = b_scale[l, n] * sum_j S[t, j] * E4M3(Bq[l, n, j])
 * (the codes and scales of each row as epilora_quant_act gives them for the
 * row). About half the adapter bytes of bf16 tables; the page reports that
 * part of its accuracy checks with stored adapters failed, so this is an
 * option for the caller, not a default. Decode batches only: M <= 32, else
 * EPILORA_ERR_UNSUPPORTED. Workspace as epilora_layer_forward (r as given);
 * other arguments, results and errors as there (all four adapter pointers
 * required).
 */
EPILORA_API int epilora_layer_forward_fp8_adapters(int fmt, int M, int N, int K,
                          const void* X, int ldx,
                          const void* Wq, const float* w_scale,
                          const uint8_t* w_block_scale, const float* w_global_scale,
                          const float* x_global_scale,
                          const uint8_t* Aq, const float* a_scale,
                          const uint8_t* Bq, const float* b_scale, int L, int r,
                          const int32_t* idx, const uint8_t* mask,
                          void* Y, int ldy,
                          void* workspace, size_t workspace_bytes,
                          int* status_dev, void* stream);

/*
 * Test hook of the single-kernel decode path: with on != 0, later calls that
 * take that path (in this process) have their shrink work items publish
 * nothing, so every finishing thread block that needs S waits until its
 * bounded wait runs out (1 s), records EPILORA_ERR_TIMEOUT in the status
 * word and returns in order (Y is then unspecified). on = 0 restores normal
 * operation. Not for production use; returns EPILORA_OK.
 */
EPILORA_API int epilora_test_drop_shrink_results(int on);

/*
 * epilora_layer_forward without a caller workspace. The EpiLoRA page has no
 * counterpart of this entry point: it serves callers that cannot hand the
 * library device memory, such as a plain C host with no device allocator of
 * its own, or code at a point where entering an allocator is not allowed (an
 * allocator's own hook, a section that must not call cudaMalloc).
 *
 * It allocates nothing. Its scratch is a fixed array of
 * EPILORA_NOALLOC_SCRATCH_BYTES bytes of static device storage inside the
 * library, one per device. The first call on a device (the device current
 * at the call) looks up that array's address with cudaGetSymbolAddress; make
 * that first call before any stream capture. Arguments, layout, results and
 * status codes are those of epilora_layer_forward without the workspace.
 *
 * Returns EPILORA_ERR_WORKSPACE, having enqueued nothing, when
 * epilora_workspace_bytes(fmt, M, K, A && B ? r : 0) exceeds
 * EPILORA_NOALLOC_SCRATCH_BYTES (8 MiB); the test is exactly that size query,
 * whose S term grows with the number of K slices of the shrink (e.g. FP8,
 * r = 64: M up to 1175 at K = 4096); EPILORA_ERR_CUDA if the address lookup
 * fails.
 * Otherwise it enqueues what epilora_layer_forward enqueues given a workspace
 * of the whole scratch (the scratch starts zeroed when the library is
 * loaded, which is what epilora_layer_forward requires of a workspace's
 * head): batches of more than 32 tokens with rank >= 32 take the expand pass
 * whenever epilora_layer_workspace_bytes fits the scratch.
 *
 * All calls on one device share the one scratch array: calls that overlap in
 * time (on different streams, or from host threads that do not order their
 * streams) race on it and produce wrong results. Order them on one stream.
 */
#define EPILORA_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
EPILORA_API int epilora_layer_forward_noalloc(int fmt, int M, int N, int K,
                          const void* X, int ldx,
                          const void* Wq, const float* w_scale,
                          const uint8_t* w_block_scale, const float* w_global_scale,
                          const float* x_global_scale,
                          const void* A, const void* B, int L, int r,
                          const int32_t* idx, const uint8_t* mask,
                          void* Y, int ldy,
                          int* status_dev, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* EPILORA_H_ */
