// epilora_layer_forward_noalloc: the fused layer with its scratch in the
// library's own static device memory instead of a caller workspace.
//
// Some callers cannot hand the library device memory: a plain C host with no
// device allocator of its own, or code at a point where entering an
// allocator is not allowed (an allocator's own hook, a section that must not
// call cudaMalloc). For them this entry point allocates nothing: its scratch
// is a fixed array of static device storage, one instance per device (each
// device's module image holds its own), whose address is looked up once per
// device. It then enqueues exactly what epilora_layer_forward enqueues.
#include <mutex>

#include "common.cuh"

namespace epi {
namespace {

constexpr size_t kScratchBytes = EPILORA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Static device storage, never freed; every byte is written before it is read.
__device__ __align__(256) unsigned char g_layer_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Address of this device's scratch (device current at the call), looked up
// on the first call per device. Returns nullptr if the lookup fails.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t rc = cudaGetSymbolAddress(&p, g_layer_scratch);
    if (rc != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();   // do not leave the lookup's error pending
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace epi

EPILORA_API int epilora_layer_forward_noalloc(int fmt, int M, int N, int K, const void* X, int ldx, const void* Wq,
                                              const float* w_scale, const uint8_t* w_block_scale,
                                              const float* w_global_scale, const float* x_global_scale,
                                              const void* A, const void* B, int L, int r, const int32_t* idx,
                                              const uint8_t* mask, void* Y, int ldy, int* status_dev,
                                              void* stream) {
  const bool adapters = A != nullptr && B != nullptr;
  if (M < 0) return EPILORA_ERR_INVALID_ARG;
  if (M == 0) return epilora_layer_forward(fmt, M, N, K, X, ldx, Wq, w_scale, w_block_scale, w_global_scale,
                                           x_global_scale, A, B, L, r, idx, mask, Y, ldy, nullptr, 0, status_dev,
                                           stream);
  const size_t need = epilora_workspace_bytes(fmt, M, K, adapters ? r : 0);
  if (need == 0) return EPILORA_ERR_INVALID_ARG;          // fmt / K / r rejected by the size query
  if (need > epi::kScratchBytes) return EPILORA_ERR_WORKSPACE;
  void* scratch = epi::scratch_for_current_device();
  if (scratch == nullptr) return EPILORA_ERR_CUDA;
  return epilora_layer_forward(fmt, M, N, K, X, ldx, Wq, w_scale, w_block_scale, w_global_scale, x_global_scale, A,
                               B, L, r, idx, mask, Y, ldy, scratch, epi::kScratchBytes, status_dev, stream);
}
