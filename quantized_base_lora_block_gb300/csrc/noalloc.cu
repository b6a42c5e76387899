// Forward pass for callers that cannot allocate device memory.
//
// Some callers of this library have no way to obtain device memory of their
// own: for example a host program that loads this library as a plug-in and may
// only hand over the input and output buffers its host application gives it,
// or a latency-critical loop that must not call cudaMalloc because cudaMalloc
// can synchronise the whole device and stall work on other streams.  The
// regular qlora_linear_fwd needs a caller-provided workspace; this variant
// takes its workspace from a fixed array that the library keeps in device
// memory instead, and allocates nothing.
//
// The array is kNoAllocScratchBytes (16 MiB) of device memory, reserved on
// every GPU that loads this library until the process exits.  Every call of
// qlora_linear_fwd_noalloc on a device uses the same array and leaves the last
// call's intermediate values in it; two calls whose work overlaps on the GPU
// (e.g. enqueued on two different streams without ordering between them)
// race on it and may produce wrong results.  Nothing in the array has to
// start at zero: each call writes every byte it later reads.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/qlora.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device.  In host
// code the name g_noalloc_scratch is only a host-side handle; the kernel must
// receive the address returned by cudaGetSymbolAddress for the current device.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

int32_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QLORA_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return QLORA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return QLORA_OK;
}

}  // namespace

extern "C" {

size_t qlora_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int32_t qlora_linear_fwd_noalloc(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha, const void* X,
                                 const void* A, const void* B, void* Y, float* T_save, void* stream) {
  const size_t need = qlora_forward_workspace_bytes(w, M, rank);
  // invalid arguments: let the regular entry point report the precise status
  // (it validates everything before it would look at the workspace)
  if (need == 0) return qlora_linear_fwd(w, M, rank, alpha, X, A, B, Y, T_save, nullptr, 0, stream);
  if (need > kNoAllocScratchBytes) return QLORA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int32_t s = scratch_for_current_device(&scratch);
  if (s != QLORA_OK) return s;
  return qlora_linear_fwd(w, M, rank, alpha, X, A, B, Y, T_save, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
