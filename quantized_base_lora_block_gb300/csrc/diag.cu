// Diagnostics of the bounded device waits.
//
// Every wait inside this library's kernels gives up after a time limit,
// records QLORA_ERR_TIMEOUT in the device error word and lets the kernel
// return, so a broken protocol ends as an error status instead of a hung GPU.
// qlora_selftest_bounded_wait exercises that path on purpose: one warp waits,
// with a caller-chosen short limit, on an mbarrier phase that nothing ever
// completes.  The wait runs out, the kernel records the timeout and returns;
// the context stays usable and qlora_last_device_error() reports the status.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/qlora.h"
#include "kernels.h"
#include "ptx.cuh"

namespace qlora {

__global__ void bounded_wait_probe_kernel(uint64_t limit_ns, int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // expects one arrival that never comes
    abort = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_for(smem_u32(&bar), 0, &abort, err, limit_ns);
  __syncthreads();
}

}  // namespace qlora

extern "C" int32_t qlora_selftest_bounded_wait(int64_t limit_ns, void* stream) {
  // a short limit only: this is a test of the error path, not a way to stall
  if (limit_ns <= 0 || limit_ns > 1000000000ll) return QLORA_ERR_INVALID;
  int* err = qlora::device_error_word();
  if (!err) return QLORA_ERR_CUDA;
  qlora::count_launch(1);
  qlora::bounded_wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_ns, err);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}
