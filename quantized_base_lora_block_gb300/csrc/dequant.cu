// Standalone decode of a whole base weight to bf16 (HBM-bound).  A block of
// 256 threads decodes 256 consecutive 64-element lines, one per thread, with
// 128-bit loads of the quantised bytes; their bf16 output is one contiguous
// 32 KB run, staged in shared memory and written with one bulk copy (a
// per-thread 128-byte store pattern kept the memory instruction queue full
// at ~2.9 TB/s).  Two staging buffers alternate so a block's store overlaps
// its next lines' decode.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace qlora {

namespace {
constexpr int kDqThreads = 256;
constexpr int kDqBuf = kDqThreads * 128;  // bytes of one staging buffer
}  // namespace

template <int FMT>
__global__ void __launch_bounds__(kDqThreads) dequant_kernel(const WeightView wv, int64_t lines,
                                                            uint4* __restrict__ out) {
  extern __shared__ __align__(128) uint8_t dq_smem[];
  const int t = threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kDqThreads;
  // the next iteration's line is loaded before this one is decoded, so two
  // lines' loads are in flight per thread
  int64_t base = (int64_t)blockIdx.x * kDqThreads;
  RawLine cur;
  if (base + t < lines) load_line<FMT>(wv, base + t, cur);
  for (int k = 0; base < lines; base += stride, ++k) {
    RawLine nxt;
    if (base + stride + t < lines) load_line<FMT>(wv, base + stride + t, nxt);
    const uint32_t buf = smem_u32(dq_smem) + (uint32_t)((k & 1) * kDqBuf);
    if (t == 0) bulk_wait_read1();  // the store that last read this buffer is done with it
    __syncthreads();
    if (base + t < lines) {
      uint4 o[8];
      decode_line<FMT>(cur, wv, o);
      // chunk order rotated by lane: the 8 lanes of a quarter-warp hit 8
      // different 16-byte bank groups
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int c = (q + t) & 7;
        sts_v4(buf + (uint32_t)(t * 128 + c * 16), o[c]);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (t == 0) {
      const int64_t n = lines - base < kDqThreads ? lines - base : kDqThreads;
      bulk_store_1d(out + base * 8, buf, (uint32_t)(n * 128));
      bulk_commit();
    }
    cur = nxt;
  }
  if (t == 0) bulk_wait0();
}

template <int FMT>
static cudaError_t launch_dq(const WeightView& wv, int64_t lines, uint4* o, unsigned blocks, cudaStream_t st) {
  static bool attr = false;  // per instantiation (setting it twice is harmless)
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(dequant_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * kDqBuf);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dequant_kernel<FMT><<<blocks, kDqThreads, 2 * kDqBuf, st>>>(wv, lines, o);
  return cudaGetLastError();
}

cudaError_t launch_dequant(int fmt, const WeightView& wv, int64_t lines, __nv_bfloat16* out, cudaStream_t st) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (lines + kDqThreads - 1) / kDqThreads;
  const int64_t cap = (int64_t)sms * 3;  // 64 KB of staging per block: 3 blocks per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  uint4* o = reinterpret_cast<uint4*>(out);
  count_launch(1);
  const unsigned b = (unsigned)blocks;
  switch (fmt) {
    case FMT_NF4: return launch_dq<FMT_NF4>(wv, lines, o, b, st);
    case FMT_Q8_0: return launch_dq<FMT_Q8_0>(wv, lines, o, b, st);
    case FMT_Q4_0: return launch_dq<FMT_Q4_0>(wv, lines, o, b, st);
    case FMT_Q4_K: return launch_dq<FMT_Q4_K>(wv, lines, o, b, st);
    case FMT_FP8: return launch_dq<FMT_FP8>(wv, lines, o, b, st);
    case FMT_NVFP4: return launch_dq<FMT_NVFP4>(wv, lines, o, b, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qlora
