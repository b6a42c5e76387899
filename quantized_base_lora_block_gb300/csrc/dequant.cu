// Standalone decode of a whole base weight to bf16 (HBM-bound): each thread
// decodes 64-element lines (grid-stride) with 128-bit loads of the quantised
// bytes and writes 128 contiguous bytes of bf16 per line.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace qlora {

template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(const WeightView wv, int64_t lines, uint4* __restrict__ out) {
  for (int64_t ln = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; ln < lines;
       ln += (int64_t)gridDim.x * blockDim.x) {
    RawLine r;
    load_line<FMT>(wv, ln, r);
    uint4 o[8];
    decode_line<FMT>(r, wv, o);
    uint4* dst = out + ln * 8;
#pragma unroll
    for (int c = 0; c < 8; ++c) dst[c] = o[c];
  }
}

cudaError_t launch_dequant(int fmt, const WeightView& wv, int64_t lines, __nv_bfloat16* out, cudaStream_t st) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (lines + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  uint4* o = reinterpret_cast<uint4*>(out);
  count_launch(1);
  switch (fmt) {
    case FMT_NF4: dequant_kernel<FMT_NF4><<<(unsigned)blocks, 256, 0, st>>>(wv, lines, o); break;
    case FMT_Q8_0: dequant_kernel<FMT_Q8_0><<<(unsigned)blocks, 256, 0, st>>>(wv, lines, o); break;
    case FMT_Q4_0: dequant_kernel<FMT_Q4_0><<<(unsigned)blocks, 256, 0, st>>>(wv, lines, o); break;
    case FMT_Q4_K: dequant_kernel<FMT_Q4_K><<<(unsigned)blocks, 256, 0, st>>>(wv, lines, o); break;
    case FMT_FP8: dequant_kernel<FMT_FP8><<<(unsigned)blocks, 256, 0, st>>>(wv, lines, o); break;
    case FMT_NVFP4: dequant_kernel<FMT_NVFP4><<<(unsigned)blocks, 256, 0, st>>>(wv, lines, o); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace qlora
