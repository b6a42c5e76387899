// Elementwise parts of gate / up with the SwiGLU activation, H = silu(G) U
// with silu(g) = g sigmoid(g) (the MLP of the Llama and Qwen3 layers):
//   swiglu_act_kernel   H from G | U (used where the GEMM epilogue does not
//                       compute it: launches of at most 128 rows);
//   swiglu_grad_kernel  dY = [dG | dU] from dH and G | U, in fp32:
//                       dG = dH U sigmoid(G) (1 + G (1 - sigmoid(G))), dU = dH silu(G).
// Eight bf16 per thread and row (16-byte streaming loads and stores).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace qlora {

namespace {

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}


}  // namespace

// Grid: x over the row's 8-element groups (blockDim.x each), y over rows;
// each thread takes two rows per step, both rows' loads issued before the
// arithmetic.
__device__ __forceinline__ uint4 ldg_stream(const __nv_bfloat16* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

__global__ void swiglu_act_kernel(const __nv_bfloat16* __restrict__ GU, __nv_bfloat16* __restrict__ H, int64_t M,
                                  int64_t I) {
  const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (c >= I) return;
  for (int64_t m = blockIdx.y; m < M; m += gridDim.y) {
    float g[8], u[8], h[8];
    unpack8(ldg_stream(GU + m * 2 * I + c), g);
    unpack8(ldg_stream(GU + m * 2 * I + I + c), u);
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = swiglu_h_f32(g[k], u[k]);
    __stcs(reinterpret_cast<uint4*>(H + m * I + c), pack8(h));
  }
}

__global__ void swiglu_grad_kernel(const __nv_bfloat16* __restrict__ GU, const __nv_bfloat16* __restrict__ dH,
                                   __nv_bfloat16* __restrict__ dY, int64_t M, int64_t I) {
  const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (c >= I) return;
  const int64_t step = gridDim.y;
  for (int64_t m0 = blockIdx.y; m0 < M; m0 += 2 * step) {
    const int64_t m1 = m0 + step;
    const bool two = m1 < M;
    uint4 rg[2], ru[2], rh[2];
    rg[0] = ldg_stream(GU + m0 * 2 * I + c);
    ru[0] = ldg_stream(GU + m0 * 2 * I + I + c);
    rh[0] = ldg_stream(dH + m0 * I + c);
    if (two) {
      rg[1] = ldg_stream(GU + m1 * 2 * I + c);
      ru[1] = ldg_stream(GU + m1 * 2 * I + I + c);
      rh[1] = ldg_stream(dH + m1 * I + c);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (j == 1 && !two) break;
      const int64_t m = j ? m1 : m0;
      float g[8], u[8], dh[8], dg[8], du[8];
      unpack8(rg[j], g);
      unpack8(ru[j], u);
      unpack8(rh[j], dh);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float sg = swiglu_sigmoid_f32(g[k]);
        dg[k] = dh[k] * u[k] * sg * (1.0f + g[k] * (1.0f - sg));
        du[k] = dh[k] * g[k] * sg;
      }
      __stcs(reinterpret_cast<uint4*>(dY + m * 2 * I + c), pack8(dg));
      __stcs(reinterpret_cast<uint4*>(dY + m * 2 * I + I + c), pack8(du));
    }
  }
}

// x: blocks of 256 threads covering the row's I / 8 groups; y: rows, so
// that the grid holds about 8 blocks per SM.
static dim3 ew_grid(int64_t M, int64_t I) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t gx = (I / 8 + 255) / 256;
  int64_t gy = (int64_t)sms * 8 / gx;
  if (gy > M) gy = M;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  return dim3((unsigned)gx, (unsigned)gy);
}

cudaError_t launch_swiglu_act(const __nv_bfloat16* GU, __nv_bfloat16* H, int64_t M, int64_t I, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  count_launch(1);
  swiglu_act_kernel<<<ew_grid(M, I), 256, 0, st>>>(GU, H, M, I);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_grad(const __nv_bfloat16* GU, const __nv_bfloat16* dH, __nv_bfloat16* dY, int64_t M,
                               int64_t I, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  count_launch(1);
  swiglu_grad_kernel<<<ew_grid(M, I), 256, 0, st>>>(GU, dH, dY, M, I);
  return cudaGetLastError();
}

}  // namespace qlora
