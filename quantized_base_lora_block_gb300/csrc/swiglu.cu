// Elementwise parts of gate / up with the SwiGLU activation, H = silu(G) U
// with silu(g) = g sigmoid(g) (the MLP of the Llama and Qwen3 layers):
//   swiglu_act_kernel   H from G | U (used where the GEMM epilogue does not
//                       compute it: launches of at most 128 rows);
//   swiglu_grad_kernel  dY = [dG | dU] from dH and G | U, in fp32:
//                       dG = dH U sigmoid(G) (1 + G (1 - sigmoid(G))), dU = dH silu(G).
// Eight bf16 per thread and step (16-byte loads and stores).
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

__global__ void swiglu_act_kernel(const __nv_bfloat16* __restrict__ GU, __nv_bfloat16* __restrict__ H, int64_t M,
                                  int64_t I) {
  const int64_t per_row = I / 8, n = M * per_row;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = t / per_row, c = (t % per_row) * 8;
    float g[8], u[8], h[8];
    unpack8(*reinterpret_cast<const uint4*>(GU + m * 2 * I + c), g);
    unpack8(*reinterpret_cast<const uint4*>(GU + m * 2 * I + I + c), u);
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = swiglu_h_f32(g[k], u[k]);
    *reinterpret_cast<uint4*>(H + m * I + c) = pack8(h);
  }
}

__global__ void swiglu_grad_kernel(const __nv_bfloat16* __restrict__ GU, const __nv_bfloat16* __restrict__ dH,
                                   __nv_bfloat16* __restrict__ dY, int64_t M, int64_t I) {
  const int64_t per_row = I / 8, n = M * per_row;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = t / per_row, c = (t % per_row) * 8;
    float g[8], u[8], dh[8], dg[8], du[8];
    unpack8(*reinterpret_cast<const uint4*>(GU + m * 2 * I + c), g);
    unpack8(*reinterpret_cast<const uint4*>(GU + m * 2 * I + I + c), u);
    unpack8(*reinterpret_cast<const uint4*>(dH + m * I + c), dh);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float s = swiglu_sigmoid_f32(g[k]);
      dg[k] = dh[k] * u[k] * s * (1.0f + g[k] * (1.0f - s));
      du[k] = dh[k] * g[k] * s;
    }
    *reinterpret_cast<uint4*>(dY + m * 2 * I + c) = pack8(dg);
    *reinterpret_cast<uint4*>(dY + m * 2 * I + I + c) = pack8(du);
  }
}

static unsigned ew_blocks(int64_t items) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t b = (items + 255) / 256;
  if (b > (int64_t)sms * 8) b = (int64_t)sms * 8;
  return (unsigned)(b > 0 ? b : 1);
}

cudaError_t launch_swiglu_act(const __nv_bfloat16* GU, __nv_bfloat16* H, int64_t M, int64_t I, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  count_launch(1);
  swiglu_act_kernel<<<ew_blocks(M * I / 8), 256, 0, st>>>(GU, H, M, I);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_grad(const __nv_bfloat16* GU, const __nv_bfloat16* dH, __nv_bfloat16* dY, int64_t M,
                               int64_t I, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  count_launch(1);
  swiglu_grad_kernel<<<ew_blocks(M * I / 8), 256, 0, st>>>(GU, dH, dY, M, I);
  return cudaGetLastError();
}

}  // namespace qlora
