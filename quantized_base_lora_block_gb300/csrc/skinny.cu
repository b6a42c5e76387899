// Skinny rank-r contractions of the LoRA adapter path (r <= 64):
//
//   row-reduce  out[p, q] = sum_j L[p, j] * S(j, q)     T = X A^T, U = dY B
//   col-reduce  out[j, q] = sum_p L[p, j] * S[p, q]     dB = dY^T T, dA^T = X^T U
//
// L is the long operand (X or dY, [P x J] bf16 row-major) and is streamed
// from HBM exactly once; S is small and stays in L2.  These are HBM-bound
// (r flops per byte of L), so they use warp-level mma.sync tiles fed by
// cp.async rather than the tcgen05 pipeline of the big GEMMs.  Each split of
// the reduction writes fp32 partial sums; a finalize kernel adds the splits in
// a fixed order, so results are bitwise reproducible run to run.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "warp_mma.cuh"

namespace qlora {

namespace {

constexpr int TP = 64;       // rows of L per tile
constexpr int TJ = 64;       // columns of L per tile
constexpr int LPITCH = 72;   // padded smem row pitch of an L tile (elements)
constexpr int NTHR = 128;
using namespace wmma16;

}  // namespace

// ---------------------------------------------------------------------------
// Row-reduce.  grid = (ceil(P/64), splits); block = 128 (warp w owns rows
// 16w..16w+15 of the CTA's 64-row tile and all Q columns).
//   S_QJ = true : S given as [Q x J] (j contiguous), e.g. A [r x K]
//   S_QJ = false: S given as [J x Q] (q contiguous), e.g. B [N x r]
// partial: fp32 [splits][P][Q].
// Grouped rows: with `tiles` non-null, CTA x handles tiles[x] = (group g,
// first row, row count) and uses S + g * s_stride (the group's adapter).
// ---------------------------------------------------------------------------
template <int Q, bool S_QJ>
__global__ void __launch_bounds__(NTHR) rr_kernel(const __nv_bfloat16* __restrict__ L, int64_t P, int64_t J,
                                                  const __nv_bfloat16* __restrict__ S, float* __restrict__ partial,
                                                  int64_t jc, const int4* __restrict__ tiles, int64_t s_stride) {
  constexpr int SP = S_QJ ? LPITCH : (Q + 8);           // smem pitch of S tile
  constexpr int S_ELEMS = S_QJ ? Q * LPITCH : TJ * (Q + 8);
  __shared__ __align__(128) __nv_bfloat16 sL[2][TP * LPITCH];
  __shared__ __align__(128) __nv_bfloat16 sS[2][S_ELEMS];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int64_t p0 = (int64_t)blockIdx.x * TP, p_lim = P;
  if (tiles != nullptr) {
    const int4 tl = tiles[blockIdx.x];
    p0 = tl.y;
    p_lim = (int64_t)tl.y + tl.z;
    S += (int64_t)tl.x * s_stride;
  }
  const int64_t j_begin = (int64_t)blockIdx.y * jc;
  const int64_t j_end = min(J, j_begin + jc);
  const int nchunks = (int)((j_end - j_begin + TJ - 1) / TJ);

  auto load_chunk = [&](int buf, int64_t j0) {
    // L tile: 64 rows x 64 cols = 512 16-byte pieces, 4 per thread
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int piece = tid + i * NTHR;
      const int r = piece >> 3, c8 = (piece & 7) * 8;
      const bool ok = (p0 + r) < p_lim;
      const __nv_bfloat16* src = L + (ok ? (p0 + r) : 0) * J + j0 + c8;
      cp_async16(s_addr(&sL[buf][r * LPITCH + c8]), src, ok);
    }
    if (S_QJ) {  // Q rows x 64 cols
      for (int piece = tid; piece < Q * 8; piece += NTHR) {
        const int r = piece >> 3, c8 = (piece & 7) * 8;
        cp_async16(s_addr(&sS[buf][r * SP + c8]), S + (int64_t)r * J + j0 + c8, true);
      }
    } else {  // 64 rows x Q cols
      for (int piece = tid; piece < TJ * (Q / 8); piece += NTHR) {
        const int r = piece / (Q / 8), c8 = (piece % (Q / 8)) * 8;
        cp_async16(s_addr(&sS[buf][r * SP + c8]), S + (j0 + r) * Q + c8, true);
      }
    }
  };

  float acc[Q / 8][4];
#pragma unroll
  for (int t = 0; t < Q / 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  if (nchunks > 0) load_chunk(0, j_begin);
  cp_async_commit();
  for (int ch = 0; ch < nchunks; ++ch) {
    const int buf = ch & 1;
    if (ch + 1 < nchunks) load_chunk(buf ^ 1, j_begin + (int64_t)(ch + 1) * TJ);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TJ / 16; ++kk) {
      uint32_t a[4];
      {
        const int i = lane >> 3;
        const int row = warp * 16 + (i & 1) * 8 + (lane & 7);
        const int col = kk * 16 + (i >> 1) * 8;
        ldsm_x4(s_addr(&sL[buf][row * LPITCH + col]), a[0], a[1], a[2], a[3]);
      }
#pragma unroll
      for (int nt = 0; nt + 1 < Q / 8; nt += 2) {  // two n8 tiles at a time
        uint32_t b0, b1, b2, b3;
        const int i = lane >> 3;
        if (S_QJ) {
          const int q = nt * 8 + (i >> 1) * 8 + (lane & 7);
          const int j = kk * 16 + (i & 1) * 8;
          ldsm_x4(s_addr(&sS[buf][q * SP + j]), b0, b1, b2, b3);
        } else {
          const int j = kk * 16 + (i & 1) * 8 + (lane & 7);
          const int q = nt * 8 + (i >> 1) * 8;
          ldsm_x4_t(s_addr(&sS[buf][j * SP + q]), b0, b1, b2, b3);
        }
        mma_bf16_16816(acc[nt], a, b0, b1);
        mma_bf16_16816(acc[nt + 1], a, b2, b3);
      }
      if (Q % 16 == 8) {  // last single n8 tile
        constexpr int nt = Q / 8 - 1;
        uint32_t b0, b1;
        const int i = (lane >> 3) & 1;
        if (S_QJ) {
          ldsm_x2(s_addr(&sS[buf][(nt * 8 + (lane & 7)) * SP + kk * 16 + i * 8]), b0, b1);
        } else {
          ldsm_x2_t(s_addr(&sS[buf][(kk * 16 + i * 8 + (lane & 7)) * SP + nt * 8]), b0, b1);
        }
        mma_bf16_16816(acc[nt], a, b0, b1);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // write partials: c0,c1 at (row g, cols 2t, 2t+1); c2,c3 at row g+8
  float* out = partial + (int64_t)blockIdx.y * P * Q;
  const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
  for (int nt = 0; nt < Q / 8; ++nt) {
    const int q = nt * 8 + 2 * t4;
    const int64_t r0 = p0 + warp * 16 + g, r1 = r0 + 8;
    if (r0 < p_lim) *reinterpret_cast<float2*>(out + r0 * Q + q) = make_float2(acc[nt][0], acc[nt][1]);
    if (r1 < p_lim) *reinterpret_cast<float2*>(out + r1 * Q + q) = make_float2(acc[nt][2], acc[nt][3]);
  }
}

// ---------------------------------------------------------------------------
// Col-reduce.  grid = (J/64, splits); block = 128 (warp w owns columns
// 16w..16w+15 of the CTA's 64-column tile).  S is fp32 [P x Q]; it is split
// on the fly into S_hi = bf16(S) and S_lo = bf16(S - S_hi), stored side by
// side as a [P x 2Q] bf16 tile, so the tensor-core products keep ~16
// significant bits of S.  partial: fp32 [splits][J][2Q] (hi half, lo half).
// ---------------------------------------------------------------------------
// Grouped rows: with `chunks` non-null, split y covers rows
// [chunks[y].y, chunks[y].z) (one group's rows) instead of [y pc, (y+1) pc).
template <int Q>
__global__ void __launch_bounds__(NTHR) cr_kernel(const __nv_bfloat16* __restrict__ L, int64_t P, int64_t J,
                                                  const float* __restrict__ S, float* __restrict__ partial,
                                                  int64_t pc, const int4* __restrict__ chunks) {
  constexpr int Q2 = 2 * Q;
  constexpr int SP = Q2 + 8;
  extern __shared__ __align__(128) uint8_t cr_smem[];
  typedef __nv_bfloat16 LTile[TP * LPITCH];
  typedef __nv_bfloat16 STile[TP * SP];
  LTile* sL = reinterpret_cast<LTile*>(cr_smem);
  STile* sS = reinterpret_cast<STile*>(cr_smem + 2 * sizeof(LTile));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t j0 = (int64_t)blockIdx.x * TJ;
  int64_t p_begin = (int64_t)blockIdx.y * pc;
  int64_t p_end = min(P, p_begin + pc);
  if (chunks != nullptr) {
    const int4 ch = chunks[blockIdx.y];
    p_begin = ch.y;
    p_end = ch.z;
  }
  const int nchunks = (int)((p_end - p_begin + TP - 1) / TP);

  auto load_chunk = [&](int buf, int64_t pp) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int piece = tid + i * NTHR;
      const int r = piece >> 3, c8 = (piece & 7) * 8;
      const bool ok = (pp + r) < p_end;
      cp_async16(s_addr(&sL[buf][r * LPITCH + c8]), L + (ok ? (pp + r) : 0) * J + j0 + c8, ok);
    }
    for (int piece = tid; piece < TP * (Q / 4); piece += NTHR) {
      const int r = piece / (Q / 4), c4 = (piece % (Q / 4)) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if ((pp + r) < p_end) v = *reinterpret_cast<const float4*>(S + (pp + r) * Q + c4);
      const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(f[k]);
        const __nv_bfloat16 lo = __float2bfloat16_rn(f[k] - __bfloat162float(hi));
        sS[buf][r * SP + c4 + k] = hi;
        sS[buf][r * SP + Q + c4 + k] = lo;
      }
    }
  };

  float acc[Q2 / 8][4];
#pragma unroll
  for (int t = 0; t < Q2 / 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  if (nchunks > 0) load_chunk(0, p_begin);
  cp_async_commit();
  for (int ch = 0; ch < nchunks; ++ch) {
    const int buf = ch & 1;
    if (ch + 1 < nchunks) load_chunk(buf ^ 1, p_begin + (int64_t)(ch + 1) * TP);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TP / 16; ++kk) {
      uint32_t a[4];
      {  // A = L^T (m = j, k = p) from the [p][j] tile, transposed load
        const int i = lane >> 3;
        const int p = kk * 16 + (i >> 1) * 8 + (lane & 7);
        const int j = warp * 16 + (i & 1) * 8;
        ldsm_x4_t(s_addr(&sL[buf][p * LPITCH + j]), a[0], a[1], a[2], a[3]);
      }
#pragma unroll
      for (int nt = 0; nt < Q2 / 8; nt += 2) {  // Q2 is a multiple of 16
        uint32_t b0, b1, b2, b3;
        const int i = lane >> 3;
        const int p = kk * 16 + (i & 1) * 8 + (lane & 7);
        const int q = nt * 8 + (i >> 1) * 8;
        ldsm_x4_t(s_addr(&sS[buf][p * SP + q]), b0, b1, b2, b3);
        mma_bf16_16816(acc[nt], a, b0, b1);
        mma_bf16_16816(acc[nt + 1], a, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  float* out = partial + (int64_t)blockIdx.y * J * Q2;
  const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
  for (int nt = 0; nt < Q2 / 8; ++nt) {
    const int q = nt * 8 + 2 * t4;
    const int64_t r0 = j0 + warp * 16 + g, r1 = r0 + 8;
    *reinterpret_cast<float2*>(out + r0 * Q2 + q) = make_float2(acc[nt][0], acc[nt][1]);
    *reinterpret_cast<float2*>(out + r1 * Q2 + q) = make_float2(acc[nt][2], acc[nt][3]);
  }
}

// ---------------------------------------------------------------------------
// Finalize: add the splits in order.
//   rows: v = sum_s partial[s][p][q];  out_f32 = v, out_scaled =
//         bf16(scale * v) (either may be null).
//   cols: v = scale * (sum_s hi[s][j][q] + sum_s lo[s][j][q]);  out[j][q], or
//         out[q][j] when transposed (fp32).
// ---------------------------------------------------------------------------
__global__ void fin_rows_kernel(const float* __restrict__ partial, int splits, int64_t PQ, float scale,
                                float* __restrict__ out_f32, __nv_bfloat16* __restrict__ out_scaled) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < PQ; i += (int64_t)gridDim.x * blockDim.x) {
    float v = 0.f;
    for (int s = 0; s < splits; ++s) v += partial[(int64_t)s * PQ + i];
    if (out_f32) out_f32[i] = v;
    if (out_scaled) out_scaled[i] = __float2bfloat16_rn(v * scale);
  }
}

// partial rows hold [hi-half products | lo-half products] (2Q columns)
__global__ void fin_cols_kernel(const float* __restrict__ partial, int splits, int64_t J, int Q, float scale,
                                float* __restrict__ out, int transposed) {
  const int64_t JQ = J * Q;
  const int64_t JQ2 = 2 * JQ;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < JQ; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = i / Q, q = i % Q;
    const int64_t o = j * 2 * Q + q;
    float hi = 0.f, lo = 0.f;
    for (int s = 0; s < splits; ++s) {
      hi += partial[(int64_t)s * JQ2 + o];
      lo += partial[(int64_t)s * JQ2 + o + Q];
    }
    float v = (hi + lo) * scale;
    if (transposed) {
      out[q * J + j] = v;
    } else {
      out[i] = v;
    }
  }
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
template <int Q>
static cudaError_t launch_rr_q(const __nv_bfloat16* L, int64_t P, int64_t J, const __nv_bfloat16* S, bool s_qj,
                               float* partial, const SplitPlan& sp, cudaStream_t st, const int4* tiles,
                               int ntiles, int64_t s_stride) {
  dim3 grid((unsigned)(tiles ? ntiles : (P + TP - 1) / TP), (unsigned)sp.splits);
  if (grid.x == 0) return cudaSuccess;
  if (s_qj)
    rr_kernel<Q, true><<<grid, NTHR, 0, st>>>(L, P, J, S, partial, sp.chunk, tiles, s_stride);
  else
    rr_kernel<Q, false><<<grid, NTHR, 0, st>>>(L, P, J, S, partial, sp.chunk, tiles, s_stride);
  return cudaGetLastError();
}

template <int Q>
static cudaError_t launch_cr_q(const __nv_bfloat16* L, int64_t P, int64_t J, const float* S, float* partial,
                               const SplitPlan& sp, cudaStream_t st, const int4* chunks) {
  constexpr size_t smem = 2 * sizeof(__nv_bfloat16) * (TP * LPITCH + TP * (2 * Q + 8));
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(cr_kernel<Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid((unsigned)(J / TJ), (unsigned)sp.splits);
  if (grid.y == 0) return cudaSuccess;
  cr_kernel<Q><<<grid, NTHR, smem, st>>>(L, P, J, S, partial, sp.chunk, chunks);
  return cudaGetLastError();
}

#define QLORA_RANK_DISPATCH(FN, ...)          \
  switch (Q) {                                \
    case 8: return FN<8>(__VA_ARGS__);        \
    case 16: return FN<16>(__VA_ARGS__);      \
    case 24: return FN<24>(__VA_ARGS__);      \
    case 32: return FN<32>(__VA_ARGS__);      \
    case 40: return FN<40>(__VA_ARGS__);      \
    case 48: return FN<48>(__VA_ARGS__);      \
    case 56: return FN<56>(__VA_ARGS__);      \
    case 64: return FN<64>(__VA_ARGS__);      \
    default: return cudaErrorInvalidValue;    \
  }

cudaError_t launch_row_reduce(const __nv_bfloat16* L, int64_t P, int64_t J, const __nv_bfloat16* S, int Q,
                              bool s_qj, float* partial, const SplitPlan& sp, cudaStream_t st, const int4* tiles,
                              int ntiles, int64_t s_stride) {
  count_launch(1);
  QLORA_RANK_DISPATCH(launch_rr_q, L, P, J, S, s_qj, partial, sp, st, tiles, ntiles, s_stride)
}

cudaError_t launch_col_reduce(const __nv_bfloat16* L, int64_t P, int64_t J, const float* S, int Q,
                              float* partial, const SplitPlan& sp, cudaStream_t st, const int4* chunks) {
  count_launch(1);
  QLORA_RANK_DISPATCH(launch_cr_q, L, P, J, S, partial, sp, st, chunks)
}

// Grouped finalize: out[g] = scale * sum of the hi/lo partials of chunks
// chunk_first[g] .. chunk_first[g+1]-1 (zero for a group without rows);
// out[g] is [J x Q] at out + g * J * Q, or [Q x J] when transposed.
__global__ void fin_cols_grouped_kernel(const float* __restrict__ partial, const int* __restrict__ chunk_first,
                                        int64_t J, int Q, float scale, float* __restrict__ out, int transposed) {
  const int g = blockIdx.y;
  const int c0 = chunk_first[g], c1 = chunk_first[g + 1];
  const int64_t JQ = J * Q, JQ2 = 2 * JQ;
  float* og = out + (int64_t)g * JQ;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < JQ; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = i / Q, q = i % Q;
    const int64_t o = j * 2 * Q + q;
    float hi = 0.f, lo = 0.f;
    for (int c = c0; c < c1; ++c) {
      hi += partial[(int64_t)c * JQ2 + o];
      lo += partial[(int64_t)c * JQ2 + o + Q];
    }
    const float v = (hi + lo) * scale;
    if (transposed)
      og[q * J + j] = v;
    else
      og[i] = v;
  }
}

cudaError_t launch_fin_cols_grouped(const float* partial, const int* chunk_first, int groups, int64_t J, int Q,
                                    float scale, float* out, bool transposed, cudaStream_t st) {
  if (groups <= 0) return cudaSuccess;
  count_launch(1);
  int64_t b = (J * Q + 255) / 256;
  dim3 grid((unsigned)(b < 64 ? b : 64), (unsigned)groups);
  fin_cols_grouped_kernel<<<grid, 256, 0, st>>>(partial, chunk_first, J, Q, scale, out, transposed ? 1 : 0);
  return cudaGetLastError();
}

static unsigned fin_grid(int64_t n) {
  int64_t b = (n + 255) / 256;
  return (unsigned)(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

cudaError_t launch_fin_rows(const float* partial, int splits, int64_t P, int Q, float scale, float* out_f32,
                            __nv_bfloat16* out_scaled, cudaStream_t st) {
  count_launch(1);
  fin_rows_kernel<<<fin_grid(P * Q), 256, 0, st>>>(partial, splits, P * Q, scale, out_f32, out_scaled);
  return cudaGetLastError();
}

cudaError_t launch_fin_cols(const float* partial, int splits, int64_t J, int Q, float scale, float* out,
                            bool transposed, cudaStream_t st) {
  count_launch(1);
  fin_cols_kernel<<<fin_grid(J * Q), 256, 0, st>>>(partial, splits, J, Q, scale, out, transposed ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace qlora
