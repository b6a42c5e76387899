// Rank-r reductions of the dense adapter path, with the split sums finished
// inside the kernel:
//
//   row reduce  out[p, q] = sum_j L[p, j] S(j, q)     T = X A^T, U = dY B
//   col reduce  out[j, q] = sum_p L[p, j] S[p, q]     dB = s dY^T T, dA^T = s X^T U
//
// L ([P x J] bf16, row-major) is streamed from HBM once, through a ring of
// 64 x 64 tiles filled by cp.async several tiles ahead of the warp-level
// mma.sync tiles that consume them.  The reduction is split over the CTAs of
// one thread-block cluster (at most 8): every CTA leaves its fp32 partial tile
// in its own shared memory, and after a cluster barrier each CTA adds a slice
// of the tile over all the cluster's CTAs in rank order (distributed shared
// memory loads) and writes the result.  The order of the sum is fixed by the
// rank, so results are bitwise reproducible run to run, and nothing but the
// result goes to global memory.
//
// The column reduction takes S as S_hi = bf16(S) and S_lo = bf16(S - S_hi)
// side by side ([P x 2Q] bf16, written by the row reduction that produces or
// passes S), so the tensor-core products keep ~16 significant bits of S; the
// finishing step adds the hi and lo sums.  One launch can carry two column
// reductions (dB and dA of the same backward call).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "warp_mma.cuh"

namespace qlora {

namespace {

constexpr int TP = 64;      // rows of L per tile
constexpr int TJ = 64;      // columns of L per tile
constexpr int LPITCH = 72;  // padded smem row pitch of an L tile (elements)
constexpr int NTHR = 128;
constexpr int kColStages = 4;  // measured: 3 and 5 stages slower (fewer bytes in flight / fewer CTAs per SM)
using namespace wmma16;

template <int Q>
struct RowStages {
  static constexpr int NS = Q <= 32 ? 4 : 3;
};

// hi = bf16(v), lo = bf16(v - hi) of 4 consecutive values; hi at dst[0..3],
// lo at dst[q_stride..q_stride+3]
__device__ __forceinline__ void store_hilo(__nv_bfloat16* dst, float4 v, int q_stride) {
  const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
  const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
  const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
  const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
  __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(dst);
  __nv_bfloat162* l2 = reinterpret_cast<__nv_bfloat162*>(dst + q_stride);
  h2[0] = h01;
  h2[1] = h23;
  l2[0] = l01;
  l2[1] = l23;
}

// 16-byte load from the shared memory of CTA `rank` of the cluster, at the
// offset of `local` in this CTA's shared memory.
__device__ __forceinline__ float4 ld_cluster_v4(const float* local, uint32_t rank) {
  const uint32_t addr = mapa_shared(s_addr(local), rank);
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

}  // namespace

// ---------------------------------------------------------------------------
// Row reduce.  grid = (ceil(P/64), splits), clusters of (1, splits); block =
// 128 (warp w owns rows 16w..16w+15 of the CTA's 64-row tile and all Q
// columns).
//   S_QJ = true : S given as [Q x J] (j contiguous), e.g. A [r x K]
//   S_QJ = false: S given as [J x Q] (q contiguous), e.g. B [N x r]
// Result: out_f32 = v and / or out_scaled = bf16(scale v).
// ---------------------------------------------------------------------------
template <int Q, bool S_QJ>
__global__ void __launch_bounds__(NTHR) rr_fin_kernel(const RowReduce jb) {
  constexpr int NS = RowStages<Q>::NS;
  constexpr int SP = S_QJ ? LPITCH : (Q + 8);  // smem pitch of the S tile
  constexpr int S_ELEMS = S_QJ ? Q * LPITCH : TJ * (Q + 8);
  extern __shared__ __align__(128) uint8_t rr_smem[];
  __nv_bfloat16* sL = reinterpret_cast<__nv_bfloat16*>(rr_smem);
  __nv_bfloat16* sS = sL + NS * TP * LPITCH;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t P = jb.P, J = jb.J;
  const int64_t j_begin = (int64_t)blockIdx.y * jb.sp.chunk;
  const int64_t j_end = min(J, j_begin + jb.sp.chunk);
  const int nchunks = j_end > j_begin ? (int)((j_end - j_begin + TJ - 1) / TJ) : 0;
  const __nv_bfloat16* __restrict__ L = jb.L;
  const __nv_bfloat16* __restrict__ S = jb.S;
  griddep_wait();
  griddep_launch_dependents();
  int64_t p0 = (int64_t)blockIdx.x * TP, p_lim = P;
  if (jb.tiles) {
    // grouped: the tile list comes from the schedule kernel earlier in the
    // stream; every CTA of the cluster has the same row tile, so a cluster
    // past the list leaves as a whole
    if ((int)blockIdx.x >= *jb.tile_count) return;
    const int4 t = jb.tiles[blockIdx.x];
    p0 = t.y;
    p_lim = (int64_t)t.y + t.z;
    S += (int64_t)t.x * jb.s_stride;
  }

  auto load_chunk = [&](int buf, int64_t j0) {
    __nv_bfloat16* dL = sL + buf * TP * LPITCH;
    __nv_bfloat16* dS = sS + buf * S_ELEMS;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // 64 x 64 tile = 512 16-byte pieces
      const int piece = tid + i * NTHR;
      const int r = piece >> 3, c8 = (piece & 7) * 8;
      const bool ok = (p0 + r) < p_lim;
      cp_async16(s_addr(dL + r * LPITCH + c8), L + (ok ? (p0 + r) : 0) * J + j0 + c8, ok);
    }
    if (S_QJ) {  // Q rows x 64 columns
      for (int piece = tid; piece < Q * 8; piece += NTHR) {
        const int r = piece >> 3, c8 = (piece & 7) * 8;
        cp_async16(s_addr(dS + r * SP + c8), S + (int64_t)r * J + j0 + c8, true);
      }
    } else if (jb.bd_nproj <= 1) {  // 64 rows x Q columns
      for (int piece = tid; piece < TJ * (Q / 8); piece += NTHR) {
        const int r = piece / (Q / 8), c8 = (piece % (Q / 8)) * 8;
        cp_async16(s_addr(dS + r * SP + c8), S + (j0 + r) * Q + c8, true);
      }
    } else {  // block-diagonal spread of B [J x bd_r]: zeros outside the row's block
      for (int piece = tid; piece < TJ * (Q / 8); piece += NTHR) {
        const int r = piece / (Q / 8), c8 = (piece % (Q / 8)) * 8;
        const int64_t j = j0 + r;
        int p = 0;
        while (p + 1 < jb.bd_nproj && j >= jb.bd_end[p]) ++p;
        const int c = c8 - p * jb.bd_r;
        const bool in = c >= 0 && c < jb.bd_r;
        cp_async16(s_addr(dS + r * SP + c8), S + j * jb.bd_r + (in ? c : 0), in);
      }
    }
  };

  float acc[Q / 8][4];
#pragma unroll
  for (int t = 0; t < Q / 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

#pragma unroll
  for (int s = 0; s < NS - 1; ++s) {
    if (s < nchunks) load_chunk(s, j_begin + (int64_t)s * TJ);
    cp_async_commit();
  }
  for (int ch = 0; ch < nchunks; ++ch) {
    cp_async_wait<NS - 2>();  // chunk ch has landed
    __syncthreads();          // ... for every thread; chunk ch-1's buffer is free
    {
      const int nx = ch + NS - 1;
      if (nx < nchunks) load_chunk(nx % NS, j_begin + (int64_t)nx * TJ);
      cp_async_commit();
    }
    const int buf = ch % NS;
    const __nv_bfloat16* tL = sL + buf * TP * LPITCH;
    const __nv_bfloat16* tS = sS + buf * S_ELEMS;
#pragma unroll
    for (int kk = 0; kk < TJ / 16; ++kk) {
      uint32_t a[4];
      {
        const int i = lane >> 3;
        const int row = warp * 16 + (i & 1) * 8 + (lane & 7);
        const int col = kk * 16 + (i >> 1) * 8;
        ldsm_x4(s_addr(tL + row * LPITCH + col), a[0], a[1], a[2], a[3]);
      }
#pragma unroll
      for (int nt = 0; nt + 1 < Q / 8; nt += 2) {  // two n8 tiles at a time
        uint32_t b0, b1, b2, b3;
        const int i = lane >> 3;
        if (S_QJ) {
          const int q = nt * 8 + (i >> 1) * 8 + (lane & 7);
          const int j = kk * 16 + (i & 1) * 8;
          ldsm_x4(s_addr(tS + q * SP + j), b0, b1, b2, b3);
        } else {
          const int j = kk * 16 + (i & 1) * 8 + (lane & 7);
          const int q = nt * 8 + (i >> 1) * 8;
          ldsm_x4_t(s_addr(tS + j * SP + q), b0, b1, b2, b3);
        }
        mma_bf16_16816(acc[nt], a, b0, b1);
        mma_bf16_16816(acc[nt + 1], a, b2, b3);
      }
      if (Q % 16 == 8) {  // last single n8 tile
        constexpr int nt = Q / 8 - 1;
        uint32_t b0, b1;
        const int i = (lane >> 3) & 1;
        if (S_QJ) {
          ldsm_x2(s_addr(tS + (nt * 8 + (lane & 7)) * SP + kk * 16 + i * 8), b0, b1);
        } else {
          ldsm_x2_t(s_addr(tS + (kk * 16 + i * 8 + (lane & 7)) * SP + nt * 8), b0, b1);
        }
        mma_bf16_16816(acc[nt], a, b0, b1);
      }
    }
  }
  cp_async_wait<0>();

  __syncthreads();  // the ring is drained; its first 64 x Q floats take the partial tile

  // partial tile [64][Q] fp32: c0,c1 at (row g, cols 2t, 2t+1); c2,c3 at row g+8
  float* sP = reinterpret_cast<float*>(rr_smem);
  {
    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int nt = 0; nt < Q / 8; ++nt) {
      const int q = nt * 8 + 2 * t4;
      const int r0 = warp * 16 + g;
      *reinterpret_cast<float2*>(sP + r0 * Q + q) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(sP + (r0 + 8) * Q + q) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  cluster_sync_all();  // every split's partial tile is in its CTA's shared memory

  // CTA `rank` sums items rank, rank + splits, ... (4 outputs each) over the
  // cluster in rank order
  const uint32_t splits = (uint32_t)jb.sp.splits;
  const uint32_t rank = cluster_ctarank();
  const int rows = (int)(p_lim - p0 < TP ? p_lim - p0 : TP);
  for (int it = (int)rank * NTHR + tid; it < rows * (Q / 4); it += (int)splits * NTHR) {
    const float* src = sP + it * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (uint32_t c = 0; c < splits; ++c) {
      const float4 t = ld_cluster_v4(src, c);
      v.x += t.x;
      v.y += t.y;
      v.z += t.z;
      v.w += t.w;
    }
    const int64_t i = p0 * Q + (int64_t)it * 4;
    if (jb.out_f32) *reinterpret_cast<float4*>(jb.out_f32 + i) = v;
    if (jb.out_scaled) {
      float sc = jb.scale;
      if (jb.nseg > 0) {  // 4 consecutive columns lie in one segment (widths are multiples of 8)
        const int q = (it * 4) % Q;
        int k = 0;
        while (k + 1 < jb.nseg && q >= jb.seg_end[k]) ++k;
        sc = jb.seg_scale[k];
      }
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(jb.out_scaled + i);
      o2[0] = __floats2bfloat162_rn(v.x * sc, v.y * sc);
      o2[1] = __floats2bfloat162_rn(v.z * sc, v.w * sc);
    }
    const int64_t h = (p0 + (it * 4) / Q) * (2 * Q) + (it * 4) % Q;  // [P x 2Q] position of the hi value
    if (jb.out_hilo) store_hilo(jb.out_hilo + h, v, Q);
    if (jb.aux_hilo) store_hilo(jb.aux_hilo + h, *reinterpret_cast<const float4*>(jb.aux_src + i), Q);
  }
  cluster_sync_all();  // no CTA leaves while its tile may still be read
}

// ---------------------------------------------------------------------------
// Column reduce.  grid = (a.tiles + b.tiles, splits), clusters of (1,
// splits): x < a.tiles serves job a, the rest job b.  CTA (tile, split) owns
// columns 64 tile .. 64 tile + 63 and rows [split chunk, (split + 1) chunk);
// warp w owns 16 of the 64 columns.  Partial tile [64][2Q] fp32 (hi half, lo
// half); result out[j][q], or out[q][j] when transposed, = scale (sum hi +
// sum lo).
// ---------------------------------------------------------------------------
// Threads of the column reduction: for wide adapter chunks (Q >= 48, a
// multiple of 16) 8 warps, warp w taking columns 16 (w % 4) .. of the tile
// and half w / 4 of the 2Q (measured: Qwen3-0.6B q|k|v backward 145 vs
// 151 us); else 4 warps with all 2Q each (8 warps of 16 S columns made the
// Q = 16 launches slower: each warp repeats the tile's transposed loads).
template <int Q>
constexpr int cr_threads() {
  return (Q % 16 == 0 && Q >= 48) ? 2 * NTHR : NTHR;
}

template <int Q>
__global__ void __launch_bounds__(cr_threads<Q>()) cr_fin_kernel(const ColReduce ja, const ColReduce jbb) {
  constexpr int NS = kColStages;
  constexpr int Q2 = 2 * Q;
  constexpr int SP = Q2 + 8;
  constexpr int CT = cr_threads<Q>();       // threads of this CTA
  constexpr int QH = CT == NTHR ? Q2 : Q;   // S columns per warp
  extern __shared__ __align__(128) uint8_t cr_smem[];
  __nv_bfloat16* sL = reinterpret_cast<__nv_bfloat16*>(cr_smem);  // NS x [64 x 72]
  __nv_bfloat16* sS = sL + NS * TP * LPITCH;                         // NS x [64 x (2Q + 8)]

  // grouped: x runs over (expert, output tile of either job)
  int x = (int)blockIdx.x, grp = 0;
  if (ja.groups > 0) {
    const int per = ja.tiles + jbb.tiles;
    grp = x / per;
    x -= grp * per;
  }
  const bool second = x >= ja.tiles;
  ColReduce jb;
  if (second)
    jb = jbb;
  else
    jb = ja;
  const int tile = second ? x - ja.tiles : x;
  const int split = (int)blockIdx.y;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t P = jb.P, J = jb.J;
  const int64_t j0 = (int64_t)tile * TJ;
  const __nv_bfloat16* __restrict__ L = jb.L;
  const __nv_bfloat16* __restrict__ S2 = jb.S2;
  griddep_wait();
  griddep_launch_dependents();
  int64_t p_begin = (int64_t)split * jb.sp.chunk;
  int64_t p_end = min(P, p_begin + jb.sp.chunk);
  if (jb.groups > 0) {
    // the expert's rows (from the schedule kernel), split evenly over the
    // cluster in 64-row chunks; the expert's block of the output
    const int2 rg = jb.ranges[grp];
    const int64_t n64 = (rg.y - rg.x + TP - 1) / TP;
    const int64_t per = (n64 + jb.sp.splits - 1) / jb.sp.splits * TP;
    p_begin = rg.x + (int64_t)split * per;
    p_end = min((int64_t)rg.y, p_begin + per);
    jb.out += (int64_t)grp * J * Q;
  }
  const int nchunks = p_end > p_begin ? (int)((p_end - p_begin + TP - 1) / TP) : 0;

  auto load_chunk = [&](int buf, int64_t pp) {
    __nv_bfloat16* dL = sL + buf * TP * LPITCH;
    __nv_bfloat16* dS = sS + buf * TP * SP;
#pragma unroll
    for (int i = 0; i < 512 / CT; ++i) {  // 64 x 64 tile = 512 16-byte pieces
      const int piece = tid + i * CT;
      const int r = piece >> 3, c8 = (piece & 7) * 8;
      const bool ok = (pp + r) < p_end;
      cp_async16(s_addr(dL + r * LPITCH + c8), L + (ok ? (pp + r) : 0) * J + j0 + c8, ok);
    }
    for (int piece = tid; piece < TP * (Q2 / 8); piece += CT) {  // 64 rows x 2Q bf16
      const int r = piece / (Q2 / 8), c8 = (piece % (Q2 / 8)) * 8;
      const bool ok = (pp + r) < p_end;
      cp_async16(s_addr(dS + r * SP + c8), S2 + (ok ? (pp + r) : 0) * Q2 + c8, ok);
    }
  };

  const int wj = warp & 3;                          // 16-column group of the tile
  const int qbase = CT == NTHR ? 0 : (warp >> 2) * QH;  // first S column of this warp
  float acc[QH / 8][4];
#pragma unroll
  for (int t = 0; t < QH / 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

#pragma unroll
  for (int s = 0; s < NS - 1; ++s) {
    if (s < nchunks) load_chunk(s, p_begin + (int64_t)s * TP);
    cp_async_commit();
  }
  for (int ch = 0; ch < nchunks; ++ch) {
    cp_async_wait<NS - 2>();
    __syncthreads();  // chunk ch landed for all; chunk ch-1's buffers are free
    {
      const int nx = ch + NS - 1;
      if (nx < nchunks) load_chunk(nx % NS, p_begin + (int64_t)nx * TP);
      cp_async_commit();
    }
    const int buf = ch % NS;
    const __nv_bfloat16* tS = sS + buf * TP * SP;
    const __nv_bfloat16* tL = sL + buf * TP * LPITCH;
#pragma unroll
    for (int kk = 0; kk < TP / 16; ++kk) {
      uint32_t a[4];
      {  // A = L^T (m = j, k = p) from the [p][j] tile, transposed load
        const int i = lane >> 3;
        const int p = kk * 16 + (i >> 1) * 8 + (lane & 7);
        const int j = wj * 16 + (i & 1) * 8;
        ldsm_x4_t(s_addr(tL + p * LPITCH + j), a[0], a[1], a[2], a[3]);
      }
#pragma unroll
      for (int nt = 0; nt < QH / 8; nt += 2) {  // QH is a multiple of 16
        uint32_t b0, b1, b2, b3;
        const int i = lane >> 3;
        const int p = kk * 16 + (i & 1) * 8 + (lane & 7);
        const int q = qbase + nt * 8 + (i >> 1) * 8;
        ldsm_x4_t(s_addr(tS + p * SP + q), b0, b1, b2, b3);
        mma_bf16_16816(acc[nt], a, b0, b1);
        mma_bf16_16816(acc[nt + 1], a, b2, b3);
      }
    }
  }
  cp_async_wait<0>();

  __syncthreads();  // the ring is drained; its first 64 x 2Q floats take the partial tile

  float* sP = reinterpret_cast<float*>(cr_smem);
  {
    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int nt = 0; nt < QH / 8; ++nt) {
      const int q = qbase + nt * 8 + 2 * t4;
      const int r0 = wj * 16 + g;
      *reinterpret_cast<float2*>(sP + r0 * Q2 + q) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(sP + (r0 + 8) * Q2 + q) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  cluster_sync_all();

  // CTA `rank` sums items rank, rank + splits, ... (4 consecutive q of one
  // column) over the cluster in rank order, hi and lo halves separately.
  // With a window only the tile's projection's columns are written.
  const uint32_t splits = (uint32_t)jb.sp.splits;
  const uint32_t rank = cluster_ctarank();
  const int QW = jb.win > 0 ? jb.win : Q;  // output columns per row
  int qoff = 0;
  if (jb.win > 0)
    for (int p = 0; p + 1 < jb.nproj; ++p) qoff += j0 >= jb.proj_end[p] ? jb.win : 0;
  for (int it = (int)rank * CT + tid; it < TJ * (QW / 4); it += (int)splits * CT) {
    int jj, q;
    if (jb.transposed) {  // out[q][j]: consecutive items along j
      q = (it / TJ) * 4;
      jj = it % TJ;
    } else {  // out[j][q]: consecutive items along q
      jj = it / (QW / 4);
      q = (it % (QW / 4)) * 4;
    }
    const float* src = sP + jj * Q2 + qoff + q;
    float4 hi = make_float4(0.f, 0.f, 0.f, 0.f), lo = hi;
    for (uint32_t c = 0; c < splits; ++c) {
      const float4 th = ld_cluster_v4(src, c);
      const float4 tl = ld_cluster_v4(src + Q, c);
      hi.x += th.x;
      hi.y += th.y;
      hi.z += th.z;
      hi.w += th.w;
      lo.x += tl.x;
      lo.y += tl.y;
      lo.z += tl.z;
      lo.w += tl.w;
    }
    float sc = jb.scale;
    float* out = jb.out;
    int qo = q, ow = QW;  // column within the output array, its width
    if (jb.nseg > 0) {  // q .. q+3 lie in one segment (widths are multiples of 8)
      int k = 0;
      while (k + 1 < jb.nseg && q >= jb.seg_end[k]) ++k;
      const int start = k > 0 ? jb.seg_end[k - 1] : 0;
      sc = jb.seg_scale[k];
      out = jb.seg_out[k];
      qo = q - start;
      ow = jb.seg_end[k] - start;
      if (!out) continue;  // a frozen adapter: no gradient
    }
    const float4 v = make_float4((hi.x + lo.x) * sc, (hi.y + lo.y) * sc, (hi.z + lo.z) * sc, (hi.w + lo.w) * sc);
    const int64_t j = j0 + jj;
    if (jb.nseg > 0) {
      if (jb.transposed) {
        out[(int64_t)(qo + 0) * J + j] = v.x;
        out[(int64_t)(qo + 1) * J + j] = v.y;
        out[(int64_t)(qo + 2) * J + j] = v.z;
        out[(int64_t)(qo + 3) * J + j] = v.w;
      } else {
        *reinterpret_cast<float4*>(out + j * ow + qo) = v;
      }
    } else if (jb.transposed) {
      jb.out[(int64_t)(q + 0) * J + j] = v.x;
      jb.out[(int64_t)(q + 1) * J + j] = v.y;
      jb.out[(int64_t)(q + 2) * J + j] = v.z;
      jb.out[(int64_t)(q + 3) * J + j] = v.w;
    } else {
      *reinterpret_cast<float4*>(jb.out + j * QW + q) = v;
    }
  }
  cluster_sync_all();  // no CTA leaves while its tile may still be read
}

// Stacked adapters: A_cat rows and B_cat columns gathered from each
// adapter's arrays, 8 bf16 (16 bytes) per thread and step.
__global__ void pack_adapters_kernel(const AdapterPack ap, int64_t N, int64_t K, __nv_bfloat16* __restrict__ A_cat,
                                     __nv_bfloat16* __restrict__ B_cat) {
  int Q = 0;
  for (int i = 0; i < ap.n; ++i) Q += ap.r[i];
  const int64_t a_pieces = (int64_t)Q * (K / 8), b_pieces = N * (Q / 8);
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < a_pieces + b_pieces;
       t += (int64_t)gridDim.x * blockDim.x) {
    if (t < a_pieces) {  // A_cat row q = row q - off_i of adapter i
      const int q = (int)(t / (K / 8));
      const int64_t c8 = (t % (K / 8)) * 8;
      int i = 0, off = 0;
      while (q >= off + ap.r[i]) off += ap.r[i++];
      *reinterpret_cast<uint4*>(A_cat + (int64_t)q * K + c8) =
          *reinterpret_cast<const uint4*>(ap.A[i] + (int64_t)(q - off) * K + c8);
    } else {  // B_cat[n][off_i + c] = B_i[n][c]
      const int64_t u = t - a_pieces;
      const int64_t n = u / (Q / 8);
      const int c8 = (int)(u % (Q / 8)) * 8;
      int i = 0, off = 0;
      while (c8 >= off + ap.r[i]) off += ap.r[i++];
      *reinterpret_cast<uint4*>(B_cat + n * Q + c8) =
          *reinterpret_cast<const uint4*>(ap.B[i] + n * ap.r[i] + (c8 - off));
    }
  }
}

cudaError_t launch_pack_adapters(const AdapterPack& ap, int64_t N, int64_t K, __nv_bfloat16* A_cat,
                                 __nv_bfloat16* B_cat, cudaStream_t st) {
  int Q = 0;
  for (int i = 0; i < ap.n; ++i) Q += ap.r[i];
  const int64_t pieces = (int64_t)Q * (K / 8) + N * (Q / 8);
  int64_t blocks = (pieces + 255) / 256;
  if (blocks > 2048) blocks = 2048;
  count_launch(1);
  pack_adapters_kernel<<<(unsigned)(blocks > 0 ? blocks : 1), 256, 0, st>>>(ap, N, K, A_cat, B_cat);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Launch with clusters of (1, splits, 1) and programmatic stream
// serialisation (the kernels wait for the previous grid before touching
// global memory); the first launch of an instantiation raises its
// shared-memory limit.
template <typename... Args>
static cudaError_t launch_clustered(void (*kern)(Args...), dim3 grid, size_t smem, int splits, cudaStream_t st,
                                    bool& attr_done, int threads, Args... args) {
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)splits;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int Q>
static cudaError_t launch_rr_fin_q(const RowReduce& r, cudaStream_t st) {
  constexpr int NS = RowStages<Q>::NS;
  const size_t smem = (size_t)NS * 2 * (TP * LPITCH + (r.s_qj ? Q * LPITCH : TJ * (Q + 8)));
  const dim3 grid((unsigned)(r.tiles ? r.max_tiles : (r.P + TP - 1) / TP), (unsigned)r.sp.splits);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  if (r.sp.splits > kMaxClusterSplits) return cudaErrorInvalidValue;
  static bool attr_qj = false, attr_jq = false;
  if (r.s_qj) return launch_clustered(rr_fin_kernel<Q, true>, grid, smem, r.sp.splits, st, attr_qj, NTHR, r);
  return launch_clustered(rr_fin_kernel<Q, false>, grid, smem, r.sp.splits, st, attr_jq, NTHR, r);
}

template <int Q>
static cudaError_t launch_cr_fin_q(const ColReduce& a, const ColReduce& b, cudaStream_t st) {
  constexpr int NS = kColStages;
  constexpr size_t smem = (size_t)NS * 2 * (TP * LPITCH + TP * (2 * Q + 8));
  const dim3 grid((unsigned)((a.tiles + b.tiles) * (a.groups > 0 ? a.groups : 1)), (unsigned)a.sp.splits);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  if (a.sp.splits > kMaxClusterSplits || (b.tiles > 0 && b.sp.splits != a.sp.splits)) return cudaErrorInvalidValue;
  static bool attr = false;
  return launch_clustered(cr_fin_kernel<Q>, grid, smem, a.sp.splits, st, attr, cr_threads<Q>(), a, b);
}

#define QLORA_RANK_DISPATCH_FIN(FN, ...)     \
  switch (Q) {                               \
    case 8: return FN<8>(__VA_ARGS__);       \
    case 16: return FN<16>(__VA_ARGS__);     \
    case 24: return FN<24>(__VA_ARGS__);     \
    case 32: return FN<32>(__VA_ARGS__);     \
    case 40: return FN<40>(__VA_ARGS__);     \
    case 48: return FN<48>(__VA_ARGS__);     \
    case 56: return FN<56>(__VA_ARGS__);     \
    case 64: return FN<64>(__VA_ARGS__);     \
    default: return cudaErrorInvalidValue;   \
  }

cudaError_t launch_row_reduce_fin(const RowReduce& r, int Q, cudaStream_t st) {
  count_launch(1);
  QLORA_RANK_DISPATCH_FIN(launch_rr_fin_q, r, st)
}

cudaError_t launch_col_reduce_fin(const ColReduce& a, const ColReduce* b, int Q, cudaStream_t st) {
  count_launch(1);
  ColReduce none = a;
  none.tiles = 0;
  const ColReduce& bb = b ? *b : none;
  QLORA_RANK_DISPATCH_FIN(launch_cr_fin_q, a, bb, st)
}

}  // namespace qlora
