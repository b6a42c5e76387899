// Schedule of a grouped (mixture-of-experts) call, built on the device.
//
// The experts' row offsets live in device memory (a router writes them
// there), so the tile lists of the grouped GEMM and of the grouped adapter
// reductions are built by one small kernel at the head of the call, without
// copying the offsets to the host or synchronising.  One thread per expert:
// it checks its offsets, counts its GEMM row tiles and 64-row reduction
// tiles, takes its place from a block-wide prefix sum and writes its tiles.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/qlora.h"
#include "kernels.h"

namespace qlora {

namespace {

constexpr int kSchedThreads = kMaxGroups;  // one thread per expert

// inclusive prefix sum over the block (Hillis-Steele, in shared memory)
__device__ __forceinline__ int block_scan(int v, int* buf) {
  const int t = threadIdx.x;
  buf[t] = v;
  __syncthreads();
  for (int d = 1; d < kSchedThreads; d <<= 1) {
    const int add = t >= d ? buf[t - d] : 0;
    __syncthreads();
    buf[t] += add;
    __syncthreads();
  }
  return buf[t];
}

}  // namespace

__global__ void __launch_bounds__(kSchedThreads) grouped_schedule_kernel(const int32_t* __restrict__ off, int E,
                                                                       int64_t M_total, int tile_rows, int nblk_f,
                                                                       int nblk_d, GroupedSched s, int* err) {
  __shared__ int bad;
  __shared__ int buf[kSchedThreads];
  const int e = threadIdx.x;
  if (e == 0) bad = 0;
  __syncthreads();
  // rows [lo, hi) of expert e; the offsets must partition [0, M_total)
  int lo = 0, hi = 0;
  if (e < E) {
    lo = off[e];
    hi = off[e + 1];
    if (lo < 0 || hi < lo || (int64_t)hi > M_total || (e == 0 && lo != 0) || (e == E - 1 && (int64_t)hi != M_total))
      atomicExch(&bad, 1);
  }
  __syncthreads();
  const bool invalid = bad != 0;
  const int c = (e < E && !invalid) ? hi - lo : 0;
  const int g = (c + tile_rows - 1) / tile_rows;  // GEMM row tiles of this expert
  const int r = (c + 63) / 64;                    // 64-row reduction tiles
  const int g_end = block_scan(g, buf);
  const int g_all = buf[kSchedThreads - 1];
  __syncthreads();
  const int r_end = block_scan(r, buf);
  const int r_all = buf[kSchedThreads - 1];
  const int g0 = g_end - g, r0 = r_end - r;
  if (e < E) {
    s.ranges[e] = invalid ? make_int2(0, 0) : make_int2(lo, hi);
    // an expert's GEMM tiles are consecutive (its weights stay in L2),
    // column block by column block, row tiles fastest
    for (int nb = 0; nb < nblk_f; ++nb)
      for (int i = 0; i < g; ++i)
        s.gemm_f[(int64_t)g0 * nblk_f + nb * g + i] = make_int4(e, lo + i * tile_rows, min(tile_rows, c - i * tile_rows), nb);
    for (int nb = 0; nb < nblk_d; ++nb)
      for (int i = 0; i < g; ++i)
        s.gemm_d[(int64_t)g0 * nblk_d + nb * g + i] = make_int4(e, lo + i * tile_rows, min(tile_rows, c - i * tile_rows), nb);
    for (int i = 0; i < r; ++i) s.rows64[r0 + i] = make_int4(e, lo + 64 * i, min(64, c - 64 * i), 0);
  }
  if (e == 0) {
    s.counts[0] = g_all * nblk_f;
    s.counts[1] = g_all * nblk_d;
    s.counts[2] = r_all;
    if (invalid && err) atomicExch(err, QLORA_ERR_INVALID);
  }
}

cudaError_t launch_grouped_schedule(const int32_t* offsets, int E, int64_t M_total, int tile_rows, int nblk_f,
                                    int nblk_d, const GroupedSched& s, int* err, cudaStream_t st) {
  if (E < 1 || E > kMaxGroups) return cudaErrorInvalidValue;
  count_launch(1);
  grouped_schedule_kernel<<<1, kSchedThreads, 0, st>>>(offsets, E, M_total, tile_rows, nblk_f, nblk_d, s, err);
  return cudaGetLastError();
}

}  // namespace qlora
