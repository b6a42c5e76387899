// Fused quantised-base LoRA GEMM on the 5th-generation tensor cores.
//
//   forward (DX = false):  out[M x N] = X[M x K] deq(W)[N x K]^T + sT[M x r] B[N x r]^T
//   dX      (DX = true):   out[M x K] = dY[M x N] deq(W)[N x K]  + sU[M x r] A[r x K]
//
// The adapter product is one extra reduction chunk appended to the tile's
// K-loop ([X | sT] . [deq(W) | B]^T), so the LoRA up-projection costs r/16
// extra MMAs per tile and no separate pass over Y.
//
// Dense problems of at most 128 rows (larger ones and grouped calls run on
// the SM-pair kernel of gemm_pair.cu).  Persistent, warp-specialised, one
// CTA per SM:
//   warp 0      TMA producer: A tiles (X or dY), and bf16 B tiles when the base
//               is bf16 or for the adapter chunk
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2..5  epilogue: tcgen05.ld TMEM -> registers -> bf16 -> global
//   warps 6..13 (quantised bases only) dequant producers: 128-bit loads of
//               the quantised blocks straight from global memory, register
//               decode, 16-byte stores into the 128B-swizzled operand layout
//               the tensor core reads.  Decoded weights never touch HBM.
// Operand tiles: A 128 x 64 bf16 (K-major, 128B swizzle); B 256 x 64 bf16,
// K-major for the forward pass, MN-major for dX (the dX pass reads W[n, k]
// with n as the reduction index).  Accumulator: 128 x 256 fp32 in TMEM,
// double-buffered (512 columns) so the epilogue of tile i overlaps the
// main loop of tile i+1.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace qlora {

namespace {

constexpr int STAGES = 4;
constexpr int A_BYTES = kBM * kBK * 2;  // 16 KB
constexpr int B_BYTES = kBN * kBK * 2;  // 32 KB
constexpr int NUM_DQ_WARPS = 8;
constexpr int TMEM_COLS = 512;

struct __align__(8) Barriers {
  uint64_t full[STAGES];
  uint64_t bready[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort;
};

constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + (size_t)STAGES * (A_BYTES + B_BYTES) + sizeof(Barriers);

template <int FMT>
constexpr int num_threads() {
  return (FMT == FMT_BF16) ? 6 * 32 : (6 + NUM_DQ_WARPS) * 32;
}

struct TileCoord {
  int m0, rows, n0;
};

__device__ __forceinline__ TileCoord tile_coord(const GemmArgs& a, int t) {
  // m fastest: concurrently running CTAs share the same weight slab
  TileCoord c;
  const int num_m = (a.M + kBM - 1) / kBM;
  const int mb = t % num_m, nb = t / num_m;
  c.m0 = mb * kBM;
  c.rows = min(kBM, a.M - c.m0);
  c.n0 = nb * kBN;
  return c;
}

}  // namespace

template <int FMT, bool DX>
__global__ void __launch_bounds__(num_threads<FMT>(), 1)
    qgemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                 const __grid_constant__ CUtensorMap tm_la, const __grid_constant__ CUtensorMap tm_lb,
                 const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA0 = smem_u32(smem);
  const uint32_t sB0 = sA0 + STAGES * A_BYTES;
  Barriers* bars = reinterpret_cast<Barriers*>(smem + STAGES * (A_BYTES + B_BYTES));
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool has_lora = args.rank > 0;
  const int nkb = args.k_red / kBK;
  const int nkb_total = nkb + (has_lora ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->bready[s]), NUM_DQ_WARPS);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->acc_full[b]), 1);
      mbar_init(smem_u32(&bars->acc_empty[b]), 4);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&bars->tmem_base), TMEM_COLS);
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_a);
    if (FMT == FMT_BF16) prefetch_tmap(&tm_w);
    if (has_lora) {
      prefetch_tmap(&tm_la);
      prefetch_tmap(&tm_lb);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      for (int t = blockIdx.x; t < args.num_tiles; t += gridDim.x) {
        const TileCoord tc = tile_coord(args, t);
        for (int kb = 0; kb < nkb_total; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(smem_u32(&bars->empty[s]), ph ^ 1, abort, args.err)) goto producer_done;
          const bool lora = kb == nkb;
          const uint32_t fb = smem_u32(&bars->full[s]);
          const uint32_t sa = sA0 + s * A_BYTES, sb = sB0 + s * B_BYTES;
          mbar_arrive_expect_tx(fb, A_BYTES + ((FMT == FMT_BF16 || lora) ? B_BYTES : 0));
          if (!lora) {
            tma_load_2d(sa, &tm_a, fb, kb * kBK, tc.m0);
            if (FMT == FMT_BF16) {
              if (!DX) {
                tma_load_2d(sb, &tm_w, fb, kb * kBK, tc.n0);
              } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * 8192, &tm_w, fb, tc.n0 + 64 * j, kb * kBK);
              }
            }
          } else {
            tma_load_2d(sa, &tm_la, fb, adapter_col(args, tc.n0), tc.m0);
            if (!DX) {
              tma_load_2d(sb, &tm_lb, fb, 0, tc.n0);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * 8192, &tm_lb, fb, tc.n0 + 64 * j, 0);
            }
          }
        }
      }
    producer_done:
      // make sure no bulk copy into this CTA's shared memory is still in
      // flight when the CTA retires (normally all completed long ago)
      if (it > 0) {
        for (uint32_t k = (it >= STAGES ? it - STAGES : 0); k < it; ++k) {
          const int s = k % STAGES;
          mbar_drain(smem_u32(&bars->full[s]), (k / STAGES) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, DX);
      uint32_t it = 0, lt = 0;
      for (int t = blockIdx.x; t < args.num_tiles; t += gridDim.x, ++lt) {
        const uint32_t ab = lt & 1, aph = (lt >> 1) & 1;
        if (!mbar_wait(smem_u32(&bars->acc_empty[ab]), aph ^ 1, abort, args.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * kBN;
        bool ok = true;
        for (int kb = 0; kb < nkb_total; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(smem_u32(&bars->full[s]), ph, abort, args.err)) { ok = false; break; }
          if (FMT != FMT_BF16) {
            if (!mbar_wait(smem_u32(&bars->bready[s]), ph, abort, args.err)) { ok = false; break; }
          }
          // operands arrive through mbarriers (TMA complete_tx, or decode
          // warps' proxy fence + release arrive): no tcgen05 fence is needed
          // here, and none is issued so consecutive stages' MMAs overlap
          const bool lora = kb == nkb;
          const int nk = lora ? (args.rank + 15) / 16 : kBK / 16;
          const uint32_t sa = sA0 + s * A_BYTES, sb = sB0 + s * B_BYTES;
          for (int kk = 0; kk < nk; ++kk) {
            const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bdesc = DX ? smem_desc_sw128(sb + kk * 2048, 8192, 1024)
                                      : smem_desc_sw128(sb + kk * 32, 16, 1024);
            tc_mma_bf16(d_tmem, adesc, bdesc, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&bars->empty[s]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&bars->acc_full[ab]));
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int row_in_tile = quarter * 32 + lane;
    uint32_t lt = 0;
    for (int t = blockIdx.x; t < args.num_tiles; t += gridDim.x, ++lt) {
      const TileCoord tc = tile_coord(args, t);
      const uint32_t ab = lt & 1, aph = (lt >> 1) & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(smem_u32(&bars->acc_full[ab]), aph, abort, args.err);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const bool row_ok = row_in_tile < tc.rows;
      __nv_bfloat16* orow = args.out + (int64_t)(tc.m0 + row_in_tile) * args.n_out + tc.n0;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) + ab * kBN + c * 32, v);
        tc_wait_ld();
        if (row_ok && tc.n0 + c * 32 < args.n_out && args.out_f32 != nullptr) {
          float4* dst = reinterpret_cast<float4*>(args.out_f32 + (int64_t)(tc.m0 + row_in_tile) * args.n_out +
                                                  tc.n0 + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        } else if (row_ok && tc.n0 + c * 32 < args.n_out) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
            o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
            o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
            o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
            dst[q] = o;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[ab]));
    }
  } else if (FMT != FMT_BF16) {
    // ------------------------------------------------------------ dequant
    const int d = (warp - 6) * 32 + lane;  // 0..255
    // forward: row d of the 256-row tile; dX: row (d & 63) of the 64-row
    // reduction chunk, 64-column sub-tile (d >> 6)
    const int srow = DX ? (d & 63) : d;
    const uint32_t soff = DX ? (uint32_t)((d >> 6) * 8192 + srow * 128) : (uint32_t)(srow * 128);
    const int swz = srow & 7;

    auto line_of = [&](const TileCoord& tc, int kb, bool& valid) -> int64_t {
      int64_t row, kl;
      if (!DX) {
        row = tc.n0 + d;
        kl = kb;
      } else {
        row = (int64_t)kb * kBK + (d & 63);
        kl = tc.n0 / 64 + (d >> 6);
      }
      valid = row < args.w_rows && kl < args.w_lines_per_row;
      return row * args.w_lines_per_row + kl;
    };

    uint32_t it = 0;
    RawLine cur;
    bool cur_valid = false;
    // prime: first work item
    int t = blockIdx.x, kb = 0;
    if (t < args.num_tiles) {
      const TileCoord tc = tile_coord(args, t);
      if (kb < nkb) {
        const int64_t ln = line_of(tc, kb, cur_valid);
        if (cur_valid) load_line<FMT>(args.wv, ln, cur);
      }
    }
    while (t < args.num_tiles) {
      // next work item
      int tn = t, kbn = kb + 1;
      if (kbn == nkb_total) { tn = t + gridDim.x; kbn = 0; }
      RawLine nxt;
      bool nxt_valid = false;
      if (tn < args.num_tiles && kbn < nkb) {
        const TileCoord tcn = tile_coord(args, tn);
        const int64_t ln = line_of(tcn, kbn, nxt_valid);
        if (nxt_valid) load_line<FMT>(args.wv, ln, nxt);
      }
      const int s = it % STAGES;
      const uint32_t ph = (it / STAGES) & 1;
      if (!mbar_wait(smem_u32(&bars->empty[s]), ph ^ 1, abort, args.err)) break;
      if (kb < nkb) {
        const uint32_t dst = sB0 + s * B_BYTES + soff;
        if (cur_valid) {
          uint4 out[8];
          decode_line<FMT>(cur, args.wv, out);
#pragma unroll
          for (int c = 0; c < 8; ++c) sts_v4(dst + ((c ^ swz) << 4), out[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) sts_v4(dst + (c << 4), make_uint4(0, 0, 0, 0));
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->bready[s]));
      cur = nxt;
      cur_valid = nxt_valid;
      t = tn;
      kb = kbn;
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
template <int FMT, bool DX>
static cudaError_t launch_one(const GemmMaps& maps, const GemmArgs& args, int num_sms, cudaStream_t st) {
  auto kern = qgemm_kernel<FMT, DX>;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = args.num_tiles < num_sms ? args.num_tiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, num_threads<FMT>(), SMEM_BYTES, st>>>(maps.a, maps.w, maps.la, maps.lb, args);
  return cudaGetLastError();
}

template <int FMT>
static cudaError_t launch_fmt(bool dx, const GemmMaps& maps, const GemmArgs& args, int num_sms, cudaStream_t st) {
  return dx ? launch_one<FMT, true>(maps, args, num_sms, st) : launch_one<FMT, false>(maps, args, num_sms, st);
}

cudaError_t launch_qgemm(int fmt, bool dx, const GemmMaps& maps, const GemmArgs& args, int num_sms, cudaStream_t st) {
  count_launch(1);
  switch (fmt) {
    case FMT_BF16: return launch_fmt<FMT_BF16>(dx, maps, args, num_sms, st);
    case FMT_NF4: return launch_fmt<FMT_NF4>(dx, maps, args, num_sms, st);
    case FMT_Q8_0: return launch_fmt<FMT_Q8_0>(dx, maps, args, num_sms, st);
    case FMT_Q4_0: return launch_fmt<FMT_Q4_0>(dx, maps, args, num_sms, st);
    case FMT_Q4_K: return launch_fmt<FMT_Q4_K>(dx, maps, args, num_sms, st);
    case FMT_FP8: return launch_fmt<FMT_FP8>(dx, maps, args, num_sms, st);
    case FMT_NVFP4: return launch_fmt<FMT_NVFP4>(dx, maps, args, num_sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qlora
