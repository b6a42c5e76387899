// Fused quantised-base LoRA GEMM on a CTA pair (tcgen05 cta_group::2).
//
// Same operation as gemm_tc.cu (forward Y = X deq(W)^T + sT B^T, or
// dX = dY deq(W) + sU A), with a 256 x 256 output tile per pair of SMs:
//   - CTA r of the pair loads rows [m0 + 128 r, +128) of the A operand and
//     decodes (or loads) its half of the B operand: output columns
//     [n0 + 128 r, +128);
//   - one thread of CTA 0 issues tcgen05.mma.cta_group::2 (M 256, N 256,
//     K 16); the tensor cores of both SMs read their own halves and each
//     SM's TMEM receives its 128 rows x 256 fp32 columns;
//   - the MMA's completion is multicast to both CTAs' "stage empty" and
//     "accumulator full" barriers.
// Each decoded weight therefore feeds 256 output rows instead of 128, and
// each SM reads only half of the B tile from its shared memory.
//
// Synchronisation across the pair: both CTAs' TMA copies (2-CTA form) land in
// their own shared memory and complete their bytes on CTA 0's "stage full"
// barrier, whose expected byte count covers both CTAs.  (Relaying CTA 1's
// completion through a thread of CTA 1 instead cost 2.4x in throughput.)
// Decode warps and epilogue warps of both CTAs arrive on CTA 0's "B ready" /
// "accumulator empty" barriers with cluster-scope release.  All waits are
// bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace qlora {

namespace {

constexpr int P_TMEM_COLS = 512;

// Tile configurations of the pair (CFG):
//   1: 256 x 256, one M256 x N256 accumulator, two TMEM buffers (bf16 bases);
//   2: 512 x 128, two M256 x N128 accumulators sharing every decoded B tile,
//      two TMEM buffers;
//   3: 512 x 256, two M256 x N256 accumulators sharing every decoded B tile,
//      one TMEM buffer (all 512 columns): each accumulator is released as
//      soon as the epilogue holds its values, so the next tile's MMAs into
//      it can start while the previous tile is still being stored;
//   4: 256 x 256 with a quantised base, two TMEM buffers (grouped calls,
//      whose experts own ~256 rows each).
// Decoding one B tile for two accumulators halves the decode work per flop.
template <int CFG>
struct PairCfg {
  static constexpr int NACC = (CFG == 1 || CFG == 4) ? 1 : 2;  // accumulators per tile
  static constexpr int TM = 256 * NACC;                   // output rows per pair tile
  static constexpr int TN = CFG == 2 ? 128 : 256;         // output columns per pair tile
  static constexpr int NBUF = NACC * TN <= 256 ? 2 : 1;   // TMEM buffers of NACC accumulators
  static constexpr int HALF_N = TN / 2;                   // B rows (or columns) per CTA
  static constexpr int A_BYTES = NACC * 128 * kBK * 2;    // this CTA's A rows
  static constexpr int B_BYTES = HALF_N * kBK * 2;        // this CTA's half of B
  static constexpr int STAGES = (CFG == 1 || CFG == 4) ? 6 : (CFG == 2 ? 5 : 4);
  static constexpr int LINES = HALF_N;                    // decoded 64-wide lines per stage per CTA
  static constexpr int GROUP_WARPS = LINES / 32;          // one line per thread of a group
  static constexpr int GROUPS = (CFG == 1 || CFG == 4) ? 3 : (CFG == 2 ? 5 : 2);  // groups rotate over stages
  static constexpr int DQ_WARPS = GROUP_WARPS * GROUPS;
  static_assert(STAGES % GROUPS == 0, "a stage must always be decoded by the same group");
  static_assert(NBUF * NACC * TN == 512, "accumulators fill TMEM");
};

// Quantised bytes through a TMA ring ("raw" ring, filled by a warp of its
// own) instead of per-thread global loads, whose one-row-per-lane pattern
// touches a separate cache line per lane and load: each item's bytes are one
// 2-D (grouped: 3-D, expert outermost) byte box per CTA (forward: the CTA's
// weight rows x one line; dX: 64 weight rows x the CTA's two lines; the box
// starts at the line's 16-byte aligned address, raw_box_bytes wide), and the
// decode warps read their lines from shared memory.  Q4_K adds a second box
// with the 16-byte super-block headers.  Used by NF4 on 512 x 256 tiles and
// by every quantised format on grouped 256 x 256 tiles, where the host finds
// the layout allows it (GemmArgs::raw_on: 16-byte multiple row length;
// grouped: experts back to back in one array).  In NF4 dX on 512 x 256 tiles
// the slot also holds the item's int8 absmax codes (a 16-byte wide box of
// the 64 rows, x rounded down to 16 bytes) and the range of group scales its
// lines use (a 1-D bulk copy), when the host finds the layout allows it
// (GemmArgs::raw_dq).  On 512 x 256 tiles the ring's shared memory comes from
// the second epilogue staging tile and a warp of its own fills it.  On
// grouped 256 x 256 tiles the box lands in the stage's B slot itself
// (INPLACE), loaded by the operand producer with the stage's A rows: the
// decode group reads its lines into registers, meets at a named barrier,
// and writes the decoded tile over them; no ring of its own, so the six
// operand stages still fit.
template <int FMT, int CFG, bool DX>
struct PairRaw {
  static constexpr bool ON = FMT != FMT_BF16 && ((FMT == FMT_NF4 && CFG == 3) || CFG == 4);
  static constexpr bool INPLACE = ON && CFG == 4;
  static constexpr bool RING = ON && !INPLACE;
  static constexpr int STAGES = DX ? 3 : 4;                     // ring slots (RING)
  static constexpr int ROWS = DX ? 64 : PairCfg<CFG>::HALF_N;   // weight rows of one item's box
  static constexpr int BOX = raw_box_bytes(FMT, DX);           // bytes per row of the box
  static constexpr int LINE = raw_line_bytes(FMT);              // bytes of one line
  static constexpr int CODE_BYTES = ROWS * BOX;                 // main box of one item for this CTA
  static constexpr int HDR_BYTES = FMT == FMT_Q4_K ? ROWS * 16 : 0;  // Q4_K: [ROWS x 16] headers after the box
  static constexpr int AQ_OFF = CODE_BYTES;                     // NF4 dX: [64 rows x 16] absmax codes
  static constexpr int SC_OFF = CODE_BYTES + 1024;              // NF4 dX: group scales
  static constexpr int SC_CAP = 64;                             // NF4 dX: group scales a slot holds
  static constexpr int RAW_DQ = FMT == FMT_NF4 && CFG == 3 && DX;
  static constexpr int BYTES = !RING ? 0 : ((RAW_DQ ? SC_OFF + 4 * SC_CAP : CODE_BYTES + HDR_BYTES) + 127) / 128 * 128;
  static_assert(!INPLACE || CODE_BYTES + HDR_BYTES <= PairCfg<CFG>::B_BYTES, "the box fits the B slot");
  static constexpr int OUT_BUFS = (CFG == 2 || (ON && CFG == 3)) ? 1 : 2;  // epilogue staging tiles
};

template <int CFG>
struct __align__(8) PairBarriers {
  uint64_t full[PairCfg<CFG>::STAGES];    // CTA 0: bytes of both CTAs' copies (CTA 1: unused)
  uint64_t bready[PairCfg<CFG>::STAGES];  // CTA 0: decode warps of both CTAs
  uint64_t empty[PairCfg<CFG>::STAGES];   // both: MMA completion (multicast)
  uint64_t acc_full[4];                   // per (buffer, accumulator): MMA completion (multicast)
  uint64_t acc_empty[4];                  // CTA 0, per (buffer, accumulator): epilogue warps of both CTAs
  uint64_t raw_full[8];                   // raw ring: code bytes landed (TMA, this CTA)
  uint64_t raw_empty[8];                  // raw ring: the decode group has read them (this CTA)
  uint32_t tmem_base;
  int abort;
  int ep_ok;  // epilogue: result of the "accumulator full" wait, for all 4 warps
};

// epilogue staging: 128-row x 64-column bf16 chunks (128B-swizzled), each
// written out with a TMA tensor store
constexpr int P_STAGE_OUT_BYTES = 128 * 64 * 2;

template <int FMT, int CFG, bool DX>
constexpr size_t p_smem_bytes() {
  using Raw = PairRaw<FMT, CFG, DX>;
  return 1024 + (size_t)PairCfg<CFG>::STAGES * (PairCfg<CFG>::A_BYTES + PairCfg<CFG>::B_BYTES) +
         (size_t)Raw::OUT_BUFS * P_STAGE_OUT_BYTES + (size_t)Raw::STAGES * Raw::BYTES + sizeof(PairBarriers<CFG>);
}
template <int FMT>
constexpr bool smem_fits_all() {
  return p_smem_bytes<FMT, 2, false>() <= 232448 && p_smem_bytes<FMT, 2, true>() <= 232448 &&
         p_smem_bytes<FMT, 3, false>() <= 232448 && p_smem_bytes<FMT, 3, true>() <= 232448 &&
         p_smem_bytes<FMT, 4, false>() <= 232448 && p_smem_bytes<FMT, 4, true>() <= 232448;
}
static_assert(smem_fits_all<FMT_NF4>() && smem_fits_all<FMT_Q8_0>() && smem_fits_all<FMT_Q4_0>() &&
                  smem_fits_all<FMT_Q4_K>() && smem_fits_all<FMT_FP8>() && smem_fits_all<FMT_NVFP4>() &&
                  p_smem_bytes<FMT_BF16, 1, true>() <= 232448,
              "shared memory per CTA");
template <int FMT, int CFG, bool DX>
constexpr bool raw_aligned() {
  using R = PairRaw<FMT, CFG, DX>;
  return R::BYTES % 128 == 0 && R::AQ_OFF % 128 == 0 && R::SC_OFF % 128 == 0 && R::CODE_BYTES % 128 == 0;
}
static_assert(raw_aligned<FMT_NF4, 3, true>() && raw_aligned<FMT_NF4, 3, false>() &&
                  raw_aligned<FMT_Q8_0, 4, true>() && raw_aligned<FMT_Q8_0, 4, false>() &&
                  raw_aligned<FMT_Q4_0, 4, true>() && raw_aligned<FMT_Q4_0, 4, false>() &&
                  raw_aligned<FMT_Q4_K, 4, true>() && raw_aligned<FMT_Q4_K, 4, false>(),
              "raw ring slots keep TMA destinations 128-byte aligned");

// warps: 0 TMA producer, 1 TMEM / MMA issuer, 2-5 epilogue, then the decode
// warps, then (raw ring) the code-byte producer
template <int FMT, int CFG>
constexpr int p_threads() {
  return (FMT == FMT_BF16) ? 6 * 32 : (6 + PairCfg<CFG>::DQ_WARPS + (PairRaw<FMT, CFG, false>::RING ? 1 : 0)) * 32;
}

// One line's bytes from its raw ring row (line starts `addr`, 4-byte
// aligned) into RawLine words 0 .. LINE/4-1: 16-byte loads from the aligned
// address at or below, shifted down by the (warp-uniform) word offset.
template <int FMT, int LINE>
__device__ __forceinline__ void read_raw_line(uint32_t addr, RawLine& r) {
  constexpr int NW = LINE / 4;                 // words of the line
  constexpr int NC = (LINE % 16) ? (LINE + 12 + 15) / 16 : LINE / 16;  // 16-byte loads
  uint32_t u[4 * (NC > 0 ? NC : 1)];
  const uint32_t base = addr & ~15u;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const uint4 v = lds_v4(base + 16 * i);
    u[4 * i] = v.x; u[4 * i + 1] = v.y; u[4 * i + 2] = v.z; u[4 * i + 3] = v.w;
  }
  if constexpr (LINE % 16 == 0) {
#pragma unroll
    for (int i = 0; i < NW; ++i) r.w[i] = u[i];
  } else {
    const uint32_t sh = (addr & 15u) >> 2;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const uint32_t a = sh & 1 ? u[i + 1] : u[i];
      const uint32_t b = sh & 1 ? u[i + 3] : u[i + 2];
      r.w[i] = sh & 2 ? b : a;
    }
  }
}

// Coordinates of an item's raw box: the first weight row, and the byte x of
// the CTA's first line in its row rounded down to 16 (Q4_K: the chunk's
// code bytes, and xh the super-block's header).  bn: this CTA's first weight
// row (forward) or output column (dX).
template <int FMT, bool DX>
__device__ __forceinline__ void raw_box_coords(int bn, int kb, int32_t& x, int32_t& xh, int32_t& row0) {
  const int64_t line0 = DX ? bn / 64 : kb;
  row0 = DX ? kb * kBK : bn;
  xh = 0;
  if constexpr (FMT == FMT_Q4_K) {
    x = (int32_t)((line0 >> 2) * 144 + 16 + 32 * (line0 & 3));
    xh = (int32_t)((line0 >> 2) * 144);
  } else {
    x = (int32_t)((raw_line_bytes(FMT) * line0) & ~int64_t(15));
  }
}

// First weight row (forward) of this CTA's share of a tile's B.
template <int CFG>
__device__ __forceinline__ int64_t b_first_row(const GemmArgs& a, int n0, uint32_t rank) {
  if (a.swiglu_i > 0) return (rank ? (int64_t)a.swiglu_i : 0) + n0 / 2;
  return n0 + PairCfg<CFG>::HALF_N * (int)rank;
}

struct PairTile {
  int m0, n0;
  int rows;  // grouped: rows of the tile that belong to its expert (from m0)
  int e;     // grouped: expert
};

struct NoGroups {
  int unused;
};


// Tile order (chosen on the host): row blocks fastest keeps the whole A
// operand hot in L2 while weight slabs stream; column blocks fastest keeps
// the weight hot while A row blocks stream.  The smaller operand is the one
// kept, so the larger one is read from DRAM once.
template <bool DX, int CFG>
__device__ __forceinline__ PairTile pair_tile(const GemmArgs& a, int t) {
  constexpr int TM = PairCfg<CFG>::TM, TN = PairCfg<CFG>::TN;
  PairTile p;
  if (a.tile_sched) {  // grouped: the schedule kernel's list
    const int4 s = a.tile_sched[t];
    p.e = s.x;
    p.m0 = s.y;
    p.rows = s.z;
    p.n0 = s.w * TN;
    return p;
  }
  const int num_m = (a.M + TM - 1) / TM;
  const int num_n = a.num_n_blk;
  p.e = 0;
  p.rows = TM;
  if (!a.n_fastest) {
    p.m0 = (t % num_m) * TM;
    p.n0 = (t / num_m) * TN;
  } else {
    p.n0 = (t % num_n) * TN;
    p.m0 = (t / num_n) * TM;
  }
  return p;
}

}  // namespace

// GROUPED: tiles from the schedule list (args.tile_sched / tile_count), each
// with its expert's weight view (tab) and adapter (3-D adapter and bf16
// weight maps, expert index outermost); a pair CTA's 128-row block may hold
// fewer rows of its expert, which are stored without the staging tile.
template <int FMT, bool DX, int CFG, bool GROUPED, bool DIRECT = false>
__global__ void __launch_bounds__(p_threads<FMT, CFG>(), 1)
    qgemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_la, const __grid_constant__ CUtensorMap tm_lb,
                      const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_aq,
                      const GemmArgs args,
                      const __grid_constant__ std::conditional_t<GROUPED, GroupTable, NoGroups> tab) {
  using Cfg = PairCfg<CFG>;
  using Raw = PairRaw<FMT, CFG, DX>;
  constexpr int P_STAGES = Cfg::STAGES, P_A_BYTES = Cfg::A_BYTES, P_B_BYTES = Cfg::B_BYTES;
  constexpr int TN = Cfg::TN, HALF_N = Cfg::HALF_N, NACC = Cfg::NACC, NBUF = Cfg::NBUF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA0 = smem_u32(smem);
  const uint32_t sB0 = sA0 + P_STAGES * P_A_BYTES;
  const uint32_t sOut = sB0 + P_STAGES * P_B_BYTES;  // 1024-aligned (stage sizes are multiples of 8 KB)
  const uint32_t sRaw = sOut + Raw::OUT_BUFS * P_STAGE_OUT_BYTES;
  PairBarriers<CFG>* bars = reinterpret_cast<PairBarriers<CFG>*>(
      smem + P_STAGES * (P_A_BYTES + P_B_BYTES) + Raw::OUT_BUFS * P_STAGE_OUT_BYTES + Raw::STAGES * Raw::BYTES);
  volatile int* abort = &bars->abort;

  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool has_lora = args.rank > 0;
  const int nkb = args.k_red / kBK;
  const int nkb_total = nkb + (has_lora ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->bready[s]), 2 * Cfg::GROUP_WARPS);  // one group's warps, both CTAs
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(smem_u32(&bars->acc_full[b]), 1);
      mbar_init(smem_u32(&bars->acc_empty[b]), 8);
    }
    for (int b = 0; b < (Raw::INPLACE ? P_STAGES : Raw::STAGES); ++b) {
      mbar_init(smem_u32(&bars->raw_full[b]), 1);
      mbar_init(smem_u32(&bars->raw_empty[b]), Cfg::GROUP_WARPS);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(&bars->tmem_base), P_TMEM_COLS);
  if (warp == 2 && lane == 0) prefetch_tmap(&tm_out);
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_a);
    if (FMT == FMT_BF16 || (Raw::ON && args.raw_on)) prefetch_tmap(&tm_w);
    if (Raw::ON && args.raw_on && ((DX && args.raw_dq) || FMT == FMT_Q4_K)) prefetch_tmap(&tm_aq);
    if (has_lora) {
      prefetch_tmap(&tm_la);
      prefetch_tmap(&tm_lb);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // peer barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  // launched with programmatic stream serialisation: the set-up above
  // overlaps the previous kernel's tail; nothing global is touched before it
  // has finished, and the next kernel may start its own set-up
  griddep_wait();
  griddep_launch_dependents();
  // grouped: the tile count comes from the schedule kernel (earlier in the
  // stream, complete once griddep_wait returned)
  const int num_tiles = GROUPED ? *args.tile_count : args.num_tiles;
  const int my_tiles = pair < num_tiles ? (num_tiles - pair + num_pairs - 1) / num_pairs : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      for (int lt = 0; lt < my_tiles; ++lt) {
        const PairTile tc = pair_tile<DX, CFG>(args, pair + lt * num_pairs);
        const int am = tc.m0 + 128 * (int)rank;     // this CTA's A rows (+256 per accumulator)
        // this CTA's half of B (forward: its first weight row; dX: first output column)
        const int bn = DX ? tc.n0 + HALF_N * (int)rank : (int)b_first_row<CFG>(args, tc.n0, rank);
        for (int kb = 0; kb < nkb_total; ++kb, ++it) {
          const int s = it % P_STAGES;
          const uint32_t ph = (it / P_STAGES) & 1;
          if (!mbar_wait_cluster(smem_u32(&bars->empty[s]), ph ^ 1, abort, args.err)) goto producer_done;
          const bool lora = kb == nkb;
          const uint32_t sa = sA0 + s * P_A_BYTES, sb = sB0 + s * P_B_BYTES;
          const uint32_t bytes = P_A_BYTES + ((FMT == FMT_BF16 || lora) ? P_B_BYTES : 0);
          // CTA 0 expects both CTAs' bytes; every copy completes on CTA 0's barrier
          if (rank == 0) mbar_arrive_expect_tx(smem_u32(&bars->full[s]), 2 * bytes);
          const uint32_t fb = mapa_shared(smem_u32(&bars->full[s]), 0);
          if constexpr (Raw::INPLACE) {
            // this CTA's quantised bytes into its B slot (decoded there)
            if (args.raw_on) {
              const uint32_t rb = smem_u32(&bars->raw_full[s]);
              if (!lora) {
                int32_t x, xh, row0;
                raw_box_coords<FMT, DX>(bn, kb, x, xh, row0);
                mbar_arrive_expect_tx(rb, Raw::CODE_BYTES + Raw::HDR_BYTES);
                if constexpr (GROUPED) {
                  tma_load_3d(sb, &tm_w, rb, x, row0, tc.e);
                  if constexpr (FMT == FMT_Q4_K) tma_load_3d(sb + Raw::CODE_BYTES, &tm_aq, rb, xh, row0, tc.e);
                } else {
                  tma_load_2d(sb, &tm_w, rb, x, row0);
                  if constexpr (FMT == FMT_Q4_K) tma_load_2d(sb + Raw::CODE_BYTES, &tm_aq, rb, xh, row0);
                }
              } else {
                mbar_arrive(rb);  // the adapter chunk: no bytes, keeps the phases in step
              }
            }
          }
          if (!lora) {
#pragma unroll
            for (int a = 0; a < NACC; ++a) tma_load_2d_pair(sa + a * 16384, &tm_a, fb, kb * kBK, am + 256 * a);
            if (FMT == FMT_BF16) {
              if (!DX) {
                if (GROUPED) tma_load_3d_pair(sb, &tm_w, fb, kb * kBK, bn, tc.e);
                else tma_load_2d_pair(sb, &tm_w, fb, kb * kBK, bn);
              } else {
#pragma unroll
                for (int j = 0; j < HALF_N / 64; ++j) {
                  if (GROUPED) tma_load_3d_pair(sb + j * 8192, &tm_w, fb, bn + 64 * j, kb * kBK, tc.e);
                  else tma_load_2d_pair(sb + j * 8192, &tm_w, fb, bn + 64 * j, kb * kBK);
                }
              }
            }
          } else {
#pragma unroll
            for (int a = 0; a < NACC; ++a)
              tma_load_2d_pair(sa + a * 16384, &tm_la, fb, adapter_col(args, tc.n0), am + 256 * a);
            if (!DX) {
              // SwiGLU: CTA 1's rows of B land rank columns in, where the
              // up projection's T sits in the adapter chunk (x < 0 is zero-filled)
              const int lbx = args.swiglu_i > 0 ? -(args.rank / 2) * (int)rank : 0;  // rank = 2 r here
              if (GROUPED) tma_load_3d_pair(sb, &tm_lb, fb, lbx, bn, tc.e);
              else tma_load_2d_pair(sb, &tm_lb, fb, lbx, bn);
            } else {
#pragma unroll
              for (int j = 0; j < HALF_N / 64; ++j) {
                if (GROUPED) tma_load_3d_pair(sb + j * 8192, &tm_lb, fb, bn + 64 * j, 0, tc.e);
                else tma_load_2d_pair(sb + j * 8192, &tm_lb, fb, bn + 64 * j, 0);
              }
            }
          }
        }
      }
    producer_done:
      // CTA 0 waits for the last copies of every stage; CTA 1's copies complete
      // on those same barriers
      if (rank == 0)
        for (uint32_t k = (it >= P_STAGES ? it - P_STAGES : 0); k < it; ++k)
          mbar_drain(smem_u32(&bars->full[k % P_STAGES]), (k / P_STAGES) & 1);
      // and each CTA for its own in-place raw boxes
      if (Raw::INPLACE && args.raw_on)
        for (uint32_t k = (it >= P_STAGES ? it - P_STAGES : 0); k < it; ++k)
          mbar_drain(smem_u32(&bars->raw_full[k % P_STAGES]), (k / P_STAGES) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(256, TN, DX);
      uint32_t it = 0;
      for (int lt = 0; lt < my_tiles; ++lt) {
        const int buf = lt % NBUF;
        const uint32_t aph = (lt / NBUF) & 1;
        bool ok = true;
        // the epilogue must have taken the buffer's values (double-buffered:
        // a tile ago; single buffer: the epilogue releases each accumulator
        // as soon as its values are in registers).  Waiting here rather than
        // right before each accumulator's first MMA measured the same for
        // the single buffer and 20% faster for bf16 tiles.
#pragma unroll
        for (int a = 0; a < NACC; ++a)
          ok = ok && mbar_wait_cluster(smem_u32(&bars->acc_empty[buf * NACC + a]), aph ^ 1, abort, args.err);
        if (!ok) break;
        tc_fence_after();
        for (int kb = 0; kb < nkb_total && ok; ++kb, ++it) {
          const int s = it % P_STAGES;
          const uint32_t ph = (it / P_STAGES) & 1;
          if (!mbar_wait_cluster(smem_u32(&bars->full[s]), ph, abort, args.err)) { ok = false; break; }
          if (FMT != FMT_BF16) {
            if (!mbar_wait_cluster(smem_u32(&bars->bready[s]), ph, abort, args.err)) { ok = false; break; }
          }
          // operands arrive through mbarriers (TMA complete_tx, or decode
          // warps' proxy fence + release arrive): no tcgen05 fence is needed
          // here, and none is issued so consecutive stages' MMAs overlap
          const bool lora = kb == nkb;
          const int nk = lora ? (args.rank + 15) / 16 : kBK / 16;
          const uint32_t sa = sA0 + s * P_A_BYTES, sb = sB0 + s * P_B_BYTES;
          for (int kk = 0; kk < nk; ++kk) {
            const uint64_t bdesc = DX ? smem_desc_sw128(sb + kk * 2048, 8192, 1024)
                                      : smem_desc_sw128(sb + kk * 32, 16, 1024);
#pragma unroll
            for (int a = 0; a < NACC; ++a) {
              const uint64_t adesc = smem_desc_sw128(sa + a * 16384 + kk * 32, 16, 1024);
              tc_mma_bf16_pair(tmem_base + buf * (NACC * TN) + a * TN, adesc, bdesc, idesc,
                               (kb > 0 || kk > 0) ? 1u : 0u);
            }
          }
          tc_commit_pair_mc(smem_u32(&bars->empty[s]));
        }
        if (!ok) break;
#pragma unroll
        for (int a = 0; a < NACC; ++a) tc_commit_pair_mc(smem_u32(&bars->acc_full[buf * NACC + a]));
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    // Per 64-column chunk: each thread loads its row's 64 fp32 values from
    // TMEM, converts them to bf16 and writes one 128-byte row of a
    // 128B-swizzled staging tile (conflict-free); one thread then stores the
    // 128 x 64 tile with a TMA tensor store.  With two staging tiles the
    // store of one chunk overlaps the conversion of the next.  Chunks wholly
    // outside the output are neither staged nor stored.
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    const int ep = (warp - 2) * 32 + lane;  // 0..127
    const int swz = row_in_tile & 7;
    uint32_t nstored = 0;  // chunks stored so far (selects the staging tile)
    for (int lt = 0; lt < my_tiles; ++lt) {
      const PairTile tc = pair_tile<DX, CFG>(args, pair + lt * num_pairs);
      const int buf = lt % NBUF;
      const uint32_t aph = (lt / NBUF) & 1;
      bool ok = true;
#pragma unroll 1
      for (int a = 0; a < NACC && ok; ++a) {
        const int slot = buf * NACC + a;
        // one thread waits; all four warps take the same decision (they meet
        // at named barriers below, which must never be left half-entered)
        if (ep == 0) bars->ep_ok = mbar_wait_cluster(smem_u32(&bars->acc_full[slot]), aph, abort, args.err) ? 1 : 0;
        named_bar(1, 128);
        ok = *reinterpret_cast<volatile int*>(&bars->ep_ok) != 0;
        named_bar(1, 128);  // everyone has read ep_ok before it is rewritten
        if (!ok) break;
        tc_fence_after();
        const int row0 = tc.m0 + 256 * a + 128 * (int)rank;
        if (!DX && !GROUPED && args.swiglu_i > 0) {
          // SwiGLU: TMEM columns [0, TN/2) hold gate, [TN/2, TN) the up
          // values of the same output columns; 32 columns of each at a
          // time, stored from registers: G, U (bf16) and H = silu(G) U
          const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * (NACC * TN) + a * TN;
          const int64_t row = row0 + row_in_tile;
          const bool rok = row < args.M;
          const int64_t I = args.swiglu_i;
#pragma unroll 1
          for (int c = 0; c < TN / 64; ++c) {
            uint32_t gv[32], uv[32];
            tmem_ld_32x32b_x32(tb + 32 * c, gv);
            tmem_ld_32x32b_x32(tb + TN / 2 + 32 * c, uv);
            tc_wait_ld();
            if (c + 1 == TN / 64) {  // every value of this accumulator is in registers: release it
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&bars->acc_empty[buf * NACC + a]), 0));
            }
            const int64_t col = tc.n0 / 2 + 32 * c;  // gate / H column
            if (rok && col < I) {
              uint4* dg = reinterpret_cast<uint4*>(args.out + row * 2 * I + col);
              uint4* du = reinterpret_cast<uint4*>(args.out + row * 2 * I + I + col);
              uint4* dh = reinterpret_cast<uint4*>(args.swiglu_h + row * I + col);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                // H from G and U as stored (bf16), like the elementwise pass
                float g[8], u[8], h[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  g[k] = __bfloat162float(__float2bfloat16_rn(__uint_as_float(gv[8 * q + k])));
                  u[k] = __bfloat162float(__float2bfloat16_rn(__uint_as_float(uv[8 * q + k])));
                  h[k] = swiglu_h_f32(g[k], u[k]);
                }
                dg[q] = make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]), pack_bf16x2(g[4], g[5]),
                                   pack_bf16x2(g[6], g[7]));
                du[q] = make_uint4(pack_bf16x2(u[0], u[1]), pack_bf16x2(u[2], u[3]), pack_bf16x2(u[4], u[5]),
                                   pack_bf16x2(u[6], u[7]));
                dh[q] = make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]),
                                   pack_bf16x2(h[6], h[7]));
              }
            }
          }
          continue;
        }
        constexpr int NCH = TN / 64;
        const uint32_t tcol = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * (NACC * TN) + a * TN;
        uint32_t v[64];
        tmem_ld_32x32b_x32(tcol, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld_32x32b_x32(tcol + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tc_wait_ld();
        // fully unrolled: the registers a TMEM load fills are read only after
        // the wait that completes it (no loop-carried copies in between)
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const bool last = c + 1 == NCH;
          if (last) {
            // every value of this accumulator is in registers: release it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&bars->acc_empty[slot]), 0));
          }
          // the same for all 128 threads.  Grouped: rows of this 128-row block
          // that belong to the tile's expert; a partly filled block is stored
          // row by row from registers (the staging tile's TMA store would
          // write the next expert's rows)
          const int nvalid = GROUPED ? min(128, tc.rows - 256 * a - 128 * (int)rank) : 128;
          const bool store = row0 < args.M && nvalid > 0 && tc.n0 + 64 * c < args.n_out;
          if (args.out_f32 != nullptr) {
            // debug: the fp32 accumulator values, row by row from registers
            if (store && row_in_tile < nvalid && row0 + row_in_tile < args.M) {
              float4* dst = reinterpret_cast<float4*>(args.out_f32 + (int64_t)(row0 + row_in_tile) * args.n_out +
                                                      tc.n0 + 64 * c);
#pragma unroll
              for (int q = 0; q < 16; ++q)
                dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                     __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
            if (!last) {
              tmem_ld_32x32b_x32(tcol + 64 * (c + 1), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
              tmem_ld_32x32b_x32(tcol + 64 * (c + 1) + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
              tc_wait_ld();
            }
            continue;
          }
          if (GROUPED && store && nvalid < 128) {
            if (row_in_tile < nvalid) {
              uint4* dst = reinterpret_cast<uint4*>(args.out + (int64_t)(row0 + row_in_tile) * args.n_out + tc.n0 + 64 * c);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const uint32_t* w = v + 8 * q;
                dst[q] = make_uint4(pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                                    pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                                    pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5])),
                                    pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7])));
              }
            }
            if (!last) {
              tmem_ld_32x32b_x32(tcol + 64 * (c + 1), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
              tmem_ld_32x32b_x32(tcol + 64 * (c + 1) + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
              tc_wait_ld();
            }
            continue;
          }
          if constexpr (DIRECT || (Raw::OUT_BUFS == 1 && !DX)) {
            if (DIRECT || args.direct_out) {
              // rows stored straight from registers, without the staging
              // tile and the TMA store (chosen by the host for forward
              // outputs of at most 4096 columns, where it measured faster)
              if (store && row0 + row_in_tile < args.M) {
                uint4* dst =
                    reinterpret_cast<uint4*>(args.out + (int64_t)(row0 + row_in_tile) * args.n_out + tc.n0 + 64 * c);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const uint32_t* w = v + 8 * q;
                  dst[q] = make_uint4(pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                                      pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                                      pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5])),
                                      pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7])));
                }
              }
              if (!last) {
                tmem_ld_32x32b_x32(tcol + 64 * (c + 1), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld_32x32b_x32(tcol + 64 * (c + 1) + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tc_wait_ld();
              }
              continue;
            }
          }
          const uint32_t stile = sOut + (nstored % Raw::OUT_BUFS) * P_STAGE_OUT_BYTES;
          if (store) {
            ++nstored;
            if (ep == 0) {  // the store that last read this staging tile is done with it
              if (Raw::OUT_BUFS == 2)
                bulk_wait_read1();
              else
                bulk_wait_read0();
            }
            named_bar(1, 128);
            const uint32_t srow = stile + (uint32_t)row_in_tile * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t* w = v + 8 * q;
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1]));
              o.y = pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3]));
              o.z = pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5]));
              o.w = pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7]));
              sts_v4(srow + ((q ^ swz) << 4), o);
            }
          }
          // the next chunk's TMEM load lands while this one is stored
          if (!last) {
            tmem_ld_32x32b_x32(tcol + 64 * (c + 1), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld_32x32b_x32(tcol + 64 * (c + 1) + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          }
          if (store) {
            fence_proxy_async_smem();
            named_bar(1, 128);
            if (ep == 0) {
              tma_store_2d(&tm_out, stile, tc.n0 + 64 * c, row0);
              bulk_commit();
            }
          }
          if (!last) tc_wait_ld();
        }
      }
      if (!ok) break;
    }
    if (ep == 0) bulk_wait0();
  } else if (FMT != FMT_BF16 && warp < 6 + Cfg::DQ_WARPS) {
    // ------------------------------------------------------------ decode
    // group g (GROUP_WARPS warps) handles the items with it % GROUPS == g;
    // thread d of the group decodes one 64-element line of this CTA's half
    // of B per item.
    constexpr int P_DQ_GROUPS = Cfg::GROUPS;
    const int g = (warp - 6) / Cfg::GROUP_WARPS;
    const int d = ((warp - 6) % Cfg::GROUP_WARPS) * 32 + lane;  // 0 .. LINES-1
    const int srow = DX ? (d & 63) : d;
    const uint32_t soff = DX ? (uint32_t)((d >> 6) * 8192 + srow * 128) : (uint32_t)(srow * 128);
    const int swz = srow & 7;
    const uint32_t total = (uint32_t)my_tiles * (uint32_t)nkb_total;
    const uint32_t bready0 = mapa_shared(smem_u32(&bars->bready[0]), 0);

    // Item iterator without divisions: (local tile, k-block) advance by
    // GROUPS items per step; the tile's line base is recomputed only when the
    // tile changes.
    struct Cursor {
      uint32_t it;
      int kb, lt;
      int64_t base;  // forward: first line of this thread's row; dX: k-line
      bool row_ok;   // forward: weight row in range; dX: k-line in range
      const WeightView* wv;  // the tile's base weight (grouped: its expert's)
    };
    auto set_tile = [&](Cursor& c) {
      if (c.lt >= my_tiles) return;
      const PairTile tc = pair_tile<DX, CFG>(args, pair + c.lt * num_pairs);
      if constexpr (GROUPED) c.wv = &tab.w[tc.e];
      if (!DX) {
        const int64_t row = b_first_row<CFG>(args, tc.n0, rank) + d;
        c.row_ok = row < args.w_rows;
        c.base = row * args.w_lines_per_row;
      } else {
        const int64_t kl = (tc.n0 + HALF_N * (int)rank) / 64 + (d >> 6);
        c.row_ok = kl < args.w_lines_per_row;
        c.base = kl;
      }
    };
    auto advance = [&](Cursor& c, int n) {
      c.it += n;
      c.kb += n;
      bool moved = false;
      while (c.kb >= nkb_total) {
        c.kb -= nkb_total;
        ++c.lt;
        moved = true;
      }
      if (moved) set_tile(c);
    };
    // line index and validity of the cursor's item (adapter chunk: invalid)
    auto line_at = [&](const Cursor& c, bool& valid) -> int64_t {
      valid = c.it < total && c.kb < nkb && c.row_ok;
      if (!DX) return c.base + c.kb;
      return ((int64_t)c.kb * kBK + (d & 63)) * args.w_lines_per_row + c.base;
    };
    // Forward, double-quantised NF4 through the raw ring: a thread's lines
    // are blocks kb, kb + GROUPS, ... of one weight row, so its absmax codes
    // come 8 at a time (one aligned word) and its group scale changes at
    // most once or twice per row.  Each is loaded when a line first needs a
    // new one and kept with the one before it; a line records which word
    // and group it needs (low 32 bits of their indices) and picks them at
    // decode time, when the load issued for it has had an item to land.
    const bool raw = Raw::ON && args.raw_on;
    const bool dq_cache = FMT == FMT_NF4 && raw && !DX && !GROUPED && args.wv.absmax == nullptr &&
                          args.wv.aq_align8;
    int64_t aq_base = -1, sc_grp = -1;
    uint32_t aq_new_lo = 0, aq_new_hi = 0, aq_old_lo = 0, aq_old_hi = 0, aq_old_base = 0xffffffffu;
    float sc_new = 0.f, sc_old = 0.f;
    uint32_t sc_old_grp = 0xffffffffu;
    auto fetch = [&](const Cursor& c, RawLine& r) -> bool {
      bool valid;
      const int64_t ln = line_at(c, valid);
      if (valid) {
        if (dq_cache) {
          const int64_t wb = ln & ~int64_t(7);
          if (wb != aq_base) {
            aq_old_lo = aq_new_lo;
            aq_old_hi = aq_new_hi;
            aq_old_base = (uint32_t)aq_base;
            const uint2 w2 = ldg_nc_v2(args.wv.absmax_q + wb);
            aq_new_lo = w2.x;
            aq_new_hi = w2.y;
            aq_base = wb;
          }
          const int64_t grp = args.wv.dq_shift >= 0 ? (ln >> args.wv.dq_shift) : ln / args.wv.dq_group;
          if (grp != sc_grp) {
            sc_old = sc_new;
            sc_old_grp = (uint32_t)sc_grp;
            sc_new = __ldg(args.wv.absmax_scale + grp);
            sc_grp = grp;
          }
          r.w[8] = (uint32_t)wb;
          r.w[9] = (uint32_t)grp;
          r.q = (int32_t)(ln & 7);
        } else if (raw && DX && args.raw_dq) {
          // everything this line needs arrives through the raw ring
        } else if (raw) {
          load_line_side<FMT>(*c.wv, ln, r);  // the code bytes come through the raw ring
        } else {
          load_line<FMT>(*c.wv, ln, r);
        }
      }
      return valid;
    };
    // the line's absmax code and group scale from the two cached entries
    auto resolve_dq = [&](RawLine& r) {
      const bool wnew = r.w[8] == (uint32_t)aq_base;
      const uint32_t lo = wnew ? aq_new_lo : aq_old_lo, hi = wnew ? aq_new_hi : aq_old_hi;
      const uint32_t word = (r.q & 4) ? hi : lo;
      const int32_t q = (int32_t)(int8_t)(uint8_t)(word >> (8 * (r.q & 3)));
      r.scale = (r.w[9] == (uint32_t)sc_grp) ? sc_new : sc_old;
      r.q = q;
      (void)aq_old_base;
      (void)sc_old_grp;
    };
    auto process = [&](const Cursor& c, RawLine& r, bool valid) -> bool {
      const int s = c.it % P_STAGES;
      const uint32_t ph = (c.it / P_STAGES) & 1;
      bool ok = true;
      if (raw) {
        // this item's code bytes: wait for them (every lane, for its own
        // acquire) and copy them to registers; a ring slot is handed back
        // after the line's stores (below)
        const uint32_t rs = Raw::INPLACE ? (uint32_t)s : c.it % Raw::STAGES;
        const uint32_t rph = Raw::INPLACE ? ph : (c.it / Raw::STAGES) & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->raw_full[rs]), rph, abort, args.err));
        // in place, a failure is only acted on at the group's barrier below,
        // which every warp of the group must reach
        if (!ok && !Raw::INPLACE) return false;
        if (ok && valid && c.kb < nkb) {
          const uint32_t slot = Raw::INPLACE ? sB0 + s * P_B_BYTES : sRaw + rs * Raw::BYTES;
          const int row = DX ? (d & 63) : d;
          // the line's first byte within its box row: the box starts at the
          // 16-byte aligned address at or below the CTA's first line
          int off;
          if constexpr (FMT == FMT_Q4_K) {
            off = DX ? 32 * (d >> 6) : 0;
          } else if (!DX) {
            off = (Raw::LINE * c.kb) & 15;
          } else {
            const int64_t kl0 = c.base - (d >> 6);
            off = Raw::LINE * (d >> 6) + (int)((Raw::LINE * kl0) & 15);
          }
          read_raw_line<FMT, Raw::LINE>(slot + (uint32_t)(row * Raw::BOX + off), r);
          if constexpr (FMT == FMT_Q4_K) {
            const uint4 h = lds_v4(slot + Raw::CODE_BYTES + (uint32_t)(row * 16));
            r.w[8] = h.x; r.w[9] = h.y; r.w[10] = h.z; r.w[11] = h.w;
          }
          if (DX && args.raw_dq) {
            // absmax code of (row, block) and the group scale of its line
            const int kblk = (int)c.base;  // this thread's k-block
            const int kblk0 = kblk - (d >> 6);
            const uint32_t qb = lds_u8(slot + Raw::AQ_OFF + (uint32_t)((d & 63) * 16 + (kblk & 15)));
            const int64_t row0 = (int64_t)c.kb * kBK;
            const int64_t g_lo = (row0 * args.w_lines_per_row + kblk0) >> args.wv.dq_shift;
            const int64_t ln = (row0 + (d & 63)) * args.w_lines_per_row + kblk;
            const int64_t gi = (ln >> args.wv.dq_shift) - (g_lo & ~int64_t(3));
            r.q = (int32_t)(int8_t)(uint8_t)qb;
            r.scale = lds_f32(slot + Raw::SC_OFF + (uint32_t)gi * 4);
          }
        }
      }
      // NF4 dX: decode in registers before waiting for the slot, so the
      // arithmetic overlaps the wait and only the stores follow the slot's
      // release (in place, the slot is free once its bytes are; elsewhere the
      // extra live registers spill)
      constexpr bool EARLY = DX && !Raw::INPLACE && FMT == FMT_NF4;
      uint4 out[8];
      if constexpr (EARLY) {
        if (ok && valid && c.kb < nkb) {
          if (dq_cache) resolve_dq(r);
          decode_line<FMT>(r, *c.wv, out);
        }
      }
      if (lane == 0 && ok) ok = mbar_wait_cluster(smem_u32(&bars->empty[s]), ph ^ 1, abort, args.err);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      // in place: every line of the group has been read before any decoded
      // line overwrites the box (and the group leaves together on a failure)
      if (Raw::INPLACE && raw) ok = named_bar_and(2 + g, 32 * Cfg::GROUP_WARPS, ok);
      if (!ok) return false;
      if (c.kb < nkb) {
        const uint32_t dst = sB0 + s * P_B_BYTES + soff;
        if (valid) {
          if constexpr (!EARLY) {
            if (dq_cache) resolve_dq(r);
            decode_line<FMT>(r, *c.wv, out);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) sts_v4(dst + ((q ^ swz) << 4), out[q]);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) sts_v4(dst + (q << 4), make_uint4(0, 0, 0, 0));
        }
      }
      // one proxy fence orders both this warp's stores of B (read by the
      // MMA) and, with the raw ring, its reads of the raw slot before the
      // slot's TMA refill (async proxy; without it a refill could land before
      // a read and a line decode the next item's bytes), so the slot is
      // handed back only after it.  The stores are published to CTA 0's MMA
      // issuer with a release restricted to this CTA's shared memory (all
      // that it has to order) and a relaxed arrive.
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster_after_smem_writes(bready0 + s * 8);
        if (Raw::RING && raw) mbar_arrive(smem_u32(&bars->raw_empty[c.it % Raw::STAGES]));
      }
      return true;
    };

    // cur: the item being processed; pre: the item whose bytes are loaded
    // next (two items ahead of cur, so two lines are in flight per thread;
    // measured on the Llama gate shape, three or four lines in flight are
    // slower)
    Cursor cur{0, 0, 0, 0, false, &args.wv};
    set_tile(cur);
    advance(cur, g);
    Cursor pre = cur;
    advance(pre, P_DQ_GROUPS);
    RawLine ra, rb;
    bool va = fetch(cur, ra);
    bool vb = fetch(pre, rb);
    advance(pre, P_DQ_GROUPS);
    while (cur.it < total) {
      if (!process(cur, ra, va)) break;
      va = fetch(pre, ra);
      advance(pre, P_DQ_GROUPS);
      advance(cur, P_DQ_GROUPS);
      if (cur.it >= total) break;
      if (!process(cur, rb, vb)) break;
      vb = fetch(pre, rb);
      advance(pre, P_DQ_GROUPS);
      advance(cur, P_DQ_GROUPS);
    }
  }

  if (Raw::RING && args.raw_on && warp == 6 + Cfg::DQ_WARPS && lane == 0) {
    // ---------------------------------------------------- raw code producer
    // the same item sequence as the decode warps: every (tile, k-block) of
    // this pair, the adapter chunk included (no bytes: a plain arrive)
    uint32_t it = 0;
    bool ok = true;
    for (int lt = 0; lt < my_tiles && ok; ++lt) {
      const PairTile tc = pair_tile<DX, CFG>(args, pair + lt * num_pairs);
      // forward: first weight row; dX: first output column
      const int ncol = DX ? tc.n0 + HALF_N * (int)rank : (int)b_first_row<CFG>(args, tc.n0, rank);
      for (int kb = 0; kb < nkb_total; ++kb, ++it) {
        const uint32_t rs = it % Raw::STAGES;
        if (!mbar_wait(smem_u32(&bars->raw_empty[rs]), ((it / Raw::STAGES) & 1) ^ 1, abort, args.err)) {
          ok = false;
          break;
        }
        const uint32_t bar = smem_u32(&bars->raw_full[rs]);
        const uint32_t slot = sRaw + rs * Raw::BYTES;
        if (kb < nkb) {
          int32_t x, xh, row0;
          raw_box_coords<FMT, DX>(ncol, kb, x, xh, row0);
          if (!(DX && args.raw_dq)) {
            mbar_arrive_expect_tx(bar, Raw::CODE_BYTES + Raw::HDR_BYTES);
            if constexpr (GROUPED) {
              tma_load_3d(slot, &tm_w, bar, x, row0, tc.e);
              if constexpr (FMT == FMT_Q4_K) tma_load_3d(slot + Raw::CODE_BYTES, &tm_aq, bar, xh, row0, tc.e);
            } else {
              tma_load_2d(slot, &tm_w, bar, x, row0);
              if constexpr (FMT == FMT_Q4_K) tma_load_2d(slot + Raw::CODE_BYTES, &tm_aq, bar, xh, row0);
            }
          } else {
            // codes, the 64 rows' absmax codes from block (kblk0 & ~15) on,
            // and the group scales from (g_lo & ~3) to g_hi rounded up to
            // whole 16-byte pieces (the host checked that the array is a
            // whole number of them and that the range fits SC_CAP)
            const int kblk0 = ncol / 64;
            const int64_t row0 = (int64_t)kb * kBK;
            const int64_t g_lo = (row0 * args.w_lines_per_row + kblk0) >> args.wv.dq_shift;
            const int64_t g_hi = ((row0 + 63) * args.w_lines_per_row + kblk0 + 1) >> args.wv.dq_shift;
            const int64_t g0 = g_lo & ~int64_t(3);
            const uint32_t sc_bytes = (uint32_t)(((g_hi - g0 + 1) + 3) & ~int64_t(3)) * 4;
            mbar_arrive_expect_tx(bar, Raw::CODE_BYTES + 1024 + sc_bytes);
            tma_load_2d(slot, &tm_w, bar, ncol / 2, kb * kBK);
            tma_load_2d(slot + Raw::AQ_OFF, &tm_aq, bar, kblk0 & ~15, kb * kBK);
            bulk_load_1d(slot + Raw::SC_OFF, args.wv.absmax_scale + g0, sc_bytes, bar);
          }
        } else {
          mbar_arrive(bar);
        }
      }
    }
    // copies still in flight land before the CTA may leave
    for (uint32_t k = (it >= (uint32_t)Raw::STAGES ? it - Raw::STAGES : 0); k < it; ++k)
      mbar_drain(smem_u32(&bars->raw_full[k % Raw::STAGES]), (k / Raw::STAGES) & 1);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, P_TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
template <int FMT, bool DX, int CFG, bool GROUPED, bool DIRECT = false>
static cudaError_t launch_pair_one(const GemmMaps& maps, const GemmArgs& args, const GroupTable* tab,
                                   cudaStream_t st) {
  auto kern = qgemm_pair_kernel<FMT, DX, CFG, GROUPED, DIRECT>;
  constexpr size_t P_SMEM_BYTES = p_smem_bytes<FMT, CFG, DX>();
  static int max_clusters = -1;  // per instantiation
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(p_threads<FMT, CFG>());
  cfg.dynamicSmemBytes = P_SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // occupancy query without the launch-order attribute
  if (max_clusters < 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    max_clusters = n > 0 ? n : 1;
  }
  // grouped: num_tiles is the schedule's upper bound (the count itself is on
  // the device)
  int pairs = args.num_tiles < max_clusters ? args.num_tiles : max_clusters;
  if (pairs <= 0) return cudaSuccess;
  if constexpr (!GROUPED) {
    // the fewest pairs that finish the tiles in the same number of rounds
    // (e.g. 128 tiles: 64 pairs, two rounds each, instead of 76 of which
    // 24 would idle through the second); the SMs left free take the work
    // launched beside the GEMM (the backward's dA / dB reduction)
    const int rounds = (args.num_tiles + pairs - 1) / pairs;
    pairs = (args.num_tiles + rounds - 1) / rounds;
  }
  cfg.gridDim = dim3(2 * pairs);
  cfg.numAttrs = 2;
  if constexpr (GROUPED) {
    if (!tab) return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, kern, maps.a, maps.w, maps.la, maps.lb, maps.out, maps.aq, args, *tab);
  } else {
    return cudaLaunchKernelEx(&cfg, kern, maps.a, maps.w, maps.la, maps.lb, maps.out, maps.aq, args, NoGroups{0});
  }
}

#ifndef QLORA_PAIR_QCFG
#define QLORA_PAIR_QCFG 3
#endif
constexpr int kQuantCfg = QLORA_PAIR_QCFG;  // tile configuration for quantised bases

int pair_tile_rows(int cfg) {
  return cfg == 1 ? PairCfg<1>::TM : (cfg == 2 ? PairCfg<2>::TM : (cfg == 3 ? PairCfg<3>::TM : PairCfg<4>::TM));
}
int pair_tile_cols(int cfg) {
  return cfg == 1 ? PairCfg<1>::TN : (cfg == 2 ? PairCfg<2>::TN : (cfg == 3 ? PairCfg<3>::TN : PairCfg<4>::TN));
}

// Quantised bases take 512 x 256 tiles (two accumulators share every decoded
// weight tile) unless the launch has so few of them that the 512 x 128 tiling
// finishes sooner: it has twice the tiles, each half the work, at ~0.8 of the
// 512 x 256 tile's efficiency (measured on the Llama gate shape: 905 vs
// 1104 TF/s).  Estimated time = waves of tiles x time of one tile.
int pair_cfg(int fmt, int64_t M, int64_t n_out, int num_sms) {
  if (fmt == FMT_BF16) return 1;
  if (kQuantCfg != 3) return kQuantCfg;
  const int64_t pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;
  const int64_t rows = (M + PairCfg<3>::TM - 1) / PairCfg<3>::TM;
  const int64_t t3 = rows * ((n_out + PairCfg<3>::TN - 1) / PairCfg<3>::TN);
  const int64_t t2 = rows * ((n_out + PairCfg<2>::TN - 1) / PairCfg<2>::TN);
  const double cost3 = (double)((t3 + pairs - 1) / pairs);
  const double cost2 = (double)((t2 + pairs - 1) / pairs) * 0.5 / 0.8;
  return cost2 < 0.9 * cost3 ? 2 : 3;
}

template <int CFG, bool G>
static cudaError_t launch_quant(int fmt, bool dx, const GemmMaps& maps, const GemmArgs& args, const GroupTable* tab,
                                cudaStream_t st) {
  switch (fmt) {
    case FMT_NF4:
      if constexpr (CFG == 3 && !G) {
        // dX with outputs of at most 4096 columns: its own instantiation
        // storing rows from registers (a run-time choice inside one kernel
        // made every dX launch slower)
        if (dx && args.direct_out) return launch_pair_one<FMT_NF4, true, CFG, G, true>(maps, args, tab, st);
      }
      return dx ? launch_pair_one<FMT_NF4, true, CFG, G>(maps, args, tab, st)
                : launch_pair_one<FMT_NF4, false, CFG, G>(maps, args, tab, st);
    case FMT_Q8_0:
      return dx ? launch_pair_one<FMT_Q8_0, true, CFG, G>(maps, args, tab, st)
                : launch_pair_one<FMT_Q8_0, false, CFG, G>(maps, args, tab, st);
    case FMT_Q4_0:
      return dx ? launch_pair_one<FMT_Q4_0, true, CFG, G>(maps, args, tab, st)
                : launch_pair_one<FMT_Q4_0, false, CFG, G>(maps, args, tab, st);
    case FMT_Q4_K:
      return dx ? launch_pair_one<FMT_Q4_K, true, CFG, G>(maps, args, tab, st)
                : launch_pair_one<FMT_Q4_K, false, CFG, G>(maps, args, tab, st);
    case FMT_FP8:
      return dx ? launch_pair_one<FMT_FP8, true, CFG, G>(maps, args, tab, st)
                : launch_pair_one<FMT_FP8, false, CFG, G>(maps, args, tab, st);
    case FMT_NVFP4:
      return dx ? launch_pair_one<FMT_NVFP4, true, CFG, G>(maps, args, tab, st)
                : launch_pair_one<FMT_NVFP4, false, CFG, G>(maps, args, tab, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_qgemm_pair(int fmt, bool dx, int cfg, const GemmMaps& maps, const GemmArgs& args,
                              cudaStream_t st) {
  count_launch(1);
  if (fmt == FMT_BF16) {
    if (cfg != 1) return cudaErrorInvalidValue;
    return dx ? launch_pair_one<FMT_BF16, true, 1, false>(maps, args, nullptr, st)
              : launch_pair_one<FMT_BF16, false, 1, false>(maps, args, nullptr, st);
  }
  if (cfg == 2) return launch_quant<2, false>(fmt, dx, maps, args, nullptr, st);
  if (cfg == 3) return launch_quant<3, false>(fmt, dx, maps, args, nullptr, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_qgemm_pair_grouped(int fmt, bool dx, const GemmMaps& maps, const GemmArgs& args,
                                      const GroupTable& tab, cudaStream_t st) {
  count_launch(1);
  if (fmt == FMT_BF16)
    return dx ? launch_pair_one<FMT_BF16, true, 1, true>(maps, args, &tab, st)
              : launch_pair_one<FMT_BF16, false, 1, true>(maps, args, &tab, st);
  return launch_quant<4, true>(fmt, dx, maps, args, &tab, st);
}

}  // namespace qlora
