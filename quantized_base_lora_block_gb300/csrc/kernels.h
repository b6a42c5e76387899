// Internal interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "decode.cuh"

namespace qlora {

// Fused projections that share their input (e.g. q, k, v): at most this
// many in one call.
constexpr int kMaxProj = 8;
// Stacked adapters on one base: at most this many in one call.
constexpr int kMaxAdapters = 4;

void count_launch(int n);
int* device_error_word();  // address of the device error word on the current device

// ---- skinny adapter contractions (reduce.cu) ---------------------------------
struct SplitPlan {
  int splits;     // number of partial sums
  int64_t chunk;  // reduction elements per split (multiple of 64)
};

// Target number of CTAs for the split reductions.  A fixed constant (not the
// device's SM count) so the summation order does not depend on the device.
constexpr int kSplitTargetCtas = 608;

// Splits of the reductions that finish their sums in the kernel (reduce.cu):
// the splits of one output tile form one thread-block cluster, so at most
// kMaxClusterSplits; at most one wave of kSplitTargetCtas CTAs; at least two
// 64-wide chunks per split.
constexpr int kMaxClusterSplits = 8;
inline SplitPlan plan_split_fin(int64_t outer_tiles, int64_t red_len) {
  const int64_t red_tiles = (red_len + 63) / 64;
  int64_t s = kSplitTargetCtas / (outer_tiles > 0 ? outer_tiles : 1);
  if (s > red_tiles / 2) s = red_tiles / 2;
  if (s > kMaxClusterSplits) s = kMaxClusterSplits;
  if (s < 1) s = 1;
  const int64_t per = (red_tiles + s - 1) / s;
  SplitPlan p;
  p.chunk = per * 64;
  p.splits = (int)((red_tiles + per - 1) / per);
  if (p.splits < 1) p.splits = 1;
  return p;
}

// Row reduce out[p, q] = sum_j L[p, j] S(j, q), L [P x J] bf16, S [Q x J]
// (s_qj) or [J x Q] bf16.  Outputs (each optional): out_f32 = v [P x Q],
// out_scaled = bf16(scale v) [P x Q], out_hilo = (bf16(v), bf16(v - bf16(v)))
// side by side [P x 2Q]; and aux_hilo = the same split of aux_src [P x Q]
// fp32, an independent array converted on the way.
struct RowReduce {
  const __nv_bfloat16* L;
  const __nv_bfloat16* S;
  int s_qj;
  int64_t P, J;
  SplitPlan sp;
  float scale;
  float* out_f32;
  __nv_bfloat16* out_scaled;
  __nv_bfloat16* out_hilo;
  const float* aux_src;
  __nv_bfloat16* aux_hilo;
  // S given as [J x Q] (s_qj == 0) only: with bd_nproj > 1, S is read as the
  // block-diagonal spread of B [J x bd_r] (row j of projection p, i.e. j in
  // [bd_end[p-1], bd_end[p]), holds B[j] in columns [p bd_r, (p+1) bd_r) and
  // zeros elsewhere; Q = bd_nproj bd_r), built while the tiles are loaded.
  int bd_nproj;
  int bd_r;
  int64_t bd_end[kMaxProj];
  // grouped: CTA row x reduces tiles[x] = (expert, first row, rows) for
  // x < *tile_count, with S + expert s_stride (the expert's adapter)
  const int4* tiles;
  const int* tile_count;
  int64_t s_stride;
  int max_tiles;  // grouped: grid rows (upper bound of the tile count)
  // stacked adapters: nseg > 0 scales out_scaled column q by seg_scale[i] for
  // q in [seg_end[i-1], seg_end[i]) instead of `scale`
  int nseg;
  int seg_end[kMaxAdapters];
  float seg_scale[kMaxAdapters];
};
// Column reduce out[j, q] = scale sum_p L[p, j] S[p, q], L [P x J] bf16
// (J a multiple of 64), S given as its hi/lo bf16 split [P x 2Q] (hi in
// columns 0..Q-1, lo in Q..2Q-1); tiles = J / 64; out [J x Q], or [Q x J]
// when transposed.
struct ColReduce {
  const __nv_bfloat16* L;
  const __nv_bfloat16* S2;
  int64_t P, J;
  SplitPlan sp;
  int tiles;
  float scale;
  float* out;
  int transposed;
  // window (fused projections' dB): win > 0 keeps, for output rows j of
  // projection p (j in [proj_end[p-1], proj_end[p])), only columns
  // [p win, (p+1) win) of the Q, written as out[j][0..win) (row stride win);
  // win == 0: all Q columns.
  int win;
  int nproj;
  int64_t proj_end[kMaxProj];
  // stacked adapters: nseg > 0 splits the Q columns into segments [seg_end[i-1],
  // seg_end[i]), each with its own scale and its own output array seg_out[i]
  // ([J x w_i], or [w_i x J] transposed, w_i its width; null: not written)
  int nseg;
  int seg_end[kMaxAdapters];
  float seg_scale[kMaxAdapters];
  float* seg_out[kMaxAdapters];
  // grouped (groups > 0, same in both jobs of a launch): output tiles of
  // every expert, reducing over the expert's rows ranges[e]; expert e's
  // output is out + e J Q (zeros for an expert without rows)
  const int2* ranges;
  int groups;
};
// Stacked adapters: A_cat [Q x K] = the adapters' A stacked by rows, B_cat
// [N x Q] = their B side by side (adapter i in columns [off_i, off_i + r_i)).
struct AdapterPack {
  int n;
  int r[kMaxAdapters];
  const __nv_bfloat16* A[kMaxAdapters];
  const __nv_bfloat16* B[kMaxAdapters];
};
cudaError_t launch_pack_adapters(const AdapterPack& ap, int64_t N, int64_t K, __nv_bfloat16* A_cat,
                                 __nv_bfloat16* B_cat, cudaStream_t st);

cudaError_t launch_row_reduce_fin(const RowReduce& r, int Q, cudaStream_t st);
// One launch for one or two column reductions with the same split plan (b
// may be null).
cudaError_t launch_col_reduce_fin(const ColReduce& a, const ColReduce* b, int Q, cudaStream_t st);

// ---- standalone decode (dequant.cu) -------------------------------------------
cudaError_t launch_dequant(int fmt, const WeightView& wv, int64_t lines, __nv_bfloat16* out, cudaStream_t st);

// ---- fused tcgen05 GEMM (gemm_tc.cu) --------------------------------------------
// Tile: 128 output rows x 256 output columns, reduction in chunks of 64.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;

// Grouped problems: up to kMaxGroups row groups (experts), each with its own
// base weight.  Dense problems use one group.
constexpr int kMaxGroups = 256;


// Per-expert weight views of a grouped GEMM, passed as a kernel parameter
// (12 KB for 256 experts), so a call uploads nothing.
struct GroupTable {
  WeightView w[kMaxGroups];
};

// Grouped (mixture-of-experts) schedule, built on the device from the
// experts' row offsets (device memory) by launch_grouped_schedule, so no
// host synchronisation is needed.  Expert e owns rows [ranges[e].x,
// ranges[e].y).  Tile lists hold (expert, first row, rows, column block);
// counts = {GEMM forward tiles, GEMM dX tiles, 64-row tiles}.  Offsets that
// are not a valid partition of [0, M_total) give empty lists and ranges and
// record QLORA_ERR_INVALID in the device error word.
struct GroupedSched {
  int* counts;
  int4* gemm_f;
  int4* gemm_d;
  int4* rows64;
  int2* ranges;
};
// Gate / up with SwiGLU, elementwise parts (swiglu.cu): H = silu(G) U from
// GU = [G | U] ([M x 2I] bf16), and dY = [dG | dU] from dH and GU.
// swiglu_h_f32 takes G and U as stored (bf16 values) and is the one formula
// both the pair GEMM's epilogue and swiglu_act_kernel use, so that H does not
// depend on which of the two computed it.
__device__ __forceinline__ float swiglu_sigmoid_f32(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }
__device__ __forceinline__ float swiglu_h_f32(float g_bf16, float u_bf16) {
  return g_bf16 * swiglu_sigmoid_f32(g_bf16) * u_bf16;
}
cudaError_t launch_swiglu_act(const __nv_bfloat16* GU, __nv_bfloat16* H, int64_t M, int64_t I, cudaStream_t st);
cudaError_t launch_swiglu_grad(const __nv_bfloat16* GU, const __nv_bfloat16* dH, __nv_bfloat16* dY, int64_t M,
                               int64_t I, cudaStream_t st);

cudaError_t launch_grouped_schedule(const int32_t* offsets, int E, int64_t M_total, int tile_rows, int nblk_f,
                                    int nblk_d, const GroupedSched& s, int* err, cudaStream_t st);

// Raw ring geometry (pair kernel): the quantised bytes of one item reach
// shared memory as one byte box per CTA: forward, one 64-element line of each
// of the CTA's weight rows; dX, the CTA's two consecutive lines of each of 64
// weight rows.  raw_line_bytes: bytes of one line in a weight row (Q4_K: the
// code bytes of one 64-element chunk, its 16-byte super-block header comes
// as a second box).  raw_box_bytes: inner box width, the line's bytes from a
// 16-byte aligned start (a Q8_0 / Q4_0 line starts up to 12 bytes past one).
__host__ __device__ constexpr int raw_line_bytes(int fmt) {
  return fmt == 1 ? 32 : fmt == 2 ? 68 : fmt == 3 ? 36 : fmt == 4 ? 32 : fmt == 5 ? 64 : fmt == 6 ? 32 : 0;
}
__host__ __device__ constexpr int raw_box_bytes(int fmt, bool dx) {
  return fmt == 2 ? (dx ? 160 : 80) : fmt == 3 ? (dx ? 96 : 48) : (dx ? 2 : 1) * raw_line_bytes(fmt);
}
// Bytes of one weight row of a format (K elements).
__host__ __device__ constexpr int64_t row_bytes_of(int fmt, int64_t K) {
  return fmt == 0 ? 2 * K : fmt == 1 ? K / 2 : fmt == 2 ? K / 32 * 34 : fmt == 3 ? K / 32 * 18
       : fmt == 4 ? K / 256 * 144 : fmt == 5 ? K : K / 2;
}

struct GemmArgs {
  int M;                 // total rows (of X / dY / output)
  int n_out;             // output columns (N forward, K for dX)
  int k_red;             // reduction length (K forward, N for dX); multiple of 64
  int rank;              // LoRA rank (0: no adapter chunk)
  int num_n_blk;         // ceil(n_out / 256)
  int num_tiles;         // total output tiles
  int64_t w_lines_per_row;  // K_w / 64
  int64_t w_rows;           // N_w
  __nv_bfloat16* out;    // [M x n_out] bf16
  float* out_f32;        // debug: when set, the fp32 accumulators are written here instead of `out`
  // grouped (pair kernel): tile t = tile_sched[t] (expert, first row, rows,
  // column block) for t < *tile_count (both device; written by the schedule
  // kernel earlier in the stream); null for dense problems
  const int4* tile_sched;
  const int* tile_count;
  WeightView wv;
  int* err;              // device error word
  int n_fastest;         // pair kernel tile order: 1 = output column blocks fastest
  int raw_on;            // pair kernel: quantised bytes through the TMA raw ring (maps.w / maps.aq)
  int raw_dq;            // pair kernel, NF4 dX: absmax codes and group scales through the raw ring
  int direct_out;        // pair kernel with one staging tile: bf16 rows stored from registers
  // Gate / up with SwiGLU (forward, pair kernel): swiglu_i = I > 0 reads the
  // base as [gate rows; up rows] (N = 2I) and gives each tile's CTA 0 the
  // gate rows and CTA 1 the matching up rows (columns n0/2 .. of each), so a
  // tile holds gate and up of the same columns; the epilogue writes G | U
  // to `out` ([M x 2I]) and H = silu(G) U to `swiglu_h` ([M x I]).  The
  // adapter chunk takes all 2 rank columns of sT; CTA 1's B box is shifted
  // by rank columns so each half meets its own T.
  int swiglu_i;
  __nv_bfloat16* swiglu_h;
  // Fused projections (forward): projection p owns output columns
  // [proj_end[p-1], proj_end[p]) and adapter columns [p rank, (p+1) rank) of
  // the adapter A operand; a tile never spans two projections.  nproj <= 1:
  // one projection.
  int nproj;
  int proj_end[kMaxProj];
};

// First adapter column (of the adapter A operand) of the projection that owns
// output column n0.
__host__ __device__ __forceinline__ int adapter_col(const GemmArgs& a, int n0) {
  int x = 0;
  for (int p = 0; p + 1 < a.nproj; ++p) x += n0 >= a.proj_end[p] ? a.rank : 0;
  return x;
}

// Tensor maps: A operand [M x k_red] (X or dY), bf16 W (format BF16 only),
// adapter A-operand (sT / sU [M x r]), adapter B-operand (B [N x r] forward,
// A [r x K] for dX).  Grouped bf16 / adapter maps are 3-D with the group
// index outermost.
struct GemmMaps {
  CUtensorMap a, w, la, lb;
  CUtensorMap out;  // pair kernel: bf16 output [M x n_out], box [64 x 128] (TMA stores)
  CUtensorMap aq;   // pair kernel, NF4 dX with raw_dq: int8 absmax codes [N x K/64], box [16 x 64]
};

cudaError_t launch_qgemm(int fmt, bool dx, const GemmMaps& maps, const GemmArgs& args, int num_sms,
                         cudaStream_t st);

// CTA-pair variant (gemm_pair.cu), dense problems only.  Tensor-map boxes:
// A / adapter-A [64 x 128]; bf16 W and adapter-B [64 x tile_cols/2] forward,
// [64 x 64] for dX.  args.num_tiles / num_n_blk count pair tiles.
// Tile configurations: 1 = 256 x 256 (bf16 bases), 3 = 512 x 256 (quantised
// bases), 2 = 512 x 128 (quantised bases, for launches whose 512 x 256 tiles
// would leave most SM pairs idle).
int pair_cfg(int fmt, int64_t M, int64_t n_out, int num_sms);
cudaError_t launch_qgemm_pair(int fmt, bool dx, int cfg, const GemmMaps& maps, const GemmArgs& args,
                              cudaStream_t st);
// Output tile of a configuration.  Forward bf16-W and adapter-B maps use
// boxes of pair_tile_cols / 2 rows.
int pair_tile_rows(int cfg);
int pair_tile_cols(int cfg);
// Grouped calls: configuration 4 (256 x 256) for quantised bases, 1 for bf16.
cudaError_t launch_qgemm_pair_grouped(int fmt, bool dx, const GemmMaps& maps, const GemmArgs& args,
                                      const GroupTable& tab, cudaStream_t st);

}  // namespace qlora
