// C ABI of the quantised-base LoRA linear (declared in include/qlora.h).
//
// Host side only: argument validation, workspace layout, TMA tensor-map
// encoding and the launch sequence of each call.  Every step of the
// computation runs in this library's kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/qlora.h"
#include "kernels.h"

namespace qlora {

__device__ int g_device_error = 0;

static std::atomic<int64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int* device_error_word() {
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(p);
  }
  return cached[dev];
}

// ---------------------------------------------------------------- helpers ---
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

static int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor of `rank` dims (innermost first), 128-byte swizzle, zero fill
// outside the tensor.
static bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                     const uint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3], s[2];
  cuuint32_t b[3], e[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, s, b, e,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static bool map2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                  uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {inner * 2};
  const uint32_t box[2] = {box_inner, box_outer};
  return make_map(m, base, 2, dims, strides, box);
}

// Byte tensor [rows x row_bytes] (row_bytes a multiple of 16), no swizzle,
// zero fill outside the tensor: NF4 code bytes, two codes per byte.
static bool map2d_u8(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                     uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[2] = {row_bytes, rows}, s[1] = {row_bytes};
  cuuint32_t b[2] = {box_bytes, box_rows}, e[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), d, s, b, e,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

static int validate_weight(const qlora_weight_desc* w) {
  if (!w) return QLORA_ERR_INVALID;
  if (w->N <= 0 || w->K <= 0 || (w->N % 64) || (w->K % 64)) return QLORA_ERR_INVALID;
  if (w->N > (1ll << 30) || w->K > (1ll << 30)) return QLORA_ERR_UNSUPPORTED;
  if (!w->data) return QLORA_ERR_INVALID;
  if (!aligned16(w->data)) return QLORA_ERR_ALIGN;
  if (w->reserved != 0) return QLORA_ERR_INVALID;
  if (w->fmt != QLORA_FMT_NF4 && (w->absmax || w->absmax_q || w->absmax_scale || w->absmax_map))
    return QLORA_ERR_INVALID;
  if (w->fmt != QLORA_FMT_FP8_E4M3 && w->fmt != QLORA_FMT_NVFP4 && w->tensor_scale) return QLORA_ERR_INVALID;
  if (w->fmt != QLORA_FMT_NVFP4 && w->block_scale) return QLORA_ERR_INVALID;
  switch (w->fmt) {
    case QLORA_FMT_BF16:
    case QLORA_FMT_Q8_0:
    case QLORA_FMT_Q4_0:
      break;
    case QLORA_FMT_Q4_K:
      if (w->K % 256) return QLORA_ERR_INVALID;
      break;
    case QLORA_FMT_FP8_E4M3:
      if (!w->tensor_scale) return QLORA_ERR_INVALID;
      if (!aligned4(w->tensor_scale)) return QLORA_ERR_ALIGN;
      break;
    case QLORA_FMT_NVFP4:
      if (!w->tensor_scale || !w->block_scale) return QLORA_ERR_INVALID;
      if (!aligned4(w->tensor_scale) || !aligned16(w->block_scale)) return QLORA_ERR_ALIGN;
      break;
    case QLORA_FMT_NF4:
      if (w->absmax) {
        if (!aligned16(w->absmax)) return QLORA_ERR_ALIGN;
        if (w->absmax_q || w->absmax_scale || w->absmax_map) return QLORA_ERR_INVALID;
      } else {
        if (!w->absmax_q || !w->absmax_scale || w->dq_group <= 0) return QLORA_ERR_INVALID;
        if (w->absmax_map && !aligned4(w->absmax_map)) return QLORA_ERR_ALIGN;
        if (w->absmax_map && !std::isfinite(w->absmax_offset)) return QLORA_ERR_INVALID;
      }
      break;
    default:
      return QLORA_ERR_INVALID;
  }
  return QLORA_OK;
}

static int validate_rank(int32_t rank) {
  if (rank < 8 || rank > 64 || (rank % 8)) return QLORA_ERR_INVALID;
  return QLORA_OK;
}

static WeightView view_of(const qlora_weight_desc* w) {
  WeightView v;
  v.data = static_cast<const uint8_t*>(w->data);
  v.absmax = w->absmax;
  v.absmax_q = w->absmax_q;
  v.absmax_scale = w->absmax_scale;
  v.amap = w->fmt == QLORA_FMT_NF4 && !w->absmax ? w->absmax_map : nullptr;
  v.aoff = w->absmax_offset;
  v.tscale = w->tensor_scale;
  v.bscale = w->block_scale;
  v.dq_group = w->dq_group > 0 ? w->dq_group : 1;
  v.aq_align8 = (reinterpret_cast<uintptr_t>(w->absmax_q) & 7u) == 0 ? 1 : 0;
  v.dq_shift = -1;
  for (int b = 0; b < 31; ++b)
    if (v.dq_group == (1 << b)) v.dq_shift = b;
  v.fmt = w->fmt;
  return v;
}

// ------------------------------------------------------- workspace layout ---
struct DenseLayout {
  size_t act_off, act_bytes;  // sT or sU, bf16 [M x r]
  size_t u_off, u_bytes;      // U as hi/lo bf16 [M x 2r] (backward)
  size_t t_off, t_bytes;      // T as hi/lo bf16 [M x 2r] (backward)
  int64_t db_tiles, da_tiles;
  SplitPlan t, u, c;          // T = X A^T, U = dY B, and dB / dA (one launch)
  size_t total;
};

static DenseLayout dense_layout(int64_t M, int64_t N, int64_t K, int r) {
  DenseLayout L;
  const int64_t row_tiles = (M + 63) / 64;
  L.db_tiles = N / 64;
  L.da_tiles = K / 64;
  L.t = plan_split_fin(row_tiles, K);
  L.u = plan_split_fin(row_tiles, N);
  L.c = plan_split_fin(L.db_tiles + L.da_tiles, M);
  L.act_off = 0;
  L.act_bytes = round256((size_t)M * r * 2);
  L.u_off = L.act_off + L.act_bytes;
  L.u_bytes = round256((size_t)M * r * 4);
  L.t_off = L.u_off + L.u_bytes;
  L.t_bytes = round256((size_t)M * r * 4);
  L.total = L.t_off + L.t_bytes;
  return L;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA; }

// ------------------------------------------------------------ side stream ---
// A second stream per device for work of a call that may run beside the
// call's main kernels: the backward call's adapter-gradient reduction runs
// beside its dX GEMM, whose last partial wave of tiles leaves SMs idle.  The
// call forks the side stream from the caller's stream and joins it back with
// events before returning, so all of the call's work stays ordered on the
// caller's stream.  The fork / launch / join sequence of one call is done
// under a lock, so calls from several host threads do not interleave it.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool ok = false;
};
static std::mutex g_side_mu;
static SideStream g_side[64];

static SideStream* side_stream_locked() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream& ss = g_side[dev];
  if (!ss.ok) {
    if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
    ss.ok = true;
  }
  return &ss;
}

// ------------------------------------------------ GEMM instrumentation ------
struct GemmRec {
  cudaEvent_t a, b;
  double flops;
};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static std::vector<GemmRec> g_prof_recs;
static std::vector<cudaEvent_t> g_prof_pool;

static cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Run `launch` (one fused GEMM launch on st), bracketed by events when
// instrumentation is on.
template <class F>
static cudaError_t timed_gemm(const GemmArgs& a, cudaStream_t st, F&& launch) {
  std::unique_lock<std::mutex> g(g_prof_mu);
  if (!g_prof_on) {
    g.unlock();
    return launch();
  }
  GemmRec r;
  r.a = prof_event();
  r.b = prof_event();
  r.flops = 2.0 * (double)a.M * (double)a.n_out * (double)(a.k_red + a.rank);
  cudaEventRecord(r.a, st);
  cudaError_t e = launch();
  cudaEventRecord(r.b, st);
  g_prof_recs.push_back(r);
  return e;
}

// pair: 0 = one CTA per tile, else the pair kernel's tile configuration.
static cudaError_t gemm_launch(int fmt, bool dx, int pair, const GemmMaps& maps, const GemmArgs& a,
                               cudaStream_t st) {
  return timed_gemm(a, st, [&] {
    return pair ? launch_qgemm_pair(fmt, dx, pair, maps, a, st) : launch_qgemm(fmt, dx, maps, a, sm_count(), st);
  });
}

// Output columns owned by each of P fused projections (cumulative ends).
struct ProjSplit {
  int P = 1;
  int64_t end[kMaxProj] = {0};
};

// Dense fused GEMM: forward (dx = false) out = A_op W^T + la lb^T with
// A_op = X [M x K], la = sT, lb = B [N x r]; dX (dx = true) out = A_op W +
// la lb with A_op = dY [M x N], la = sU, lb = A [r x K].  la has la_cols
// columns; with fused projections (forward, ps->P > 1) a tile's adapter chunk
// takes the `rank` columns of its projection.
// out_f32 (debug): when set, the fp32 accumulators are written there
// ([M x n_out]) instead of bf16 to `out`.  swiglu_i > 0 (forward, a base of
// [gate rows; up rows] with I rows each, fused as two projections): `out`
// receives G | U and swiglu_h H = silu(G) U ([M x I]) — from the pair
// kernel's epilogue, or for launches of at most 128 rows by an elementwise
// pass over G | U.
static cudaError_t run_dense_gemm(const qlora_weight_desc* w, bool dx, int64_t M, int rank, int la_cols,
                                  const ProjSplit* ps, const void* a_op, const void* la, const void* lb, void* out,
                                  cudaStream_t st, float* out_f32 = nullptr, int64_t swiglu_i = 0,
                                  void* swiglu_h = nullptr) {
  if (out_f32) out = out_f32;  // the bf16 store map is then built but never used
  const int64_t N = w->N, K = w->K;
  // pair tiles on an SM pair; short problems use one CTA per 128 x 256 tile
  const int pair = M > kBM ? pair_cfg(w->fmt, M, dx ? K : N, sm_count()) : 0;
  const int tile_rows = pair ? pair_tile_rows(pair) : kBM;
  const int tile_cols = pair ? pair_tile_cols(pair) : kBN;
  const uint32_t brows = pair ? (uint32_t)(tile_cols / 2) : 256;
  GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  bool ok;
  if (!dx) {
    ok = map2d(&maps.a, a_op, K, M, 64, 128) && map2d(&maps.la, la, la_cols, M, 64, 128) &&
         map2d(&maps.lb, lb, rank, N, 64, brows);
    if (w->fmt == QLORA_FMT_BF16) ok = ok && map2d(&maps.w, w->data, K, N, 64, brows);
  } else {
    ok = map2d(&maps.a, a_op, N, M, 64, 128) && map2d(&maps.la, la, la_cols, M, 64, 128) &&
         map2d(&maps.lb, lb, K, rank, 64, 64);
    if (w->fmt == QLORA_FMT_BF16) ok = ok && map2d(&maps.w, w->data, K, N, 64, 64);
  }
  if (pair) ok = ok && map2d(&maps.out, out, dx ? K : N, M, 64, 128);
  // NF4 on 512 x 256 pair tiles: code bytes [N x K/2] through the raw ring,
  // one box per item (forward: 128 weight rows x one 64-element block; dX:
  // 64 weight rows x the CTA's two blocks)
  if (pair == 3 && w->fmt == QLORA_FMT_NF4)
    ok = ok && (dx ? map2d_u8(&maps.w, w->data, K / 2, N, 64, 64) : map2d_u8(&maps.w, w->data, K / 2, N, 32, 128));
  // dX with a double-quantised absmax: the int8 codes [N x K/64] and the
  // group scales also through the raw ring, where the layout allows: 16-byte
  // aligned arrays, code rows a multiple of 16 bytes, power-of-two groups, a
  // scale array of whole 16-byte pieces, and an item's scales within the
  // ring slot's 64 (at most ((63 K/64 + 1) >> log2 group) + 8 of them)
  int raw_dq = 0;
  if (ok && pair == 3 && dx && w->fmt == QLORA_FMT_NF4 && !w->absmax) {
    const int64_t lpr = K / 64;
    const WeightView v = view_of(w);
    const int64_t groups = (N * lpr + v.dq_group - 1) / v.dq_group;
    if (lpr % 16 == 0 && aligned16(w->absmax_q) && aligned16(w->absmax_scale) && v.dq_shift >= 0 &&
        groups % 4 == 0 && ((63 * lpr + 1) >> v.dq_shift) + 8 <= 64)
      raw_dq = map2d_u8(&maps.aq, w->absmax_q, lpr, N, 16, 64) ? 1 : 0;
  }
  if (!ok) return cudaErrorInvalidValue;
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.M = (int)M;
  a.n_out = (int)(dx ? K : N);
  a.k_red = (int)(dx ? N : K);
  a.rank = rank;
  a.num_n_blk = (a.n_out + tile_cols - 1) / tile_cols;
  a.num_tiles = (int)(((M + tile_rows - 1) / tile_rows) * a.num_n_blk);
  a.w_lines_per_row = K / 64;
  a.w_rows = N;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.out_f32 = out_f32;
  a.wv = view_of(w);
  a.err = device_error_word();
  a.raw_dq = raw_dq;
  a.raw_on = (pair == 3 && w->fmt == QLORA_FMT_NF4) ? 1 : 0;
  // the configurations with one epilogue staging tile (512 x 128 tiles; NF4
  // on 512 x 256 tiles) store outputs of at most 4096 columns straight from
  // registers: measured on the Llama layer, o and down forward 2-5 % and
  // gate|up dX 2 % faster that way, wider outputs 1-4 % slower
  a.direct_out = (pair == 2 || (pair == 3 && w->fmt == QLORA_FMT_NF4)) && a.n_out <= 4096 ? 1 : 0;
  // Tile order.  Forward: row blocks fastest while the activation fits in L2
  // next to the streamed weight slabs (measured: gate 133 MB of DRAM traffic
  // this way vs 234 MB the other way); beyond ~64 MB (e.g. the 14336-wide
  // down projection) column blocks fastest, so each activation row block is
  // read once (543 -> 253 MB).  dX: column blocks fastest, so each dY row
  // block is read once.
  a.n_fastest = dx ? 1 : ((double)M * (double)a.k_red * 2.0 > 64e6 ? 1 : 0);
  if (!dx && ps && ps->P > 1) {
    a.nproj = ps->P;
    for (int p = 0; p < ps->P; ++p) a.proj_end[p] = (int)ps->end[p];
  }
  if (swiglu_i > 0 && pair) {
    // one adapter chunk of both projections' columns; each CTA's B half is
    // shifted onto its projection's columns in the kernel
    a.swiglu_i = (int)swiglu_i;
    a.swiglu_h = static_cast<__nv_bfloat16*>(swiglu_h);
    a.rank = la_cols;
    a.nproj = 0;
  }
  cudaError_t e = gemm_launch(w->fmt, dx, pair, maps, a, st);
  if (e == cudaSuccess && swiglu_i > 0 && !pair)
    e = launch_swiglu_act(static_cast<const __nv_bfloat16*>(out), static_cast<__nv_bfloat16*>(swiglu_h), M,
                          swiglu_i, st);
  return e;
}


// ------------------------------------------------------------- grouped ------
// Workspace of a grouped call.  The tile lists are sized for their upper
// bounds (expert e has ceil(c_e / rows) <= c_e / rows + 1 row tiles), so the
// layout depends on E and M_total only and the lists are filled on the device
// from the device offsets.
constexpr int kGroupTileRows = 256;  // rows of a grouped GEMM tile

struct GroupedLayout {
  int E = 0, r = 0;
  int64_t M = 0, N = 0, K = 0;
  int nblk_f = 0, nblk_d = 0;   // GEMM column blocks, forward / dX
  int max_gemm_rows = 0;        // bound on the GEMM row tiles of all experts
  int max_rows64 = 0;           // bound on the 64-row reduction tiles
  size_t off_counts = 0, off_gf = 0, off_gd = 0, off_rr = 0, off_rg = 0;
  size_t off_act = 0, off_u2 = 0, off_t2 = 0, total = 0;
};

static int validate_grouped(const qlora_weight_desc* ex, int E, int64_t M_total, int r) {
  if (!ex || E <= 0 || E > kMaxGroups || M_total < 0) return QLORA_ERR_INVALID;
  int v = validate_rank(r);
  if (v != QLORA_OK) return v;
  for (int e = 0; e < E; ++e) {
    if ((v = validate_weight(&ex[e])) != QLORA_OK) return v;
    if (ex[e].fmt != ex[0].fmt || ex[e].N != ex[0].N || ex[e].K != ex[0].K) return QLORA_ERR_INVALID;
  }
  if (M_total > (1 << 30)) return QLORA_ERR_UNSUPPORTED;
  return QLORA_OK;
}

static GroupedLayout grouped_layout(const qlora_weight_desc* ex, int E, int64_t M, int r) {
  GroupedLayout L;
  L.E = E;
  L.r = r;
  L.M = M;
  L.N = ex[0].N;
  L.K = ex[0].K;
  L.nblk_f = (int)((L.N + 255) / 256);
  L.nblk_d = (int)((L.K + 255) / 256);
  L.max_gemm_rows = (int)((M + kGroupTileRows - 1) / kGroupTileRows) + E;
  L.max_rows64 = (int)((M + 63) / 64) + E;
  size_t o = 0;
  L.off_counts = o;
  o = round256(o + 4 * sizeof(int));
  L.off_gf = o;
  o = round256(o + sizeof(int4) * (size_t)L.max_gemm_rows * L.nblk_f);
  L.off_gd = o;
  o = round256(o + sizeof(int4) * (size_t)L.max_gemm_rows * L.nblk_d);
  L.off_rr = o;
  o = round256(o + sizeof(int4) * (size_t)L.max_rows64);
  L.off_rg = o;
  o = round256(o + sizeof(int2) * (size_t)E);
  L.off_act = o;  // sT (forward) or sU (backward), bf16 [M x r]
  o = round256(o + (size_t)M * r * 2);
  L.off_u2 = o;  // U as hi/lo bf16 [M x 2r] (backward)
  o = round256(o + (size_t)M * r * 4);
  L.off_t2 = o;  // T as hi/lo bf16 [M x 2r] (backward)
  o = round256(o + (size_t)M * r * 4);
  L.total = o;
  return L;
}

static GroupedSched grouped_sched(const GroupedLayout& L, uint8_t* ws) {
  GroupedSched g;
  g.counts = reinterpret_cast<int*>(ws + L.off_counts);
  g.gemm_f = reinterpret_cast<int4*>(ws + L.off_gf);
  g.gemm_d = reinterpret_cast<int4*>(ws + L.off_gd);
  g.rows64 = reinterpret_cast<int4*>(ws + L.off_rr);
  g.ranges = reinterpret_cast<int2*>(ws + L.off_rg);
  return g;
}

// bf16 [E][mid][inner] as a 3-D tensor (innermost first), box {64, rows, 1}
static bool map3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t E, uint32_t box_rows) {
  const uint64_t dims[3] = {inner, mid, E};
  const uint64_t strides[2] = {inner * 2, inner * mid * 2};
  const uint32_t box[3] = {64, box_rows, 1};
  return make_map(m, base, 3, dims, strides, box);
}

// Expert bases back to back in one array [E][N][row bytes] (read through
// one 3-D map: required for bf16, the fast path for quantised bases)
static bool experts_stacked(const qlora_weight_desc* ex, int E) {
  const uint8_t* b0 = static_cast<const uint8_t*>(ex[0].data);
  const size_t stride = (size_t)ex[0].N * (size_t)row_bytes_of(ex[0].fmt, ex[0].K);
  for (int e = 1; e < E; ++e)
    if (static_cast<const uint8_t*>(ex[e].data) != b0 + (size_t)e * stride) return false;
  return true;
}

// Byte tensor [E][N][row_bytes] (row_bytes a multiple of 16), box
// {box_bytes, box_rows, 1}, no swizzle
static bool map3d_u8(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t E,
                     uint32_t box_bytes, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3] = {row_bytes, rows, E}, s[2] = {row_bytes, row_bytes * rows};
  cuuint32_t b[3] = {box_bytes, box_rows, 1}, e[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), d, s, b, e,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Grouped fused GEMM over the schedule's tile list: forward Y = X deq(W_e)^T
// + sT B_e^T, dX = dY deq(W_e) + sU A_e, 256 x 256 tiles on SM pairs.
static cudaError_t run_grouped_gemm(const qlora_weight_desc* ex, const GroupedLayout& L, bool dx,
                                    const GroupedSched& g, const void* a_op, const void* la, const void* lb,
                                    void* out, cudaStream_t st) {
  const int64_t M = L.M, N = L.N, K = L.K;
  const int E = L.E, r = L.r;
  GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  bool ok;
  if (!dx) {
    ok = map2d(&maps.a, a_op, K, M, 64, 128) && map2d(&maps.la, la, r, M, 64, 128) &&
         map3d(&maps.lb, lb, r, N, E, 128);
    if (ex[0].fmt == QLORA_FMT_BF16) ok = ok && map3d(&maps.w, ex[0].data, K, N, E, 128);
  } else {
    ok = map2d(&maps.a, a_op, N, M, 64, 128) && map2d(&maps.la, la, r, M, 64, 128) &&
         map3d(&maps.lb, lb, K, r, E, 64);
    if (ex[0].fmt == QLORA_FMT_BF16) ok = ok && map3d(&maps.w, ex[0].data, K, N, E, 64);
  }
  ok = ok && map2d(&maps.out, out, dx ? K : N, M, 64, 128);
  // quantised bases back to back with 16-byte multiple rows: their bytes
  // through the raw ring (one 3-D byte box per item; Q4_K headers as a second)
  const int fmt = ex[0].fmt;
  const int64_t rb = row_bytes_of(fmt, K);
  int raw_on = 0;
  if (ok && fmt != QLORA_FMT_BF16 && rb % 16 == 0 && experts_stacked(ex, E)) {
    const uint32_t rows = dx ? 64 : 128;
    raw_on = map3d_u8(&maps.w, ex[0].data, rb, N, E, raw_box_bytes(fmt, dx), rows) ? 1 : 0;
    if (raw_on && fmt == QLORA_FMT_Q4_K) raw_on = map3d_u8(&maps.aq, ex[0].data, rb, N, E, 16, rows) ? 1 : 0;
  }
  if (!ok) return cudaErrorInvalidValue;
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.M = (int)M;
  a.n_out = (int)(dx ? K : N);
  a.k_red = (int)(dx ? N : K);
  a.rank = r;
  a.num_n_blk = dx ? L.nblk_d : L.nblk_f;
  a.num_tiles = L.max_gemm_rows * a.num_n_blk;  // bound; the count is on the device
  a.w_lines_per_row = K / 64;
  a.w_rows = N;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.tile_sched = dx ? g.gemm_d : g.gemm_f;
  a.tile_count = g.counts + (dx ? 1 : 0);
  a.raw_on = raw_on;
  a.wv = view_of(&ex[0]);
  a.err = device_error_word();
  static thread_local GroupTable tab;  // 12 KB: kept off the stack
  for (int e = 0; e < E; ++e) tab.w[e] = view_of(&ex[e]);
  return timed_gemm(a, st, [&] { return launch_qgemm_pair_grouped(ex[0].fmt, dx, maps, a, tab, st); });
}

// Splits of the grouped column reductions: one CTA per (expert, output tile)
// already gives E (tiles) CTAs; split each expert's rows only when that is
// far below the target.
static SplitPlan grouped_col_split(const GroupedLayout& L, int64_t tiles) {
  SplitPlan sp;
  int64_t s = kSplitTargetCtas / std::max<int64_t>(tiles * L.E, 1);
  const int64_t mean_rows64 = std::max<int64_t>((L.M + 63) / 64 / L.E, 1);
  s = std::min<int64_t>(s, std::max<int64_t>(mean_rows64 / 2, 1));
  s = std::min<int64_t>(std::max<int64_t>(s, 1), kMaxClusterSplits);
  sp.splits = (int)s;
  sp.chunk = 0;  // grouped: each expert's rows are split evenly
  return sp;
}

}  // namespace qlora

using namespace qlora;

// =============================================================================
extern "C" {

const char* qlora_status_string(int32_t s) {
  switch (s) {
    case QLORA_OK: return "ok";
    case QLORA_ERR_INVALID: return "invalid argument";
    case QLORA_ERR_UNSUPPORTED: return "unsupported";
    case QLORA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case QLORA_ERR_CUDA: return "CUDA error";
    case QLORA_ERR_TIMEOUT: return "device wait timed out";
    case QLORA_ERR_WORKSPACE: return "workspace missing or too small";
    case QLORA_ERR_STATE: return "streaming pool used out of order";
    default: return "unknown status";
  }
}

int32_t qlora_version(void) { return 200; }

int64_t qlora_launch_count(void) { return g_launches.load(); }

int32_t qlora_profile_gemm(int32_t enable) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  if (enable) {
    for (auto& r : g_prof_recs) {
      g_prof_pool.push_back(r.a);
      g_prof_pool.push_back(r.b);
    }
    g_prof_recs.clear();
  }
  g_prof_on = enable != 0;
  return QLORA_OK;
}

int32_t qlora_profile_gemm_read(double* total_ms, int64_t* launches, double* flops) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  double ms = 0.0, fl = 0.0;
  for (auto& r : g_prof_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return QLORA_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return QLORA_ERR_CUDA;
    ms += t;
    fl += r.flops;
  }
  if (total_ms) *total_ms = ms;
  if (launches) *launches = (int64_t)g_prof_recs.size();
  if (flops) *flops = fl;
  return QLORA_OK;
}

int32_t qlora_device_error(int32_t clear) {
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return QLORA_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return QLORA_ERR_CUDA;
  if (clear) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_device_error, &z, sizeof(int)) != cudaSuccess) return QLORA_ERR_CUDA;
  }
  return v;
}

int32_t qlora_last_device_error(void* stream, int32_t clear) {
  // stream-ordered read: the copy runs after the stream's earlier work, and
  // only this stream is waited for
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* word = device_error_word();
  if (!word) return QLORA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyAsync(&v, word, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return QLORA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return QLORA_ERR_CUDA;
  if (clear && v != 0) {
    if (cudaMemsetAsync(word, 0, sizeof(int), st) != cudaSuccess) return QLORA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return QLORA_ERR_CUDA;
  }
  return v;
}

size_t qlora_workspace_bytes(const qlora_weight_desc* w, int64_t M, int32_t rank) {
  if (validate_weight(w) != QLORA_OK || validate_rank(rank) != QLORA_OK || M < 0) return 0;
  if (M == 0) return 256;
  return dense_layout(M, w->N, w->K, rank).total;
}

size_t qlora_forward_workspace_bytes(const qlora_weight_desc* w, int64_t M, int32_t rank) {
  if (validate_weight(w) != QLORA_OK || validate_rank(rank) != QLORA_OK || M < 0) return 0;
  if (M == 0) return 256;
  const DenseLayout L = dense_layout(M, w->N, w->K, rank);
  return L.act_off + L.act_bytes;
}

int32_t dequant_blocks(const qlora_weight_desc* w, void* W_bf16, void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  if (!W_bf16) return QLORA_ERR_INVALID;
  if (!aligned16(W_bf16)) return QLORA_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t lines = w->N * (w->K / 64);
  if (w->fmt == QLORA_FMT_BF16)
    return cuda_status(cudaMemcpyAsync(W_bf16, w->data, (size_t)(w->N * w->K * 2), cudaMemcpyDeviceToDevice, st));
  return cuda_status(launch_dequant(w->fmt, view_of(w), lines, static_cast<__nv_bfloat16*>(W_bf16), st));
}

}  // extern "C"

namespace qlora {

// Fused projections: P >= 1, widths summing to N; with P > 1 each width a
// multiple of 256 (no GEMM tile spans two projections) and P rank <= 64
// (their adapters form one reduction chunk).
static int validate_split(const qlora_weight_desc* w, int32_t P, const int64_t* n_split, int32_t rank,
                          ProjSplit& ps) {
  if (P < 1 || P > kMaxProj || !n_split) return QLORA_ERR_INVALID;
  int64_t o = 0;
  for (int p = 0; p < P; ++p) {
    if (n_split[p] <= 0) return QLORA_ERR_INVALID;
    if (P > 1 && n_split[p] % 256) return QLORA_ERR_UNSUPPORTED;
    o += n_split[p];
    ps.end[p] = o;
  }
  if (o != w->N) return QLORA_ERR_INVALID;
  if ((int64_t)P * rank > 64) return QLORA_ERR_UNSUPPORTED;
  ps.P = P;
  return QLORA_OK;
}

// Workspace of a (possibly fused) call: the dense layout for the P rank
// adapter columns.
static size_t multi_workspace(const qlora_weight_desc* w, const ProjSplit& ps, int64_t M, int rank) {
  return dense_layout(M, w->N, w->K, ps.P * rank).total;
}

// Y32 (debug): when set, Y is written there as fp32 instead of bf16 to Y.
// H (gate / up with SwiGLU, two projections of I rows): Y receives G | U and
// H = silu(G) U.
static int32_t linear_fwd_impl(const qlora_weight_desc* w, const ProjSplit& ps, int64_t M, int32_t rank,
                               float alpha, const void* X, const void* A, const void* B, void* Y, float* T_save,
                               void* workspace, size_t ws_bytes, void* stream, float* Y32 = nullptr,
                               void* H = nullptr) {
  if (M < 0 || !std::isfinite(alpha)) return QLORA_ERR_INVALID;
  if (M == 0) return QLORA_OK;
  if (M > (1ll << 31) - 256) return QLORA_ERR_UNSUPPORTED;
  if (!X || !A || !B || !Y || !T_save) return QLORA_ERR_INVALID;
  if (!aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(Y) || !aligned16(T_save))
    return QLORA_ERR_ALIGN;
  const int64_t N = w->N, K = w->K;
  const int Q = ps.P * rank;  // adapter columns of all projections
  const DenseLayout L = dense_layout(M, N, K, Q);
  // the forward uses only the scaled-activation region of the layout
  if (!workspace || ws_bytes < L.act_off + L.act_bytes) return QLORA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QLORA_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* sT = reinterpret_cast<__nv_bfloat16*>(ws + L.act_off);
  const float s = alpha / (float)rank;

  // 1) T = X A^T (split over K; A is every projection's adapter stacked by
  //    rows): T_save = T (fp32), sT = bf16(s T)
  RowReduce rt = {};
  rt.L = static_cast<const __nv_bfloat16*>(X);
  rt.S = static_cast<const __nv_bfloat16*>(A);
  rt.s_qj = 1;
  rt.P = M;
  rt.J = K;
  rt.sp = L.t;
  rt.scale = s;
  rt.out_f32 = T_save;
  rt.out_scaled = sT;
  if (launch_row_reduce_fin(rt, Q, st) != cudaSuccess) return QLORA_ERR_CUDA;

  // 2) Y = X deq(W)^T + sT B^T, each tile's adapter chunk from its projection
  const int64_t swiglu_i = H ? ps.end[0] : 0;
  return cuda_status(run_dense_gemm(w, false, M, rank, Q, &ps, X, sT, B, Y, st, Y32, swiglu_i, H));
}

// dX32 (debug): when set, dX is written there as fp32 instead of bf16 to dX.
static int32_t linear_bwd_impl(const qlora_weight_desc* w, const ProjSplit& ps, int64_t M, int32_t rank,
                               float alpha, const void* X, const void* A, const void* B, const float* T_save,
                               const void* dY, void* dX, float* dA, float* dB, void* workspace, size_t ws_bytes,
                               void* stream, float* dX32 = nullptr) {
  if (M < 0 || !std::isfinite(alpha)) return QLORA_ERR_INVALID;
  if (!dA || !dB) return QLORA_ERR_INVALID;
  const int64_t N = w->N, K = w->K;
  const int Q = ps.P * rank;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M == 0) {  // no rows: the adapter gradients are zero
    if (cudaMemsetAsync(dA, 0, (size_t)Q * K * 4, st) != cudaSuccess) return QLORA_ERR_CUDA;
    return cuda_status(cudaMemsetAsync(dB, 0, (size_t)N * rank * 4, st));
  }
  if (M > (1ll << 31) - 256) return QLORA_ERR_UNSUPPORTED;
  if (!X || !A || !B || !T_save || !dY) return QLORA_ERR_INVALID;
  if (!aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(T_save) || !aligned16(dY) ||
      !aligned16(dA) || !aligned16(dB) || (dX && !aligned16(dX)))
    return QLORA_ERR_ALIGN;
  const DenseLayout L = dense_layout(M, N, K, Q);
  if (!workspace || ws_bytes < multi_workspace(w, ps, M, rank)) return QLORA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QLORA_ERR_ALIGN;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* sU = reinterpret_cast<__nv_bfloat16*>(ws + L.act_off);
  __nv_bfloat16* U2 = reinterpret_cast<__nv_bfloat16*>(ws + L.u_off);
  __nv_bfloat16* T2 = reinterpret_cast<__nv_bfloat16*>(ws + L.t_off);
  const float s = alpha / (float)rank;
  const __nv_bfloat16* Xb = static_cast<const __nv_bfloat16*>(X);
  const __nv_bfloat16* dYb = static_cast<const __nv_bfloat16*>(dY);

  // 1) U = dY B (split over N): sU = bf16(s U) for the dX GEMM, U and T_save
  //    as hi/lo bf16 pairs for the dA / dB reductions.  Fused projections:
  //    B is read spread block-diagonally, so projection p's columns of U see
  //    only its own rows of dY and B.
  RowReduce ru = {};
  ru.L = dYb;
  ru.S = static_cast<const __nv_bfloat16*>(B);
  if (ps.P > 1) {
    ru.bd_nproj = ps.P;
    ru.bd_r = rank;
    for (int p = 0; p < ps.P; ++p) ru.bd_end[p] = ps.end[p];
  }
  ru.s_qj = 0;
  ru.P = M;
  ru.J = N;
  ru.sp = L.u;
  ru.scale = s;
  ru.out_scaled = sU;
  ru.out_hilo = U2;
  ru.aux_src = T_save;
  ru.aux_hilo = T2;
  if (launch_row_reduce_fin(ru, Q, st) != cudaSuccess) return QLORA_ERR_CUDA;

  // 2) dB = s dY^T T and dA = s U^T X (split over M, one launch); dA is
  //    reduced as dA^T [K x Q] and written transposed; fused projections
  //    keep, per row of dB, the columns of its own projection
  ColReduce cb = {};
  cb.L = dYb;
  cb.S2 = T2;
  cb.P = M;
  cb.J = N;
  cb.sp = L.c;
  cb.tiles = (int)L.db_tiles;
  cb.scale = s;
  cb.out = dB;
  cb.transposed = 0;
  if (ps.P > 1) {
    cb.win = rank;
    cb.nproj = ps.P;
    for (int p = 0; p < ps.P; ++p) cb.proj_end[p] = ps.end[p];
  }
  ColReduce ca = {};
  ca.L = Xb;
  ca.S2 = U2;
  ca.P = M;
  ca.J = K;
  ca.sp = L.c;
  ca.tiles = (int)L.da_tiles;
  ca.scale = s;
  ca.out = dA;
  ca.transposed = 1;
  if (!dX) return cuda_status(launch_col_reduce_fin(cb, &ca, Q, st));

  // 3) dX = dY deq(W) + sU A on the caller's stream (over all projections'
  //    rows: their input gradients summed), with step 2 beside it on the
  //    side stream (both only read what step 1 wrote)
  std::lock_guard<std::mutex> g(g_side_mu);
  SideStream* ss = side_stream_locked();
  if (!ss) {
    if (run_dense_gemm(w, true, M, Q, Q, nullptr, dY, sU, A, dX, st, dX32) != cudaSuccess) return QLORA_ERR_CUDA;
    return cuda_status(launch_col_reduce_fin(cb, &ca, Q, st));
  }
  cudaError_t e = cudaEventRecord(ss->fork, st);
  if (e == cudaSuccess) e = run_dense_gemm(w, true, M, Q, Q, nullptr, dY, sU, A, dX, st, dX32);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->s, ss->fork, 0);
  if (e == cudaSuccess) e = launch_col_reduce_fin(cb, &ca, Q, ss->s);
  if (e == cudaSuccess) e = cudaEventRecord(ss->join, ss->s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ss->join, 0);
  return cuda_status(e);
}

}  // namespace qlora

extern "C" {

int32_t qlora_linear_fwd(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha, const void* X,
                         const void* A, const void* B, void* Y, float* T_save, void* workspace, size_t ws_bytes,
                         void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  if ((v = validate_rank(rank)) != QLORA_OK) return v;
  ProjSplit ps;
  ps.end[0] = w->N;
  return linear_fwd_impl(w, ps, M, rank, alpha, X, A, B, Y, T_save, workspace, ws_bytes, stream);
}

int32_t qlora_linear_bwd(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha, const void* X,
                         const void* A, const void* B, const float* T_save, const void* dY, void* dX, float* dA,
                         float* dB, void* workspace, size_t ws_bytes, void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  if ((v = validate_rank(rank)) != QLORA_OK) return v;
  ProjSplit ps;
  ps.end[0] = w->N;
  return linear_bwd_impl(w, ps, M, rank, alpha, X, A, B, T_save, dY, dX, dA, dB, workspace, ws_bytes, stream);
}

// Gate / up with SwiGLU: the fused two-projection call over [gate rows; up
// rows] with the activation in the forward's epilogue and its derivative in
// an elementwise pass before the backward.
static int validate_swiglu(const qlora_weight_desc* w, int32_t rank, ProjSplit& ps) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  if ((v = validate_rank(rank)) != QLORA_OK) return v;
  if (w->N % 512) return QLORA_ERR_UNSUPPORTED;  // I = N/2 a multiple of 256
  if (2 * rank > 64) return QLORA_ERR_UNSUPPORTED;
  ps.P = 2;
  ps.end[0] = w->N / 2;
  ps.end[1] = w->N;
  return QLORA_OK;
}

size_t qlora_swiglu_workspace_bytes(const qlora_weight_desc* w, int64_t M, int32_t rank) {
  ProjSplit ps;
  if (M < 0 || validate_swiglu(w, rank, ps) != QLORA_OK) return 0;
  if (M == 0) return 256;
  return round256((size_t)M * w->N * 2) + multi_workspace(w, ps, M, rank);
}

int32_t qlora_swiglu_fwd(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha, const void* X,
                         const void* A, const void* B, void* H, void* GU, float* T_save, void* workspace,
                         size_t ws_bytes, void* stream) {
  ProjSplit ps;
  const int v = validate_swiglu(w, rank, ps);
  if (v != QLORA_OK) return v;
  if (M > 0 && !H) return QLORA_ERR_INVALID;
  if (H && !aligned16(H)) return QLORA_ERR_ALIGN;
  return linear_fwd_impl(w, ps, M, rank, alpha, X, A, B, GU, T_save, workspace, ws_bytes, stream, nullptr, H);
}

int32_t qlora_swiglu_bwd(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha, const void* X,
                         const void* A, const void* B, const float* T_save, const void* GU, const void* dH,
                         void* dX, float* dA, float* dB, void* workspace, size_t ws_bytes, void* stream) {
  ProjSplit ps;
  const int v = validate_swiglu(w, rank, ps);
  if (v != QLORA_OK) return v;
  if (M < 0 || !std::isfinite(alpha)) return QLORA_ERR_INVALID;
  if (M == 0) return linear_bwd_impl(w, ps, M, rank, alpha, X, A, B, T_save, nullptr, dX, dA, dB, workspace, ws_bytes,
                                     stream);
  if (!GU || !dH) return QLORA_ERR_INVALID;
  if (!aligned16(GU) || !aligned16(dH)) return QLORA_ERR_ALIGN;
  if (!workspace || ws_bytes < qlora_swiglu_workspace_bytes(w, M, rank)) return QLORA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QLORA_ERR_ALIGN;
  // dY = [dG | dU] in the workspace's head, the backward's own layout after it
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t dy_bytes = round256((size_t)M * w->N * 2);
  __nv_bfloat16* dY = reinterpret_cast<__nv_bfloat16*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_swiglu_grad(static_cast<const __nv_bfloat16*>(GU), static_cast<const __nv_bfloat16*>(dH), dY, M,
                         w->N / 2, st) != cudaSuccess)
    return QLORA_ERR_CUDA;
  return linear_bwd_impl(w, ps, M, rank, alpha, X, A, B, T_save, dY, dX, dA, dB, ws + dy_bytes,
                         ws_bytes - dy_bytes, stream);
}

// Debug: the same calls with the GEMM output (Y, resp. dX) written as the
// fp32 accumulator values instead of bf16.
int32_t qlora_debug_linear_fwd_f32(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha, const void* X,
                                   const void* A, const void* B, float* Y32, float* T_save, void* workspace,
                                   size_t ws_bytes, void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  if ((v = validate_rank(rank)) != QLORA_OK) return v;
  if (!Y32) return QLORA_ERR_INVALID;
  ProjSplit ps;
  ps.end[0] = w->N;
  return linear_fwd_impl(w, ps, M, rank, alpha, X, A, B, Y32, T_save, workspace, ws_bytes, stream, Y32);
}

int32_t qlora_debug_linear_bwd_f32(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha, const void* X,
                                   const void* A, const void* B, const float* T_save, const void* dY, float* dX32,
                                   float* dA, float* dB, void* workspace, size_t ws_bytes, void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  if ((v = validate_rank(rank)) != QLORA_OK) return v;
  if (!dX32) return QLORA_ERR_INVALID;
  ProjSplit ps;
  ps.end[0] = w->N;
  return linear_bwd_impl(w, ps, M, rank, alpha, X, A, B, T_save, dY, dX32, dA, dB, workspace, ws_bytes, stream,
                         dX32);
}

size_t qlora_multi_workspace_bytes(const qlora_weight_desc* w, int32_t P, const int64_t* n_split, int64_t M,
                                   int32_t rank) {
  ProjSplit ps;
  if (validate_weight(w) != QLORA_OK || validate_rank(rank) != QLORA_OK || M < 0 ||
      validate_split(w, P, n_split, rank, ps) != QLORA_OK)
    return 0;
  if (M == 0) return 256;
  return multi_workspace(w, ps, M, rank);
}

int32_t qlora_multi_linear_fwd(const qlora_weight_desc* w, int32_t P, const int64_t* n_split, int64_t M,
                               int32_t rank, float alpha, const void* X, const void* A, const void* B, void* Y,
                               float* T_save, void* workspace, size_t ws_bytes, void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  if ((v = validate_rank(rank)) != QLORA_OK) return v;
  ProjSplit ps;
  if ((v = validate_split(w, P, n_split, rank, ps)) != QLORA_OK) return v;
  return linear_fwd_impl(w, ps, M, rank, alpha, X, A, B, Y, T_save, workspace, ws_bytes, stream);
}

int32_t qlora_multi_linear_bwd(const qlora_weight_desc* w, int32_t P, const int64_t* n_split, int64_t M,
                               int32_t rank, float alpha, const void* X, const void* A, const void* B,
                               const float* T_save, const void* dY, void* dX, float* dA, float* dB,
                               void* workspace, size_t ws_bytes, void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  if ((v = validate_rank(rank)) != QLORA_OK) return v;
  ProjSplit ps;
  if ((v = validate_split(w, P, n_split, rank, ps)) != QLORA_OK) return v;
  return linear_bwd_impl(w, ps, M, rank, alpha, X, A, B, T_save, dY, dX, dA, dB, workspace, ws_bytes, stream);
}

// ---------------------------------------------------------------- stacked ---
}  // extern "C"

namespace qlora {

struct StackedPlan {
  AdapterPack ap;
  int Q = 0;
  int seg_end[kMaxAdapters];
  float seg_scale[kMaxAdapters];
  DenseLayout L;
  size_t a_off = 0, b_off = 0, total = 0;
};

static int plan_stacked(const qlora_weight_desc* w, int64_t M, int32_t n, const qlora_adapter* ad, StackedPlan& P) {
  if (n < 1 || n > kMaxAdapters || !ad) return QLORA_ERR_INVALID;
  P.ap.n = n;
  P.Q = 0;
  for (int i = 0; i < n; ++i) {
    if (validate_rank(ad[i].rank) != QLORA_OK || !std::isfinite(ad[i].alpha)) return QLORA_ERR_INVALID;
    P.ap.r[i] = ad[i].rank;
    P.ap.A[i] = static_cast<const __nv_bfloat16*>(ad[i].A);
    P.ap.B[i] = static_cast<const __nv_bfloat16*>(ad[i].B);
    P.Q += ad[i].rank;
    P.seg_end[i] = P.Q;
    P.seg_scale[i] = ad[i].alpha / (float)ad[i].rank;
  }
  if (P.Q > 64) return QLORA_ERR_UNSUPPORTED;
  P.L = dense_layout(M, w->N, w->K, P.Q);
  P.a_off = P.L.total;
  P.b_off = P.a_off + round256((size_t)P.Q * w->K * 2);
  P.total = P.b_off + round256((size_t)w->N * P.Q * 2);
  return QLORA_OK;
}

static int check_adapter_ptrs(const StackedPlan& P) {
  for (int i = 0; i < P.ap.n; ++i) {
    if (!P.ap.A[i] || !P.ap.B[i]) return QLORA_ERR_INVALID;
    if (!aligned16(P.ap.A[i]) || !aligned16(P.ap.B[i])) return QLORA_ERR_ALIGN;
  }
  return QLORA_OK;
}

}  // namespace qlora

extern "C" {

size_t qlora_stacked_workspace_bytes(const qlora_weight_desc* w, int64_t M, int32_t n_adapters,
                                     const qlora_adapter* adapters) {
  StackedPlan P;
  if (validate_weight(w) != QLORA_OK || M < 0 || plan_stacked(w, M, n_adapters, adapters, P) != QLORA_OK) return 0;
  if (M == 0) return 256;
  return P.total;
}

int32_t qlora_stacked_linear_fwd(const qlora_weight_desc* w, int64_t M, int32_t n_adapters,
                                 const qlora_adapter* adapters, const void* X, void* Y, float* T_save,
                                 void* workspace, size_t ws_bytes, void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  StackedPlan P;
  if ((v = plan_stacked(w, M, n_adapters, adapters, P)) != QLORA_OK) return v;
  if (M < 0) return QLORA_ERR_INVALID;
  if (M == 0) return QLORA_OK;
  if (M > (1ll << 31) - 256) return QLORA_ERR_UNSUPPORTED;
  if (!X || !Y || !T_save) return QLORA_ERR_INVALID;
  if ((v = check_adapter_ptrs(P)) != QLORA_OK) return v;
  if (!aligned16(X) || !aligned16(Y) || !aligned16(T_save)) return QLORA_ERR_ALIGN;
  if (!workspace || ws_bytes < P.total) return QLORA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QLORA_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* sT = reinterpret_cast<__nv_bfloat16*>(ws + P.L.act_off);
  __nv_bfloat16* Acat = reinterpret_cast<__nv_bfloat16*>(ws + P.a_off);
  __nv_bfloat16* Bcat = reinterpret_cast<__nv_bfloat16*>(ws + P.b_off);
  // 0) the adapters stacked: A_cat [Q x K], B_cat [N x Q]
  if (launch_pack_adapters(P.ap, w->N, w->K, Acat, Bcat, st) != cudaSuccess) return QLORA_ERR_CUDA;
  // 1) T = X A_cat^T: T_save = T, sT = s_i T_i per adapter
  RowReduce rt = {};
  rt.L = static_cast<const __nv_bfloat16*>(X);
  rt.S = Acat;
  rt.s_qj = 1;
  rt.P = M;
  rt.J = w->K;
  rt.sp = P.L.t;
  rt.scale = 1.f;
  rt.out_f32 = T_save;
  rt.out_scaled = sT;
  rt.nseg = P.ap.n;
  for (int i = 0; i < P.ap.n; ++i) {
    rt.seg_end[i] = P.seg_end[i];
    rt.seg_scale[i] = P.seg_scale[i];
  }
  if (launch_row_reduce_fin(rt, P.Q, st) != cudaSuccess) return QLORA_ERR_CUDA;
  // 2) Y = X deq(W)^T + sT B_cat^T: every adapter in the one adapter chunk
  return cuda_status(run_dense_gemm(w, false, M, P.Q, P.Q, nullptr, X, sT, Bcat, Y, st));
}

int32_t qlora_stacked_linear_bwd(const qlora_weight_desc* w, int64_t M, int32_t n_adapters,
                                 const qlora_adapter* adapters, const void* X, const float* T_save, const void* dY,
                                 void* dX, float* const* dA, float* const* dB, void* workspace, size_t ws_bytes,
                                 void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  StackedPlan P;
  if ((v = plan_stacked(w, M, n_adapters, adapters, P)) != QLORA_OK) return v;
  if (M < 0 || !dA || !dB) return QLORA_ERR_INVALID;
  const int64_t N = w->N, K = w->K;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int i = 0; i < P.ap.n; ++i)
    if ((dA[i] && !aligned16(dA[i])) || (dB[i] && !aligned16(dB[i]))) return QLORA_ERR_ALIGN;
  if (M == 0) {  // no rows: the adapter gradients are zero
    for (int i = 0; i < P.ap.n; ++i) {
      if (dA[i] && cudaMemsetAsync(dA[i], 0, (size_t)P.ap.r[i] * K * 4, st) != cudaSuccess) return QLORA_ERR_CUDA;
      if (dB[i] && cudaMemsetAsync(dB[i], 0, (size_t)N * P.ap.r[i] * 4, st) != cudaSuccess) return QLORA_ERR_CUDA;
    }
    return QLORA_OK;
  }
  if (M > (1ll << 31) - 256) return QLORA_ERR_UNSUPPORTED;
  if (!X || !T_save || !dY) return QLORA_ERR_INVALID;
  if ((v = check_adapter_ptrs(P)) != QLORA_OK) return v;
  if (!aligned16(X) || !aligned16(T_save) || !aligned16(dY) || (dX && !aligned16(dX))) return QLORA_ERR_ALIGN;
  if (!workspace || ws_bytes < P.total) return QLORA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QLORA_ERR_ALIGN;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* sU = reinterpret_cast<__nv_bfloat16*>(ws + P.L.act_off);
  __nv_bfloat16* U2 = reinterpret_cast<__nv_bfloat16*>(ws + P.L.u_off);
  __nv_bfloat16* T2 = reinterpret_cast<__nv_bfloat16*>(ws + P.L.t_off);
  __nv_bfloat16* Acat = reinterpret_cast<__nv_bfloat16*>(ws + P.a_off);
  __nv_bfloat16* Bcat = reinterpret_cast<__nv_bfloat16*>(ws + P.b_off);
  const __nv_bfloat16* Xb = static_cast<const __nv_bfloat16*>(X);
  const __nv_bfloat16* dYb = static_cast<const __nv_bfloat16*>(dY);
  if (launch_pack_adapters(P.ap, N, K, Acat, Bcat, st) != cudaSuccess) return QLORA_ERR_CUDA;
  // 1) U = dY B_cat: sU = s_i U_i per adapter; U and T_save as hi/lo pairs
  RowReduce ru = {};
  ru.L = dYb;
  ru.S = Bcat;
  ru.s_qj = 0;
  ru.P = M;
  ru.J = N;
  ru.sp = P.L.u;
  ru.scale = 1.f;
  ru.out_scaled = sU;
  ru.out_hilo = U2;
  ru.aux_src = T_save;
  ru.aux_hilo = T2;
  ru.nseg = P.ap.n;
  for (int i = 0; i < P.ap.n; ++i) {
    ru.seg_end[i] = P.seg_end[i];
    ru.seg_scale[i] = P.seg_scale[i];
  }
  if (launch_row_reduce_fin(ru, P.Q, st) != cudaSuccess) return QLORA_ERR_CUDA;
  // 2) dB_i = s_i dY^T T_i and dA_i = s_i U_i^T X, each adapter's columns to
  //    its own arrays (none for a frozen adapter)
  ColReduce cb = {};
  cb.L = dYb;
  cb.S2 = T2;
  cb.P = M;
  cb.J = N;
  cb.sp = P.L.c;
  cb.tiles = (int)P.L.db_tiles;
  cb.scale = 1.f;
  cb.transposed = 0;
  cb.nseg = P.ap.n;
  ColReduce ca = cb;
  ca.L = Xb;
  ca.S2 = U2;
  ca.J = K;
  ca.tiles = (int)P.L.da_tiles;
  ca.transposed = 1;
  for (int i = 0; i < P.ap.n; ++i) {
    cb.seg_end[i] = ca.seg_end[i] = P.seg_end[i];
    cb.seg_scale[i] = ca.seg_scale[i] = P.seg_scale[i];
    cb.seg_out[i] = dB[i];
    ca.seg_out[i] = dA[i];
  }
  if (!dX) return cuda_status(launch_col_reduce_fin(cb, &ca, P.Q, st));
  // 3) dX = dY deq(W) + sU A_cat, with step 2 beside it on the side stream
  std::lock_guard<std::mutex> g(g_side_mu);
  SideStream* ss = side_stream_locked();
  if (!ss) {
    if (run_dense_gemm(w, true, M, P.Q, P.Q, nullptr, dY, sU, Acat, dX, st) != cudaSuccess) return QLORA_ERR_CUDA;
    return cuda_status(launch_col_reduce_fin(cb, &ca, P.Q, st));
  }
  cudaError_t e = cudaEventRecord(ss->fork, st);
  if (e == cudaSuccess) e = run_dense_gemm(w, true, M, P.Q, P.Q, nullptr, dY, sU, Acat, dX, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->s, ss->fork, 0);
  if (e == cudaSuccess) e = launch_col_reduce_fin(cb, &ca, P.Q, ss->s);
  if (e == cudaSuccess) e = cudaEventRecord(ss->join, ss->s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ss->join, 0);
  return cuda_status(e);
}

size_t qlora_grouped_workspace_bytes(const qlora_weight_desc* experts, int32_t E, int64_t M_total, int32_t rank) {
  if (validate_grouped(experts, E, M_total, rank) != QLORA_OK) return 0;
  return grouped_layout(experts, E, M_total, rank).total;
}

int32_t grouped_moe_qlora_fwd(const qlora_weight_desc* experts, int32_t E, const int32_t* offsets, int64_t M_total,
                              int32_t rank, float alpha, const void* X, const void* A, const void* B, void* Y,
                              float* T_save, void* workspace, size_t ws_bytes, void* stream) {
  int v = validate_grouped(experts, E, M_total, rank);
  if (v != QLORA_OK) return v;
  if (!std::isfinite(alpha) || !offsets) return QLORA_ERR_INVALID;
  if (M_total == 0) return QLORA_OK;
  if (!X || !A || !B || !Y || !T_save) return QLORA_ERR_INVALID;
  if (!aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(Y) || !aligned16(T_save)) return QLORA_ERR_ALIGN;
  if (experts[0].fmt == QLORA_FMT_BF16 && !experts_stacked(experts, E)) return QLORA_ERR_UNSUPPORTED;
  const GroupedLayout L = grouped_layout(experts, E, M_total, rank);
  if (!workspace || ws_bytes < L.total) return QLORA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QLORA_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const GroupedSched g = grouped_sched(L, ws);
  const float s = alpha / (float)rank;
  __nv_bfloat16* sT = reinterpret_cast<__nv_bfloat16*>(ws + L.off_act);

  // 0) tile lists from the device offsets
  cudaError_t e = launch_grouped_schedule(offsets, E, M_total, kGroupTileRows, L.nblk_f, L.nblk_d, g,
                                          device_error_word(), st);
  if (e != cudaSuccess) return QLORA_ERR_CUDA;
  // 1) T = X A_e^T over each expert's rows: T_save = T, sT = bf16(s T)
  RowReduce rt = {};
  rt.L = static_cast<const __nv_bfloat16*>(X);
  rt.S = static_cast<const __nv_bfloat16*>(A);
  rt.s_qj = 1;
  rt.P = M_total;
  rt.J = L.K;
  rt.sp = plan_split_fin(L.max_rows64, L.K);
  rt.scale = s;
  rt.out_f32 = T_save;
  rt.out_scaled = sT;
  rt.tiles = g.rows64;
  rt.tile_count = g.counts + 2;
  rt.s_stride = (int64_t)rank * L.K;
  rt.max_tiles = L.max_rows64;
  if (launch_row_reduce_fin(rt, rank, st) != cudaSuccess) return QLORA_ERR_CUDA;
  // 2) Y = X deq(W_e)^T + sT B_e^T
  return cuda_status(run_grouped_gemm(experts, L, false, g, X, sT, B, Y, st));
}

int32_t grouped_moe_qlora_bwd(const qlora_weight_desc* experts, int32_t E, const int32_t* offsets, int64_t M_total,
                              int32_t rank, float alpha, const void* X, const void* A, const void* B,
                              const float* T_save, const void* dY, void* dX, float* dA, float* dB, void* workspace,
                              size_t ws_bytes, void* stream) {
  int v = validate_grouped(experts, E, M_total, rank);
  if (v != QLORA_OK) return v;
  if (!std::isfinite(alpha) || !offsets || !dA || !dB) return QLORA_ERR_INVALID;
  const int64_t N = experts[0].N, K = experts[0].K;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M_total == 0) {  // no rows: every expert's adapter gradients are zero
    if (cudaMemsetAsync(dA, 0, (size_t)E * rank * K * 4, st) != cudaSuccess) return QLORA_ERR_CUDA;
    return cuda_status(cudaMemsetAsync(dB, 0, (size_t)E * N * rank * 4, st));
  }
  if (!X || !A || !B || !T_save || !dY) return QLORA_ERR_INVALID;
  if (!aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(T_save) || !aligned16(dY) || !aligned16(dA) ||
      !aligned16(dB) || (dX && !aligned16(dX)))
    return QLORA_ERR_ALIGN;
  if (dX && experts[0].fmt == QLORA_FMT_BF16 && !experts_stacked(experts, E)) return QLORA_ERR_UNSUPPORTED;
  const GroupedLayout L = grouped_layout(experts, E, M_total, rank);
  if (!workspace || ws_bytes < L.total) return QLORA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QLORA_ERR_ALIGN;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const GroupedSched g = grouped_sched(L, ws);
  const float s = alpha / (float)rank;
  __nv_bfloat16* sU = reinterpret_cast<__nv_bfloat16*>(ws + L.off_act);
  __nv_bfloat16* U2 = reinterpret_cast<__nv_bfloat16*>(ws + L.off_u2);
  __nv_bfloat16* T2 = reinterpret_cast<__nv_bfloat16*>(ws + L.off_t2);
  const __nv_bfloat16* dYb = static_cast<const __nv_bfloat16*>(dY);

  // 0) tile lists from the device offsets
  cudaError_t e = launch_grouped_schedule(offsets, E, M_total, kGroupTileRows, L.nblk_f, L.nblk_d, g,
                                          device_error_word(), st);
  if (e != cudaSuccess) return QLORA_ERR_CUDA;
  // 1) U = dY B_e over each expert's rows: sU = bf16(s U) for the dX GEMM,
  //    U and T_save as hi/lo bf16 pairs for the dA / dB reductions
  RowReduce ru = {};
  ru.L = dYb;
  ru.S = static_cast<const __nv_bfloat16*>(B);
  ru.s_qj = 0;
  ru.P = M_total;
  ru.J = N;
  ru.sp = plan_split_fin(L.max_rows64, N);
  ru.scale = s;
  ru.out_scaled = sU;
  ru.out_hilo = U2;
  ru.aux_src = T_save;
  ru.aux_hilo = T2;
  ru.tiles = g.rows64;
  ru.tile_count = g.counts + 2;
  ru.s_stride = N * rank;
  ru.max_tiles = L.max_rows64;
  if (launch_row_reduce_fin(ru, rank, st) != cudaSuccess) return QLORA_ERR_CUDA;

  // 2) dB_e = s dY_e^T T_e and dA_e = s U_e^T X_e (one launch over (expert,
  //    output tile)); an expert without rows gets zeros
  const SplitPlan sp = grouped_col_split(L, N / 64 + K / 64);
  ColReduce cb = {};
  cb.L = dYb;
  cb.S2 = T2;
  cb.P = M_total;
  cb.J = N;
  cb.sp = sp;
  cb.tiles = (int)(N / 64);
  cb.scale = s;
  cb.out = dB;
  cb.transposed = 0;
  cb.ranges = g.ranges;
  cb.groups = E;
  ColReduce ca = cb;
  ca.L = static_cast<const __nv_bfloat16*>(X);
  ca.S2 = U2;
  ca.J = K;
  ca.tiles = (int)(K / 64);
  ca.out = dA;
  ca.transposed = 1;
  if (!dX) return cuda_status(launch_col_reduce_fin(cb, &ca, rank, st));

  // 3) dX = dY deq(W_e) + sU A_e on the caller's stream, step 2 beside it on
  //    the side stream
  std::lock_guard<std::mutex> lk(g_side_mu);
  SideStream* ss = side_stream_locked();
  if (!ss) {
    if (run_grouped_gemm(experts, L, true, g, dY, sU, A, dX, st) != cudaSuccess) return QLORA_ERR_CUDA;
    return cuda_status(launch_col_reduce_fin(cb, &ca, rank, st));
  }
  e = cudaEventRecord(ss->fork, st);
  if (e == cudaSuccess) e = run_grouped_gemm(experts, L, true, g, dY, sU, A, dX, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->s, ss->fork, 0);
  if (e == cudaSuccess) e = launch_col_reduce_fin(cb, &ca, rank, ss->s);
  if (e == cudaSuccess) e = cudaEventRecord(ss->join, ss->s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ss->join, 0);
  return cuda_status(e);
}

}  // extern "C"
