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

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

static int validate_weight(const qlora_weight_desc* w) {
  if (!w) return QLORA_ERR_INVALID;
  if (w->N <= 0 || w->K <= 0 || (w->N % 64) || (w->K % 64)) return QLORA_ERR_INVALID;
  if (w->N > (1ll << 30) || w->K > (1ll << 30)) return QLORA_ERR_UNSUPPORTED;
  if (!w->data) return QLORA_ERR_INVALID;
  if (!aligned16(w->data)) return QLORA_ERR_ALIGN;
  switch (w->fmt) {
    case QLORA_FMT_BF16:
    case QLORA_FMT_Q8_0:
    case QLORA_FMT_Q4_0:
      break;
    case QLORA_FMT_NF4:
      if (w->absmax) {
        if (!aligned16(w->absmax)) return QLORA_ERR_ALIGN;
      } else {
        if (!w->absmax_q || !w->absmax_scale || w->dq_group <= 0) return QLORA_ERR_INVALID;
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
  v.dq_group = w->dq_group > 0 ? w->dq_group : 1;
  v.fmt = w->fmt;
  return v;
}

// ------------------------------------------------------- workspace layout ---
struct DenseLayout {
  size_t act_off, act_bytes;  // sT or sU, bf16 [M x r]
  size_t u_off, u_bytes;      // U, fp32 [M x r] (backward)
  size_t part_off, part_bytes;
  SplitPlan t, u, db, da;
  size_t total;
};

static DenseLayout dense_layout(int64_t M, int64_t N, int64_t K, int r) {
  DenseLayout L;
  const int64_t mt = (M + 63) / 64;
  L.t = plan_split(mt, K);
  L.u = plan_split(mt, N);
  L.db = plan_split(N / 64, M);
  L.da = plan_split(K / 64, M);
  L.act_off = 0;
  L.act_bytes = round256((size_t)M * r * 2);
  L.u_off = L.act_off + L.act_bytes;
  L.u_bytes = round256((size_t)M * r * 4);
  size_t p = (size_t)L.t.splits * M * r;
  p = std::max(p, (size_t)L.u.splits * M * r);
  p = std::max(p, (size_t)L.db.splits * N * r * 2);  // hi/lo halves
  p = std::max(p, (size_t)L.da.splits * K * r * 2);
  L.part_off = L.u_off + L.u_bytes;
  L.part_bytes = round256(p * 4);
  L.total = L.part_off + L.part_bytes;
  return L;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA; }

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

// Launch the fused GEMM, bracketed by events when instrumentation is on.
static cudaError_t gemm_dispatch(int fmt, bool dx, bool pair, const GemmMaps& maps, const GemmArgs& a,
                                cudaStream_t st) {
  return pair ? launch_qgemm_pair(fmt, dx, maps, a, st) : launch_qgemm(fmt, dx, false, maps, a, sm_count(), st);
}

static cudaError_t gemm_launch(int fmt, bool dx, bool pair, const GemmMaps& maps, const GemmArgs& a,
                               cudaStream_t st) {
  std::unique_lock<std::mutex> g(g_prof_mu);
  if (!g_prof_on) {
    g.unlock();
    return gemm_dispatch(fmt, dx, pair, maps, a, st);
  }
  GemmRec r;
  r.a = prof_event();
  r.b = prof_event();
  r.flops = 2.0 * (double)a.M * (double)a.n_out * (double)(a.k_red + a.rank);
  cudaEventRecord(r.a, st);
  cudaError_t e = gemm_dispatch(fmt, dx, pair, maps, a, st);
  cudaEventRecord(r.b, st);
  g_prof_recs.push_back(r);
  return e;
}

// Dense fused GEMM: forward (dx = false) out = A_op W^T + la lb^T with
// A_op = X [M x K], la = sT, lb = B [N x r]; dX (dx = true) out = A_op W +
// la lb with A_op = dY [M x N], la = sU, lb = A [r x K].
static cudaError_t run_dense_gemm(const qlora_weight_desc* w, bool dx, int64_t M, int rank, const void* a_op,
                                  const void* la, const void* lb, void* out, cudaStream_t st) {
  const int64_t N = w->N, K = w->K;
  const bool pair = M > kBM;  // 256-row tiles on a CTA pair; short problems use one CTA per tile
  const uint32_t brows = pair ? 128 : 256;
  GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  bool ok;
  if (!dx) {
    ok = map2d(&maps.a, a_op, K, M, 64, 128) && map2d(&maps.la, la, rank, M, 64, 128) &&
         map2d(&maps.lb, lb, rank, N, 64, brows);
    if (w->fmt == QLORA_FMT_BF16) ok = ok && map2d(&maps.w, w->data, K, N, 64, brows);
  } else {
    ok = map2d(&maps.a, a_op, N, M, 64, 128) && map2d(&maps.la, la, rank, M, 64, 128) &&
         map2d(&maps.lb, lb, K, rank, 64, 64);
    if (w->fmt == QLORA_FMT_BF16) ok = ok && map2d(&maps.w, w->data, K, N, 64, 64);
  }
  if (!ok) return cudaErrorInvalidValue;
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.M = (int)M;
  a.n_out = (int)(dx ? K : N);
  a.k_red = (int)(dx ? N : K);
  a.rank = rank;
  a.num_n_blk = (a.n_out + kBN - 1) / kBN;
  const int64_t row_tile = pair ? 256 : kBM;
  a.num_tiles = (int)(((M + row_tile - 1) / row_tile) * a.num_n_blk);
  a.w_lines_per_row = K / 64;
  a.w_rows = N;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.wv = view_of(w);
  a.err = device_error_word();
  return gemm_launch(w->fmt, dx, pair, maps, a, st);
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

int32_t qlora_version(void) { return 100; }

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

size_t qlora_workspace_bytes(const qlora_weight_desc* w, int64_t M, int32_t rank) {
  if (validate_weight(w) != QLORA_OK || validate_rank(rank) != QLORA_OK || M < 0) return 0;
  if (M == 0) return 256;
  return dense_layout(M, w->N, w->K, rank).total;
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

int32_t qlora_linear_fwd(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha, const void* X,
                         const void* A, const void* B, void* Y, float* T_save, void* workspace, size_t ws_bytes,
                         void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  if ((v = validate_rank(rank)) != QLORA_OK) return v;
  if (M < 0 || !std::isfinite(alpha)) return QLORA_ERR_INVALID;
  if (M == 0) return QLORA_OK;
  if (M > (1ll << 31) - 256) return QLORA_ERR_UNSUPPORTED;
  if (!X || !A || !B || !Y || !T_save) return QLORA_ERR_INVALID;
  if (!aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(Y) || !aligned16(T_save))
    return QLORA_ERR_ALIGN;
  const int64_t N = w->N, K = w->K;
  const DenseLayout L = dense_layout(M, N, K, rank);
  if (!workspace || ws_bytes < L.total) return QLORA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QLORA_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* sT = reinterpret_cast<__nv_bfloat16*>(ws + L.act_off);
  float* part = reinterpret_cast<float*>(ws + L.part_off);
  const float s = alpha / (float)rank;

  // 1) T = X A^T (split over K), T_save = bf16(T), sT = bf16(s T)
  cudaError_t e = launch_row_reduce(static_cast<const __nv_bfloat16*>(X), M, K,
                                    static_cast<const __nv_bfloat16*>(A), rank, true, part, L.t, st);
  if (e != cudaSuccess) return QLORA_ERR_CUDA;
  e = launch_fin_rows(part, L.t.splits, M, rank, s, static_cast<float*>(T_save), sT, st);
  if (e != cudaSuccess) return QLORA_ERR_CUDA;

  // 2) Y = X deq(W)^T + sT B^T
  return cuda_status(run_dense_gemm(w, false, M, rank, X, sT, B, Y, st));
}

int32_t qlora_linear_bwd(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha, const void* X,
                         const void* A, const void* B, const float* T_save, const void* dY, void* dX, float* dA,
                         float* dB, void* workspace, size_t ws_bytes, void* stream) {
  int v = validate_weight(w);
  if (v != QLORA_OK) return v;
  if ((v = validate_rank(rank)) != QLORA_OK) return v;
  if (M < 0 || !std::isfinite(alpha)) return QLORA_ERR_INVALID;
  if (!dA || !dB) return QLORA_ERR_INVALID;
  const int64_t N = w->N, K = w->K;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M == 0) {  // no rows: the adapter gradients are zero
    if (cudaMemsetAsync(dA, 0, (size_t)rank * K * 4, st) != cudaSuccess) return QLORA_ERR_CUDA;
    return cuda_status(cudaMemsetAsync(dB, 0, (size_t)N * rank * 4, st));
  }
  if (M > (1ll << 31) - 256) return QLORA_ERR_UNSUPPORTED;
  if (!X || !A || !B || !T_save || !dY) return QLORA_ERR_INVALID;
  if (!aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(T_save) || !aligned16(dY) ||
      !aligned16(dA) || !aligned16(dB) || (dX && !aligned16(dX)))
    return QLORA_ERR_ALIGN;
  const DenseLayout L = dense_layout(M, N, K, rank);
  if (!workspace || ws_bytes < L.total) return QLORA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QLORA_ERR_ALIGN;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* sU = reinterpret_cast<__nv_bfloat16*>(ws + L.act_off);
  float* U = reinterpret_cast<float*>(ws + L.u_off);
  float* part = reinterpret_cast<float*>(ws + L.part_off);
  const float s = alpha / (float)rank;
  const __nv_bfloat16* Xb = static_cast<const __nv_bfloat16*>(X);
  const __nv_bfloat16* dYb = static_cast<const __nv_bfloat16*>(dY);

  // 1) U = dY B (split over N): U fp32, sU = bf16(s U)
  cudaError_t e = launch_row_reduce(dYb, M, N, static_cast<const __nv_bfloat16*>(B), rank, false, part, L.u, st);
  if (e == cudaSuccess) e = launch_fin_rows(part, L.u.splits, M, rank, s, U, sU, st);
  // 2) dB = s dY^T T (split over M)
  if (e == cudaSuccess)
    e = launch_col_reduce(dYb, M, N, static_cast<const float*>(T_save), rank, part, L.db, st);
  if (e == cudaSuccess) e = launch_fin_cols(part, L.db.splits, N, rank, s, dB, false, st);
  if (e != cudaSuccess) return QLORA_ERR_CUDA;

  // 3) dX = dY deq(W) + sU A
  if (dX) {
    e = run_dense_gemm(w, true, M, rank, dY, sU, A, dX, st);
    if (e != cudaSuccess) return QLORA_ERR_CUDA;
  }

  // 4) dA = s U^T X (split over M), computed as dA^T [K x r] then transposed
  e = launch_col_reduce(Xb, M, K, U, rank, part, L.da, st);
  if (e == cudaSuccess) e = launch_fin_cols(part, L.da.splits, K, rank, s, dA, true, st);
  return cuda_status(e);
}

size_t qlora_grouped_workspace_bytes(const qlora_weight_desc* experts, int32_t E, const int32_t* offsets,
                                     int32_t rank) {
  (void)experts;
  (void)E;
  (void)offsets;
  (void)rank;
  return 0;
}

int32_t grouped_moe_qlora_fwd(const qlora_weight_desc*, int32_t, const int32_t*, int32_t, float, const void*,
                              const void*, const void*, void*, float*, void*, size_t, void*) {
  return QLORA_ERR_UNSUPPORTED;
}

int32_t grouped_moe_qlora_bwd(const qlora_weight_desc*, int32_t, const int32_t*, int32_t, float, const void*,
                              const void*, const void*, const float*, const void*, void*, float*, float*, void*,
                              size_t, void*) {
  return QLORA_ERR_UNSUPPORTED;
}

}  // extern "C"
