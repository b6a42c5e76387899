/*
 * qlora.h -- C ABI of the GB300 (sm_103a) LoRA linear over a frozen,
 * block-quantised base weight.
 *
 * The operation (forward and the "fast backward formulas" of LoRA; bytechap
 * GGUF blog, "How it works"; the base is frozen, "read, never written", Soup
 * show post, first paragraph):
 *
 *     s  = alpha / r
 *     T  = X A^T                          [M x r]
 *     Y  = X deq(Wq)^T + s T B^T          [M x N]
 *     U  = dY B                           [M x r]
 *     dX = dY deq(Wq) + s U A             [M x K]
 *     dB = s dY^T T                       [N x r]
 *     dA = s U^T X                        [r x K]
 *
 * Base formats (Surogate README, capability table, "LoRA & QLoRA": BF16 and
 * BnB/NF4 bases; bytechap GGUF blog, "How it works": GGUF bases):
 *   BF16  W itself, bf16 [N x K] row-major.
 *   NF4   64 consecutive K-elements per block, two 4-bit codes per byte
 *         (element 2j in the high nibble of byte j), codes [N*K/2] bytes;
 *         per block an fp32 absmax [N*K/64], or (double quantisation) an int8
 *         absmax_q [N*K/64] with one fp32 absmax_scale per dq_group (=256)
 *         consecutive blocks.  Decoded value:
 *             bf16_rn( f32_rn( level[c] * absmax' ) ),
 *             absmax' = absmax or f32_rn( f32(absmax_q) * absmax_scale ).
 *         level[] = the 16 NormalFloat-4 levels (normal quantiles incl. an
 *         exact 0, scaled to [-1, 1]) as fp32.  QLoRA-style double
 *         quantisation (absmax_map set): the absmax byte indexes a 256-entry
 *         fp32 map and an offset is added back:
 *             absmax' = f32_rn( f32_rn( map[(uint8)absmax_q] * absmax_scale )
 *                               + absmax_offset ).
 *   Q8_0  GGUF: blocks of 32 along K, 34 bytes {fp16 d; int8 q[32]};
 *         value = bf16_rn( q * f32(d) ).
 *   Q4_0  GGUF: blocks of 32 along K, 18 bytes {fp16 d; uint8 qs[16]};
 *         element i < 16 = low nibble of qs[i], element i+16 = high nibble;
 *         value = bf16_rn( (nib - 8) * f32(d) ).
 *   Q4_K  GGUF K-quant (Surogate README, "Native GGUF" row; quickstart
 *         "--type q4_k_m"): super-blocks of 256 along K (K % 256 == 0), 144
 *         bytes {fp16 d; fp16 dmin; 12 bytes: eight 6-bit sub-block scales
 *         sc[j] and mins m[j]; 128 code bytes}; sub-block j = 32 elements.
 *         Sub-blocks 0..3: sc = byte j & 63, m = byte j+4 & 63; 4..7:
 *         sc = (byte j+4 & 15) | (byte j-4 >> 6) << 4,
 *         m = (byte j+4 >> 4) | (byte j >> 6) << 4.  Code bytes 32c..32c+31
 *         hold sub-block 2c in their low nibbles and 2c+1 in their high.
 *         value = bf16_rn( f32_rn( f32(d) sc q - f32(dmin) m ) ).
 *   FP8_E4M3  (Surogate README, "LoRA & QLoRA" and "Native precision
 *         recipes" rows; heatdrop.ai summary: E4M3 recipe) one E4M3 code
 *         per element [N*K] (OCP 8-bit float: bias 7, no infinities,
 *         S.1111.111 = NaN) and one fp32 tensor_scale;
 *         value = bf16_rn( f32_rn( e4m3(c) * tensor_scale ) ).
 *   NVFP4 E2M1 codes, two per byte [N*K/2] (element 2j in the LOW nibble of
 *         byte j), one E4M3 block_scale per 16 consecutive K-elements
 *         [N*K/16] and one fp32 tensor_scale;
 *         value = bf16_rn( f32_rn( e2m1(c) * f32_rn( e4m3(s) * tensor_scale ) ) ).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers unless stated otherwise, owned
 *     and allocated by the caller, 16-byte aligned, row-major, densely packed.
 *   - X, A, B, Y, dY, dX are bf16 (passed as void*); T_save, dA, dB are fp32;
 *     dA and dB are overwritten (not accumulated).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     only enqueues work on it and returns; nothing synchronises.
 *     qlora_linear_bwd also runs part of its work on a per-device stream of
 *     the library's own, forked from `stream` and joined back into it with
 *     events inside the call, so all of a call's work is still ordered on
 *     `stream`.
 *   - Arguments are validated before anything is launched; a rejected call
 *     launches nothing and returns a negative qlora_status.
 *   - A kernel whose internal wait runs out (it never should) records
 *     QLORA_ERR_TIMEOUT in a device error word, which qlora_device_error()
 *     reads after the caller has synchronised.
 *   - Limits: N % 64 == 0, K % 64 == 0, 8 <= rank <= 64 with rank % 8 == 0,
 *     M >= 0 (M == 0 is a no-op that returns QLORA_OK).
 */
#ifndef QLORA_H_
#define QLORA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QLORA_FMT_BF16 = 0,
  QLORA_FMT_NF4 = 1,
  QLORA_FMT_Q8_0 = 2,
  QLORA_FMT_Q4_0 = 3,
  QLORA_FMT_Q4_K = 4,     /* GGUF K-quant, super-blocks of 256 */
  QLORA_FMT_FP8_E4M3 = 5, /* OCP E4M3 codes with one fp32 tensor scale */
  QLORA_FMT_NVFP4 = 6     /* E2M1 codes, E4M3 scale per 16, fp32 tensor scale */
} qlora_format;

typedef enum {
  QLORA_OK = 0,
  QLORA_ERR_INVALID = -1,     /* bad shape, rank, null pointer, format */
  QLORA_ERR_UNSUPPORTED = -2, /* valid request this library does not cover */
  QLORA_ERR_ALIGN = -3,       /* pointer not 16-byte aligned */
  QLORA_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed */
  QLORA_ERR_TIMEOUT = -5,     /* a bounded device wait gave up */
  QLORA_ERR_WORKSPACE = -6,   /* workspace missing or too small */
  QLORA_ERR_STATE = -7        /* streaming pool used out of order */
} qlora_status;

/* Frozen base weight W [N x K] in one of the formats above.  Every pointer
 * is a read-only device pointer; unused ones must be NULL. */
typedef struct {
  int32_t fmt;                /* qlora_format */
  int32_t dq_group;           /* NF4 double quantisation group (256), else 0 */
  int64_t N;                  /* output features (rows of W) */
  int64_t K;                  /* input features (columns of W) */
  const void* data;           /* BF16: bf16[N*K]; NF4: uint8[N*K/2];
                                 Q8_0: 34-byte blocks [N*K/32];
                                 Q4_0: 18-byte blocks [N*K/32];
                                 Q4_K: 144-byte super-blocks [N*K/256];
                                 FP8_E4M3: uint8[N*K]; NVFP4: uint8[N*K/2] */
  const float* absmax;        /* NF4 without double quantisation: fp32[N*K/64] */
  const int8_t* absmax_q;     /* NF4 with double quantisation: int8[N*K/64] */
  const float* absmax_scale;  /* NF4 with double quantisation:
                                 fp32[ceil(N*K/64 / dq_group)] */
  const float* absmax_map;    /* NF4 with double quantisation through an 8-bit
                                 map: fp32[256]; NULL = plain int8 codes */
  const float* tensor_scale;  /* FP8_E4M3, NVFP4: fp32[1] */
  const uint8_t* block_scale; /* NVFP4: E4M3 codes [N*K/16], 16-byte aligned */
  float absmax_offset;        /* NF4 with absmax_map: added to every absmax */
  int32_t reserved;           /* must be 0 */
} qlora_weight_desc;

/* Human-readable name of a status code (static string, never NULL). */
const char* qlora_status_string(int32_t status);

/* Library ABI version (major * 100 + minor). */
int32_t qlora_version(void);

/* Bytes of device workspace that qlora_linear_fwd and qlora_linear_bwd need
 * for this weight shape, M and rank (the larger of the two).  0 on invalid
 * arguments.  The workspace holds the scaled adapter activation s*T or s*U
 * (bf16) and, for the backward pass, U = dY B and T_save as bf16 hi / lo
 * pairs.  Its contents need no initialisation and are not kept between
 * calls; calls that may overlap on the GPU need separate workspaces. */
size_t qlora_workspace_bytes(const qlora_weight_desc* w, int64_t M, int32_t rank);

/* Bytes of workspace qlora_linear_fwd alone needs (the scaled activation
 * s*T, bf16 [M x rank], 256-byte rounded); at most qlora_workspace_bytes.
 * 0 on invalid arguments. */
size_t qlora_forward_workspace_bytes(const qlora_weight_desc* w, int64_t M, int32_t rank);

/* Decode the whole base weight to bf16: W_bf16[N*K] (device, caller-owned)
 * receives deq(Wq) bit-exactly as defined above.  For QLORA_FMT_BF16 it is a
 * copy. */
int32_t dequant_blocks(const qlora_weight_desc* w, void* W_bf16, void* stream);

/* Forward: Y[M x N] = X deq(Wq)^T + s (X A^T) B^T, and T_save[M x rank] =
 * X A^T (fp32, kept for the backward pass).
 *   X [M x K], A [rank x K], B [N x rank], Y [M x N] bf16; T_save [M x rank]
 *   fp32.  The adapter term enters Y through bf16(s T).
 *   workspace: device, at least qlora_workspace_bytes(w, M, rank) bytes.
 * The base is decoded inside the GEMM's operand producer; the decoded weight
 * never goes to global memory. */
int32_t qlora_linear_fwd(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha,
                         const void* X, const void* A, const void* B,
                         void* Y, float* T_save,
                         void* workspace, size_t ws_bytes, void* stream);

/* Backward: dX[M x K] = dY deq(Wq) + s (dY B) A;  dA[rank x K] (fp32) =
 * s (dY B)^T X;  dB[N x rank] (fp32) = s dY^T T_save.  dX may be NULL (then
 * only dA and dB are produced).  T_save is the forward's fp32 output.  U = dY B
 * and T_save enter dA and dB as bf16 hi / lo pairs (~16 significant bits);
 * the adapter term of dX enters through bf16(s U).  The base is never
 * written. */
int32_t qlora_linear_bwd(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha,
                         const void* X, const void* A, const void* B,
                         const float* T_save, const void* dY,
                         void* dX, float* dA, float* dB,
                         void* workspace, size_t ws_bytes, void* stream);

/* Debug forms of the two calls above: identical, except that the GEMM
 * output is written as its fp32 accumulator values (Y32 [M x N], resp.
 * dX32 [M x K], fp32, device, 16-byte aligned) instead of bf16, so that a
 * test can see the error of the computation without the bf16 output
 * rounding.  dX32 may not be NULL.  Slower (no staged output stores); for
 * tests only. */
int32_t qlora_debug_linear_fwd_f32(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha,
                                   const void* X, const void* A, const void* B,
                                   float* Y32, float* T_save,
                                   void* workspace, size_t ws_bytes, void* stream);
int32_t qlora_debug_linear_bwd_f32(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha,
                                   const void* X, const void* A, const void* B,
                                   const float* T_save, const void* dY,
                                   float* dX32, float* dA, float* dB,
                                   void* workspace, size_t ws_bytes, void* stream);

/* ---- gate / up projections with the SwiGLU activation ------------------------
 * The MLP input side of the Llama / Qwen3 layers: two LoRA linears over the
 * same X (gate and up) fused as one call (see the fused projections below),
 * with the activation H = silu(G) * U, silu(g) = g sigmoid(g), computed in
 * the forward GEMM's epilogue from the fp32 accumulators (launches of more
 * than 128 rows; an elementwise pass over G | U otherwise).
 *   w: the two bases stacked by rows, [gate rows; up rows], N = 2 I with
 *      I % 256 == 0; A: bf16 [2][rank][K] (gate, up); B: bf16 [2I][rank]
 *      (gate rows, then up rows); 2 rank <= 64.
 *   forward outputs: H bf16 [M][I]; GU bf16 [M][2I] = G | U (the
 *      pre-activations, kept for the backward); T_save fp32 [M][2 rank].
 *   backward: from dH bf16 [M][I] and GU, dG = dH U sigmoid(G) (1 + G (1 -
 *      sigmoid(G))) and dU = dH silu(G) (fp32, stored bf16 in the
 *      workspace), then the fused two-projection backward: dX bf16 [M][K]
 *      (gate's and up's input gradients summed; may be NULL), dA fp32
 *      [2][rank][K], dB fp32 [2I][rank].
 *   workspace: qlora_swiglu_workspace_bytes (covers both calls). */
size_t qlora_swiglu_workspace_bytes(const qlora_weight_desc* w, int64_t M, int32_t rank);
int32_t qlora_swiglu_fwd(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha,
                         const void* X, const void* A, const void* B,
                         void* H, void* GU, float* T_save,
                         void* workspace, size_t ws_bytes, void* stream);
int32_t qlora_swiglu_bwd(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha,
                         const void* X, const void* A, const void* B,
                         const float* T_save, const void* GU, const void* dH,
                         void* dX, float* dA, float* dB,
                         void* workspace, size_t ws_bytes, void* stream);

/* ---- fused projections that share their input ------------------------------
 * The P LoRA linears that read the same X in a decoder layer (q, k, v of the
 * attention block; gate and up of the MLP) as one call each way: one pass of
 * X for every projection's T, one GEMM over all their base rows, one pass of
 * dY for every U, one dX GEMM that reduces over all their output columns, so
 * dX is the sum of the projections' input gradients (what the layer feeding
 * X receives).  Surogate README, design bullet "Kernels that do more per
 * launch".
 *   w: the projections' base weights stacked by rows, one [N x K] weight in
 *      any format, N = sum n_split[p] (projection p's rows after those of
 *      projections < p).
 *   n_split: HOST int64[P], 1 <= P <= 8, each a multiple of 256 when P > 1;
 *      P rank <= 64.
 *   A: bf16 [P][rank][K] (projection p's adapter A_p);  B: bf16 [N][rank]
 *      (projection p's B_p in its rows);  s = alpha / rank for all.
 *   forward:  Y [M][N] bf16 (projection p in its column block) = X deq(W)^T
 *             + s T_p B_p^T per block;  T_save [M][P rank] fp32 (T_p in
 *             columns p rank ..).
 *   backward: dY [M][N] (projection p in its column block);
 *             dX [M][K] = sum_p (dY_p deq(W_p) + s U_p A_p) (may be NULL);
 *             dA fp32 [P][rank][K], dB fp32 [N][rank] per projection.
 *   workspace: qlora_multi_workspace_bytes() bytes.
 * With P = 1 these are qlora_linear_fwd / _bwd. */
size_t qlora_multi_workspace_bytes(const qlora_weight_desc* w, int32_t P, const int64_t* n_split, int64_t M,
                                   int32_t rank);
int32_t qlora_multi_linear_fwd(const qlora_weight_desc* w, int32_t P, const int64_t* n_split, int64_t M,
                               int32_t rank, float alpha, const void* X, const void* A, const void* B, void* Y,
                               float* T_save, void* workspace, size_t ws_bytes, void* stream);
int32_t qlora_multi_linear_bwd(const qlora_weight_desc* w, int32_t P, const int64_t* n_split, int64_t M,
                               int32_t rank, float alpha, const void* X, const void* A, const void* B,
                               const float* T_save, const void* dY, void* dX, float* dA, float* dB,
                               void* workspace, size_t ws_bytes, void* stream);

/* ---- stacked adapters --------------------------------------------------------
 * Several LoRA pairs on the same frozen base, applied together without
 * merging any of them into the base, so an adapter can be trained on top of
 * others (heatdrop.ai summary, "Key highlights": stacked LoRA; Surogate
 * README, "LoRA & QLoRA" row).  Adapter i: rank r_i, scale s_i = alpha_i / r_i,
 * A_i bf16 [r_i x K], B_i bf16 [N x r_i] (device).
 *   forward:  Y = X deq(W)^T + sum_i s_i (X A_i^T) B_i^T;
 *             T_save [M x sum r_i] fp32, T_i = X A_i^T in columns off_i ..
 *   backward: dX = dY deq(W) + sum_i s_i (dY B_i) A_i (dX may be NULL);
 *             dA_i = s_i (dY B_i)^T X, dB_i = s_i dY^T T_i into dA[i] fp32
 *             [r_i x K], dB[i] fp32 [N x r_i]; dA, dB are HOST arrays of
 *             n_adapters device pointers, and a NULL entry leaves that
 *             adapter without gradient (a frozen adapter under a trained one).
 *   Limits: 1 <= n_adapters <= 4, each r_i a multiple of 8 in [8, 64],
 *   sum r_i <= 64.  The adapters are packed into the workspace
 *   (qlora_stacked_workspace_bytes()) and run as one adapter chunk of the
 *   fused GEMM. */
typedef struct {
  int32_t rank;   /* r_i */
  float alpha;    /* s_i = alpha / r_i */
  const void* A;  /* bf16 [r_i x K], device */
  const void* B;  /* bf16 [N x r_i], device */
} qlora_adapter;

size_t qlora_stacked_workspace_bytes(const qlora_weight_desc* w, int64_t M, int32_t n_adapters,
                                     const qlora_adapter* adapters);
int32_t qlora_stacked_linear_fwd(const qlora_weight_desc* w, int64_t M, int32_t n_adapters,
                                 const qlora_adapter* adapters, const void* X, void* Y, float* T_save,
                                 void* workspace, size_t ws_bytes, void* stream);
int32_t qlora_stacked_linear_bwd(const qlora_weight_desc* w, int64_t M, int32_t n_adapters,
                                 const qlora_adapter* adapters, const void* X, const float* T_save,
                                 const void* dY, void* dX, float* const* dA, float* const* dB,
                                 void* workspace, size_t ws_bytes, void* stream);

/* Forward pass that allocates nothing, for callers that cannot allocate
 * device memory (e.g. a plug-in that may only use the buffers its host
 * application passes in, or a loop that must not call cudaMalloc because it
 * can synchronise the device).  The paper has no counterpart to this call.
 * Same arguments and results as qlora_linear_fwd, minus the workspace: the
 * workspace is a fixed 16 MiB array kept in device memory by the library
 * (qlora_noalloc_scratch_bytes()), reserved on every GPU that loads the
 * library until the process exits.  Returns QLORA_ERR_WORKSPACE, launching
 * nothing, when qlora_forward_workspace_bytes(w, M, rank) exceeds that size
 * (2 M rank bytes: M rank <= 8 Mi, e.g. 524,288 rows at rank 16).  The
 * first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls on a device share the array: calls whose GPU work
 * overlaps (e.g. on two unordered streams) race on it and may give wrong
 * results.  No part of the array needs to start at zero. */
int32_t qlora_linear_fwd_noalloc(const qlora_weight_desc* w, int64_t M, int32_t rank, float alpha,
                                 const void* X, const void* A, const void* B,
                                 void* Y, float* T_save, void* stream);
size_t qlora_noalloc_scratch_bytes(void);

/* ---- grouped (mixture-of-experts) variant -------------------------------
 * The same layer for E experts (bytechap GGUF blog: fast LoRA backward for
 * linear and MoE layers), each expert applied to its own rows.  Rows of X /
 * dY / Y / dX / T_save are sorted by expert: expert e owns rows offsets[e] ..
 * offsets[e+1]-1.
 *
 * offsets: DEVICE int32[E+1] (as a router leaves them; never read on the
 *   host, so the call neither copies nor synchronises).  They must satisfy
 *   offsets[0] == 0, offsets[e] <= offsets[e+1], offsets[E] == M_total;
 *   empty experts are allowed.  This is checked on the device: offsets that
 *   break it make the call write nothing (Y, dX, dA, dB undefined) and record
 *   QLORA_ERR_INVALID in the device error word (qlora_last_device_error).
 * M_total: HOST, the number of rows (0 <= M_total <= 2^30); it sizes the
 *   workspace and the launch grids.
 * experts: HOST array of E <= 256 weight descriptors, all with the same fmt,
 *   N and K.  bf16 bases must lie back to back in one array [E][N][K]
 *   (experts[e].data == experts[0].data + e N K), else
 *   QLORA_ERR_UNSUPPORTED; quantised bases may lie anywhere.
 * A: bf16 [E][rank][K], B: bf16 [E][N][rank], T_save: fp32 [M_total][rank],
 * dA: fp32 [E][rank][K], dB: fp32 [E][N][rank]; an expert with no rows gets
 * dA = dB = 0.  dX may be NULL.  Device pointers, 16-byte aligned.
 * Workspace: qlora_grouped_workspace_bytes(experts, E, M_total, rank) (0 for
 * invalid arguments); it holds the device-built tile lists, so the same
 * workspace must not be in use by another call at the same time.  The
 * backward call runs its dA / dB reduction on a second stream of the library
 * beside its dX GEMM, joined back into `stream` before it returns. */
size_t qlora_grouped_workspace_bytes(const qlora_weight_desc* experts, int32_t E,
                                     int64_t M_total, int32_t rank);

int32_t grouped_moe_qlora_fwd(const qlora_weight_desc* experts, int32_t E,
                              const int32_t* offsets, int64_t M_total,
                              int32_t rank, float alpha,
                              const void* X, const void* A, const void* B,
                              void* Y, float* T_save,
                              void* workspace, size_t ws_bytes, void* stream);

int32_t grouped_moe_qlora_bwd(const qlora_weight_desc* experts, int32_t E,
                              const int32_t* offsets, int64_t M_total,
                              int32_t rank, float alpha,
                              const void* X, const void* A, const void* B,
                              const float* T_save, const void* dY,
                              void* dX, float* dA, float* dB,
                              void* workspace, size_t ws_bytes, void* stream);

/* ---- layer streaming ------------------------------------------------------
 * A frozen base kept in pinned host memory is streamed into a fixed pool of
 * device buffers one layer ahead of use on a dedicated copy stream (Soup show
 * post, first paragraph: "a small pool of pre-allocated VRAM buffers, one
 * decoder layer at a time, prefetched one ahead on a dedicated CUDA stream").
 *
 * qlora_stream_create: allocates `slots` device buffers of `slot_bytes` each
 *   (the only device memory this library allocates at run time; the
 *   no-alloc forward's scratch is a fixed array in the library's image), a
 *   copy stream and events.
 * qlora_stream_prefetch: announce that `layer` is needed next.  If it is
 *   still resident nothing is copied; otherwise enqueue the host->device copy
 *   of `bytes` bytes at `host_src` (pinned host memory, valid until the copy
 *   ran) into the least recently used slot that is neither acquired nor
 *   holding an announced, not yet acquired layer, tagged with `layer`.  The
 *   copy waits for the work enqueued before every release of that slot since
 *   it was last filled, on whichever streams those releases named (a layer
 *   acquired on several unordered streams is overwritten only after all of
 *   them).  QLORA_ERR_STATE if no slot is free (prefetching too far ahead),
 *   QLORA_ERR_INVALID if `bytes` exceeds the slot size.
 * qlora_stream_acquire: make `compute_stream` wait for the copy of `layer`
 *   and return the slot's device address in *dev_ptr.  QLORA_ERR_STATE if no
 *   slot holds `layer` (never prefetched, or already overwritten).
 * qlora_stream_release: record on `compute_stream` that work reading `layer`
 *   has been enqueued (one release per acquire); the slot may be refilled
 *   after that work and the work of the slot's other releases.
 * qlora_stream_destroy: synchronise and free everything. */
int32_t qlora_stream_create(int32_t slots, size_t slot_bytes, void** handle);
int32_t qlora_stream_prefetch(void* handle, int32_t layer, const void* host_src, size_t bytes);
int32_t qlora_stream_acquire(void* handle, int32_t layer, void* compute_stream, void** dev_ptr);
int32_t qlora_stream_release(void* handle, int32_t layer, void* compute_stream);
int32_t qlora_stream_destroy(void* handle);

/* Read the device error word written by bounded waits (QLORA_OK if none).
 * Call after synchronising the streams the library used.  clear != 0 resets
 * it.  This call synchronises the device. */
int32_t qlora_device_error(int32_t clear);

/* Stream-ordered read of the same word (the call list's
 * qlora_last_device_error): enqueues a device->host copy of the word on
 * `stream`, waits for that stream only (no device-wide synchronisation) and
 * returns the value, i.e. any error recorded by work enqueued on `stream`
 * before this call (including the backward call's side-stream work, which is
 * joined back into the caller's stream).  The word is shared by all streams
 * of the device, so an error recorded by another stream's finished work is
 * reported too.  clear != 0 resets the word (stream-ordered) when it was
 * set. */
int32_t qlora_last_device_error(void* stream, int32_t clear);

/* Diagnostic of the bounded-wait error path: launches on `stream` one warp
 * that waits, for at most limit_ns nanoseconds (1 .. 1e9), on an mbarrier
 * phase that nothing completes.  The wait runs out, records
 * QLORA_ERR_TIMEOUT in the device error word and the kernel returns; the
 * context stays usable.  Returns QLORA_OK once launched, QLORA_ERR_INVALID for
 * a limit outside the range.  No counterpart on the pages: it exists so a
 * test can check that a device wait that runs out ends as an error status. */
int32_t qlora_selftest_bounded_wait(int64_t limit_ns, void* stream);

/* Number of this library's kernels launched since load (host-side count). */
int64_t qlora_launch_count(void);

/* Instrumentation of the fused tensor-core GEMM (the dominant kernel).
 * qlora_profile_gemm(1) clears the record and starts recording a CUDA event
 * pair around every fused-GEMM launch, on the stream it is launched on;
 * qlora_profile_gemm(0) stops recording.  qlora_profile_gemm_read()
 * synchronises on the recorded events and returns the summed device time
 * (ms), the number of launches and their summed algorithmic flops
 * (2 M n_out (k_red + rank) per launch).  Host pointers; any may be NULL. */
int32_t qlora_profile_gemm(int32_t enable);
int32_t qlora_profile_gemm_read(double* total_ms, int64_t* launches, double* flops);

#ifdef __cplusplus
}
#endif

#endif /* QLORA_H_ */
