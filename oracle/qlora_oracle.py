"""Plain fp64 CPU oracle for the LoRA linear over a frozen block-quantised base.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg may import this module.  It shares
no code with the CUDA library and imports nothing from it.

What it computes, and where it comes from:

* The layer (forward and "fast backward" formulas of LoRA, bytechap GGUF blog,
  "How it works"; frozen base "read, never written", Soup show post, first
  paragraph):
      T  = X A^T                     (rank-r down projection)
      Y  = X deq(Wq)^T + s T B^T,    s = alpha / r
      U  = dY B
      dX = dY deq(Wq) + s U A
      dB = s dY^T T
      dA = s U^T X
  There is no gradient for the frozen base.  All products are evaluated in
  fp64 on the stored (bf16 / dequantised) values.

* Block formats (Surogate README, "LoRA & QLoRA" row: BnB/NF4 bases; GGUF
  blog: GGUF Q8_0/Q4_0 bases).  The pages print no table or block layout; the
  readings used here:
      NF4   64 codes per block along K, two per byte (element 2j in the high
            nibble of byte j), fp32 absmax per block, or int8 absmax with one
            fp32 scale per 256 blocks (double quantisation).  Levels: the
            NormalFloat-4 construction (16 normal quantiles incl. an exact 0,
            scaled to [-1, 1]), stored as fp32.
            value = bf16_rn( f32_rn( level[c] * absmax' ) ),
            absmax' = absmax or f32_rn( f32(q) * scale2 ).
      Q4_0  32 elements per 18-byte block {fp16 d, 16 bytes}; element i < 16
            in the low nibble of byte i, element i+16 in its high nibble.
            value = bf16_rn( (nib - 8) * f32(d) )   (the product is exact)
      Q8_0  32 elements per 34-byte block {fp16 d, int8[32]}.
            value = bf16_rn( q * f32(d) )           (the product is exact)
      bf16  the stored value.

  Further base formats (Surogate README: "Native GGUF" row names K-quants,
  the quickstart quantises to q4_k_m; "LoRA & QLoRA" and "Native precision
  recipes" rows name FP8 and NVFP4 bases; heatdrop.ai summary: FP8 E4M3 and
  NVFP4 (E2M1) recipes).  The pages print no layout; the readings:
      NF4 with an 8-bit map (QLoRA-style double quantisation): the absmax
            byte is an index into a 256-entry fp32 map and a fixed offset is
            added back:  absmax' = f32_rn( f32_rn(map[q] * scale2) + offset )
      Q4_K  GGUF super-blocks of 256 elements, 144 bytes {fp16 d, fp16 dmin,
            12 bytes of eight 6-bit sub-block scales sc[j] and mins m[j],
            128 bytes of 4-bit codes}; sub-block j = 32 elements.
            value = bf16_rn( f32_rn( (d sc[j]) q - (dmin m[j]) ) )
            (both products are exact in fp32, so one rounding)
      FP8   E4M3 codes (OCP 8-bit float, no infinities, S.1111.111 = NaN),
            one per element, with one fp32 scale for the whole tensor.
            value = bf16_rn( f32_rn( e4m3(c) * scale ) )
      NVFP4 E2M1 codes, two per byte (element 2j in the LOW nibble of byte
            j), an E4M3 scale per 16 consecutive elements and one fp32
            scale for the whole tensor.
            value = bf16_rn( f32_rn( e2m1(c) * f32_rn( e4m3(s_blk) * scale ) ) )
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

# NormalFloat-4 levels, fp32 (QLoRA's NormalFloat: 8 positive and 7 negative
# standard-normal quantiles at probabilities evenly spaced from
# delta = ((1 - 1/30) + (1 - 1/32)) / 2 to 1/2, plus an exact zero, divided by
# the largest quantile, rounded to fp32).
NF4_LEVELS = np.array([
    -1.0, -0.6961928, -0.52507293, -0.39491743,
    -0.28444132, -0.1847734, -0.09104998, 0.0,
    0.079580314, 0.16093014, 0.24611226, 0.33791512,
    0.44070974, 0.5626169, 0.72295666, 1.0,
], dtype=np.float32)


# ----------------------------------------------------------------------------
# rounding helpers
# ----------------------------------------------------------------------------
def bf16_round_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 to the nearest bf16 value (ties to even), returned as fp32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return u.astype(np.uint32).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# dequantisation (block decode)
# ----------------------------------------------------------------------------
def _dequant_nf4(w: Dict, N: int, K: int) -> np.ndarray:
    packed = np.asarray(w["data"], dtype=np.uint8).reshape(-1)
    assert packed.size == N * K // 2
    codes = np.empty(N * K, dtype=np.uint8)
    codes[0::2] = packed >> 4
    codes[1::2] = packed & 0x0F
    codes = codes.reshape(-1, 64)
    nblk = codes.shape[0]
    if "absmax" in w and w["absmax"] is not None:
        amax = np.asarray(w["absmax"], dtype=np.float32).reshape(-1)
    else:
        scale2 = np.asarray(w["absmax_scale"], dtype=np.float32).reshape(-1)
        group = int(w.get("dq_group", 256))
        g = np.arange(nblk) // group
        if w.get("absmax_map") is None:
            q = np.asarray(w["absmax_q"], dtype=np.int8).reshape(-1).astype(np.float32)
            amax = (q * scale2[g]).astype(np.float32)          # fp32 product
        else:
            # the byte indexes the 8-bit map; then scale and offset, each step
            # rounded to fp32
            idx = np.asarray(w["absmax_q"]).reshape(-1).view(np.uint8).astype(np.int64)
            amap = np.asarray(w["absmax_map"], dtype=np.float32).reshape(256)
            amax = (amap[idx] * scale2[g]).astype(np.float32)
            amax = (amax + np.float32(w["absmax_offset"])).astype(np.float32)
    assert amax.size == nblk
    prod = (NF4_LEVELS[codes] * amax[:, None]).astype(np.float32)  # fp32 product
    return bf16_round_f32(prod).astype(np.float64).reshape(N, K)


def _gguf_blocks(w: Dict, N: int, K: int, rec: int) -> np.ndarray:
    data = np.asarray(w["data"], dtype=np.uint8).reshape(-1)
    assert data.size == N * K // 32 * rec
    return data.reshape(-1, rec)


def _dequant_q4_0(w: Dict, N: int, K: int) -> np.ndarray:
    blk = _gguf_blocks(w, N, K, 18)
    d = blk[:, 0:2].copy().view("<f2").astype(np.float32).reshape(-1)
    qs = blk[:, 2:18]
    nib = np.concatenate([qs & 0x0F, qs >> 4], axis=1).astype(np.int32)  # [nb, 32]
    prod = ((nib - 8).astype(np.float32) * d[:, None]).astype(np.float32)
    return bf16_round_f32(prod).astype(np.float64).reshape(N, K)


def _dequant_q8_0(w: Dict, N: int, K: int) -> np.ndarray:
    blk = _gguf_blocks(w, N, K, 34)
    d = blk[:, 0:2].copy().view("<f2").astype(np.float32).reshape(-1)
    q = blk[:, 2:34].copy().view(np.int8).astype(np.float32)
    prod = (q * d[:, None]).astype(np.float32)
    return bf16_round_f32(prod).astype(np.float64).reshape(N, K)


def _dequant_q4_k(w: Dict, N: int, K: int) -> np.ndarray:
    assert K % 256 == 0
    data = np.asarray(w["data"], dtype=np.uint8).reshape(-1)
    assert data.size == N * K // 256 * 144
    sb = data.reshape(-1, 144)
    d = sb[:, 0:2].copy().view("<f2").astype(np.float32).reshape(-1)
    dmin = sb[:, 2:4].copy().view("<f2").astype(np.float32).reshape(-1)
    sc, mn = q4_k_scale_min(sb[:, 4:16])                      # [nsb, 8] each
    qs = sb[:, 16:144].reshape(-1, 4, 32)                     # 4 chunks of 32 bytes
    # chunk c: low nibbles are sub-block 2c, high nibbles sub-block 2c+1
    q = np.stack([qs & 0x0F, qs >> 4], axis=2).reshape(-1, 8, 32).astype(np.float32)
    dsc = (d[:, None] * sc.astype(np.float32)).astype(np.float32)      # exact
    mmn = (dmin[:, None] * mn.astype(np.float32)).astype(np.float32)   # exact
    prod = (dsc[:, :, None] * q).astype(np.float32)                    # exact
    val = (prod - mmn[:, :, None]).astype(np.float32)                  # one rounding
    return bf16_round_f32(val).astype(np.float64).reshape(N, K)


def q4_k_scale_min(b: np.ndarray):
    """Eight 6-bit scales and mins from the 12 packed bytes of a Q4_K
    super-block ([n, 12] uint8 -> two [n, 8] int arrays).  Sub-blocks 0..3:
    scale = low 6 bits of byte j, min = low 6 bits of byte j+4.  Sub-blocks
    4..7: low 4 bits from byte j+4 (scale: its low nibble, min: its high
    nibble), top 2 bits from the top 2 bits of byte j-4 (scale) and byte j
    (min)."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    sc = np.empty((b.shape[0], 8), dtype=np.int64)
    mn = np.empty((b.shape[0], 8), dtype=np.int64)
    for j in range(4):
        sc[:, j] = b[:, j] & 63
        mn[:, j] = b[:, j + 4] & 63
    for j in range(4, 8):
        sc[:, j] = (b[:, j + 4] & 0x0F) | ((b[:, j - 4] >> 6) << 4)
        mn[:, j] = (b[:, j + 4] >> 4) | ((b[:, j] >> 6) << 4)
    return sc, mn


def e4m3_value(code) -> np.ndarray:
    """OCP 8-bit float E4M3 (bias 7, 3 mantissa bits, subnormals, no
    infinities; exponent and mantissa all ones is NaN), as fp64."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0x0F
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    v = sign * mag
    return np.where((e == 15) & (m == 7), np.nan, v)


def e2m1_value(code) -> np.ndarray:
    """4-bit float E2M1 (bias 1, 1 mantissa bit, a subnormal 0.5, no
    infinities or NaN), as fp64; only the low 4 bits of `code` are used."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64) & 0x0F
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2((e - 1).astype(np.float64)))
    return sign * mag


def _dequant_fp8(w: Dict, N: int, K: int) -> np.ndarray:
    c = np.asarray(w["data"], dtype=np.uint8).reshape(-1)
    assert c.size == N * K
    scale = np.float32(np.asarray(w["tensor_scale"], dtype=np.float32).reshape(-1)[0])
    prod = (e4m3_value(c).astype(np.float32) * scale).astype(np.float32)   # e4m3 is exact in fp32
    return bf16_round_f32(prod).astype(np.float64).reshape(N, K)


def _dequant_nvfp4(w: Dict, N: int, K: int) -> np.ndarray:
    assert K % 16 == 0
    packed = np.asarray(w["data"], dtype=np.uint8).reshape(-1)
    assert packed.size == N * K // 2
    codes = np.empty(N * K, dtype=np.uint8)
    codes[0::2] = packed & 0x0F
    codes[1::2] = packed >> 4
    sblk = np.asarray(w["block_scale"], dtype=np.uint8).reshape(-1)
    assert sblk.size == N * K // 16
    scale = np.float32(np.asarray(w["tensor_scale"], dtype=np.float32).reshape(-1)[0])
    b = (e4m3_value(sblk).astype(np.float32) * scale).astype(np.float32)  # block factor, fp32
    v = (e2m1_value(codes).astype(np.float32).reshape(-1, 16) * b[:, None]).astype(np.float32)
    return bf16_round_f32(v).astype(np.float64).reshape(N, K)


def dequant(w: Dict) -> np.ndarray:
    """Decoded base weight deq(Wq) as fp64 [N, K] (every value a bf16 value)."""
    N, K, fmt = int(w["N"]), int(w["K"]), w["fmt"]
    if fmt == "bf16":
        return bf16_bits_to_f64(w["data"]).reshape(N, K)
    if fmt == "nf4":
        return _dequant_nf4(w, N, K)
    if fmt == "q4_0":
        return _dequant_q4_0(w, N, K)
    if fmt == "q8_0":
        return _dequant_q8_0(w, N, K)
    if fmt == "q4_k":
        return _dequant_q4_k(w, N, K)
    if fmt == "fp8_e4m3":
        return _dequant_fp8(w, N, K)
    if fmt == "nvfp4":
        return _dequant_nvfp4(w, N, K)
    raise ValueError(fmt)


def dequant_bf16_bits(w: Dict) -> np.ndarray:
    """deq(Wq) as bf16 bit patterns (uint16 [N, K]) for bit-exact comparison."""
    v = dequant(w).astype(np.float32)
    return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------
def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def linear_fwd(X, Wd, A, B, alpha: float):
    """Y = X Wd^T + s (X A^T) B^T, s = alpha / r.  Returns (Y, T)."""
    X, Wd, A, B = _f64(X), _f64(Wd), _f64(A), _f64(B)
    r = A.shape[0]
    s = float(alpha) / r
    T = X @ A.T
    Y = X @ Wd.T + s * (T @ B.T)
    return Y, T


def linear_fwd_rows(X_rows, Wd, A, B, alpha: float):
    """Forward on a subset of rows (rows are independent)."""
    return linear_fwd(X_rows, Wd, A, B, alpha)


def linear_bwd(X, Wd, A, B, dY, alpha: float):
    """Backward of the layer.  Returns dict with U, dX, dA, dB (fp64)."""
    X, Wd, A, B, dY = _f64(X), _f64(Wd), _f64(A), _f64(B), _f64(dY)
    r = A.shape[0]
    s = float(alpha) / r
    T = X @ A.T
    U = dY @ B
    dX = dY @ Wd + s * (U @ A)
    dB = s * (dY.T @ T)
    dA = s * (U.T @ X)
    return {"T": T, "U": U, "dX": dX, "dA": dA, "dB": dB}


def linear_bwd_rows(dY_rows, Wd, A, B, alpha: float):
    """dX on a subset of rows: dY_rows Wd + s (dY_rows B) A."""
    dY, Wd, A, B = _f64(dY_rows), _f64(Wd), _f64(A), _f64(B)
    s = float(alpha) / A.shape[0]
    return dY @ Wd + s * ((dY @ B) @ A)


def linear_bwd_adapter_grads(X, A, B, dY, alpha: float):
    """dA, dB (and T, U) over all rows without touching the base weight."""
    X, A, B, dY = _f64(X), _f64(A), _f64(B), _f64(dY)
    s = float(alpha) / A.shape[0]
    T = X @ A.T
    U = dY @ B
    return {"T": T, "U": U, "dA": s * (U.T @ X), "dB": s * (dY.T @ T)}


# ----------------------------------------------------------------------------
# grouped (mixture-of-experts) variant: the same layer per expert over the
# rows routed to it (rows sorted by expert, offsets[E+1]).
# ----------------------------------------------------------------------------
def grouped_fwd(X, Wds: Sequence[np.ndarray], A, B, offsets, alpha: float):
    X = _f64(X)
    E = len(Wds)
    N = Wds[0].shape[0]
    r = np.asarray(A).shape[1]
    Y = np.zeros((X.shape[0], N))
    T = np.zeros((X.shape[0], r))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            Y[lo:hi], T[lo:hi] = linear_fwd(X[lo:hi], Wds[e], A[e], B[e], alpha)
    return Y, T


def grouped_bwd(X, Wds: Sequence[np.ndarray], A, B, dY, offsets, alpha: float):
    X, dY = _f64(X), _f64(dY)
    E = len(Wds)
    K = X.shape[1]
    N = Wds[0].shape[0]
    r = np.asarray(A).shape[1]
    dX = np.zeros((X.shape[0], K))
    dA = np.zeros((E, r, K))
    dB = np.zeros((E, N, r))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            g = linear_bwd(X[lo:hi], Wds[e], A[e], B[e], dY[lo:hi], alpha)
            dX[lo:hi], dA[e], dB[e] = g["dX"], g["dA"], g["dB"]
    return {"dX": dX, "dA": dA, "dB": dB}


# ----------------------------------------------------------------------------
# fused projections that share their input (q, k, v of attention; gate, up of
# the MLP): P LoRA linears over the same X, each with its own base rows and
# adapter, computed as one call.  Y is the projections' outputs side by side;
# the input gradient is the sum of the projections' input gradients (what the
# layer that feeds X receives); dA, dB stay per projection.  (Surogate README,
# design bullet "Kernels that do more per launch".)
# ----------------------------------------------------------------------------
def multi_linear_fwd(X, Wds: Sequence[np.ndarray], As: Sequence[np.ndarray], Bs: Sequence[np.ndarray],
                     alpha: float):
    """Returns (Y [M, sum N_p], T [M, P r]) with projection p in its own column block."""
    outs = [linear_fwd(X, Wd, A, B, alpha) for Wd, A, B in zip(Wds, As, Bs)]
    return np.concatenate([y for y, _ in outs], axis=1), np.concatenate([t for _, t in outs], axis=1)


def multi_linear_bwd(X, Wds: Sequence[np.ndarray], As: Sequence[np.ndarray], Bs: Sequence[np.ndarray], dY,
                     alpha: float):
    """dY [M, sum N_p] (projection p in its column block).  Returns dict with dX
    (summed over projections), dA [P, r, K], dB [sum N_p, r] (projection p's
    rows in its block), T and U [M, P r]."""
    dY = _f64(dY)
    offs = np.cumsum([0] + [np.asarray(W).shape[0] for W in Wds])
    gs = [linear_bwd(X, Wd, A, B, dY[:, offs[p]:offs[p + 1]], alpha)
          for p, (Wd, A, B) in enumerate(zip(Wds, As, Bs))]
    return {"dX": sum(g["dX"] for g in gs), "dA": np.stack([g["dA"] for g in gs]),
            "dB": np.concatenate([g["dB"] for g in gs], axis=0),
            "T": np.concatenate([g["T"] for g in gs], axis=1), "U": np.concatenate([g["U"] for g in gs], axis=1)}


# ----------------------------------------------------------------------------
# stacked adapters: several LoRA pairs on the same frozen base, trained (or
# kept frozen) on top of each other without merging them into the base
# (heatdrop.ai summary, "Key highlights"; Surogate README, "LoRA & QLoRA"
# row).  Adapter i has its own rank r_i and scale s_i = alpha_i / r_i.
# ----------------------------------------------------------------------------
def stacked_linear_fwd(X, Wd, As: Sequence[np.ndarray], Bs: Sequence[np.ndarray], alphas: Sequence[float]):
    """Y = X Wd^T + sum_i s_i (X A_i^T) B_i^T.  Returns (Y, T) with T = [T_0 | T_1 | ...]."""
    X, Wd = _f64(X), _f64(Wd)
    Y = X @ Wd.T
    Ts = []
    for A, B, alpha in zip(As, Bs, alphas):
        A, B = _f64(A), _f64(B)
        s = float(alpha) / A.shape[0]
        T = X @ A.T
        Y = Y + s * (T @ B.T)
        Ts.append(T)
    return Y, np.concatenate(Ts, axis=1)


def stacked_linear_bwd(X, Wd, As: Sequence[np.ndarray], Bs: Sequence[np.ndarray], dY, alphas: Sequence[float]):
    """dX = dY Wd + sum_i s_i (dY B_i) A_i;  dA_i = s_i U_i^T X, dB_i = s_i dY^T T_i.
    Returns dict with dX and lists dA, dB."""
    X, Wd, dY = _f64(X), _f64(Wd), _f64(dY)
    dX = dY @ Wd
    dA, dB = [], []
    for A, B, alpha in zip(As, Bs, alphas):
        A, B = _f64(A), _f64(B)
        s = float(alpha) / A.shape[0]
        T = X @ A.T
        U = dY @ B
        dX = dX + s * (U @ A)
        dA.append(s * (U.T @ X))
        dB.append(s * (dY.T @ T))
    return {"dX": dX, "dA": dA, "dB": dB}


# ----------------------------------------------------------------------------
# gate / up projections with the SwiGLU activation (the MLP of the Llama and
# Qwen3 layers the workloads are shaped after): two LoRA linears over the same
# X, G = X Wg^T + s Tg Bg^T and U = X Wu^T + s Tu Bu^T, and
#     H = silu(G) * U,   silu(g) = g * sigmoid(g).
# Backward from dH: dG = dH * U * sigmoid(G) * (1 + G (1 - sigmoid(G))),
# dU = dH * silu(G), then the fused-projection backward with dY = [dG | dU]
# (the input gradient summed over both projections).
# ----------------------------------------------------------------------------
def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def swiglu_fwd(X, Wg, Wu, Ag, Au, Bg, Bu, alpha: float):
    """Returns (H [M, I], G [M, I], U [M, I], T [M, 2r] = [Tg | Tu])."""
    G, Tg = linear_fwd(X, Wg, Ag, Bg, alpha)
    U, Tu = linear_fwd(X, Wu, Au, Bu, alpha)
    H = G * _sigmoid(G) * U
    return H, G, U, np.concatenate([Tg, Tu], axis=1)


def swiglu_grad_gate_up(G, U, dH):
    """(dG, dU) of H = silu(G) * U."""
    G, U, dH = _f64(G), _f64(U), _f64(dH)
    sg = _sigmoid(G)
    return dH * U * sg * (1.0 + G * (1.0 - sg)), dH * G * sg


def swiglu_bwd(X, Wg, Wu, Ag, Au, Bg, Bu, dH, alpha: float, G=None, U=None):
    """dX (summed over gate and up), dA [2, r, K], dB [2 I, r] (gate rows, then
    up rows).  G, U: the pre-activations the backward starts from (default:
    recomputed exactly)."""
    if G is None or U is None:
        _, G, U, _ = swiglu_fwd(X, Wg, Wu, Ag, Au, Bg, Bu, alpha)
    dG, dU = swiglu_grad_gate_up(G, U, dH)
    g = multi_linear_bwd(X, [Wg, Wu], [Ag, Au], [Bg, Bu], np.concatenate([dG, dU], axis=1), alpha)
    return {"dX": g["dX"], "dA": g["dA"], "dB": g["dB"], "dG": dG, "dU": dU}

