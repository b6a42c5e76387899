"""Seeded synthetic inputs for the quantised-base LoRA linear.

This module is shared by the CPU oracle's tests and the CUDA path's tests and
benchmark.  It draws random tensors, rounds them to the storage types the
layer consumes (bf16 activations/adapters, fp32 weights before quantisation)
and packs frozen base weights into the four block formats.  It holds none of
the layer's arithmetic: no dequantisation, no products, no gradients.

Packing (quantisation) is input preparation: the frozen base arrives already
quantised (Surogate README, capability table, "LoRA & QLoRA" row names
BnB/NF4 bases; bytechap GGUF blog, "How it works", uses GGUF bases).  Any
byte pattern is a valid input to the layer; the rules below only decide which
codes a given fp32 weight turns into.

Stream ids: every tensor is drawn from ``numpy.random.default_rng`` seeded
with ``[seed, layer, linear, stream]`` so each tensor has its own PCG64
sub-stream and a tensor's values do not depend on what else was drawn.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

# Sub-stream ids, one per tensor kind.
S_X, S_W, S_A, S_B, S_DY, S_ROUTER = 0, 1, 2, 3, 4, 5

FORMATS = ("bf16", "nf4", "q8_0", "q4_0", "q4_k", "fp8_e4m3", "nvfp4")


# ----------------------------------------------------------------------------
# plain value conversions used to store drawn values
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rng_for(seed: int, layer: int, linear: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(layer), int(linear), int(stream)])


def normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """N(0, std) drawn in fp64, rounded to fp32, then to bf16 (uint16 bits)."""
    x = rng.standard_normal(size=shape, dtype=np.float64) * std
    return f32_to_bf16_bits(x.astype(np.float32))


def normal_f32(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float64) * std
    return x.astype(np.float32)


# ----------------------------------------------------------------------------
# Block packers (quantisers).  They produce the frozen base's bytes.
# ----------------------------------------------------------------------------
def _nf4_levels() -> np.ndarray:
    """NormalFloat-4 levels: 8 positive and 7 negative standard-normal
    quantiles at evenly spaced probabilities from delta to 1/2, plus 0,
    divided by the largest (QLoRA's NormalFloat construction)."""
    from scipy.stats import norm

    delta = 0.5 * ((1.0 - 1.0 / 30.0) + (1.0 - 1.0 / 32.0))
    pos = norm.ppf(np.linspace(delta, 0.5, 9)[:-1])
    neg = -norm.ppf(np.linspace(delta, 0.5, 8)[:-1])
    lv = np.sort(np.concatenate([pos, [0.0], neg]))
    return (lv / lv.max()).astype(np.float32)


_NF4_MID: Optional[np.ndarray] = None


def _nf4_midpoints() -> np.ndarray:
    global _NF4_MID
    if _NF4_MID is None:
        lv = _nf4_levels().astype(np.float64)
        _NF4_MID = 0.5 * (lv[1:] + lv[:-1])  # exact in fp64
    return _NF4_MID


def float8_map() -> np.ndarray:
    """An 8-bit float map for absmax codes (QLoRA-style double
    quantisation): the values of the 256 E4M3 codes divided by the largest
    (448), the two NaN codes standing in for +1 and -1.  Computed with the
    E4M3 conversion of PyTorch."""
    import torch

    v = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    v[0x7F], v[0xFF] = 448.0, -448.0
    return (v / 448.0).astype(np.float32)


def pack_nf4(w: np.ndarray, double_quant: bool, dq_group: int = 256, dq_map: bool = False) -> Dict[str, np.ndarray]:
    """w: fp32 [N, K], K % 64 == 0.  Blocks of 64 consecutive K-elements.

    absmax = max|w| over the block (fp32).  code = the nearest NF4 level to
    w/absmax (ties to the lower index); an all-zero block gets the zero code 7.
    Two codes per byte: element 2j in the high nibble of byte j.

    Double quantisation: absmax values are grouped 256 at a time (flattened
    block order); scale2 = max(absmax in group)/127 (fp32) and
    absmax_q = clamp(round_half_even(absmax/scale2), 0, 127) as int8.  Codes
    are chosen with the exact fp32 absmax (codes first, then the constants).

    dq_map (QLoRA style): offset = mean of all absmax values (fp32); per group
    scale2 = max |absmax - offset| (fp32); the code is the index of the
    float8_map() entry nearest to (absmax - offset) / scale2 (lowest index on
    ties); stored as bytes in absmax_q with the map and the offset.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % 64 == 0
    blocks = w.reshape(-1, 64)
    amax = np.abs(blocks).max(axis=1).astype(np.float32)
    codes = np.empty(blocks.shape, dtype=np.uint8)
    mid = _nf4_midpoints()
    step = 1 << 16
    for i in range(0, blocks.shape[0], step):
        b = blocks[i:i + step]
        a = amax[i:i + step]
        safe = np.where(a > 0, a, np.float32(1.0))
        x = (b / safe[:, None]).astype(np.float32).astype(np.float64)
        c = np.searchsorted(mid, x, side="left").astype(np.uint8)
        c[a == 0] = 7
        codes[i:i + step] = c
    flat = codes.reshape(-1)
    packed = ((flat[0::2] << 4) | flat[1::2]).astype(np.uint8)
    out = {"fmt": "nf4", "N": N, "K": K, "data": packed}
    if double_quant and dq_map:
        nb = amax.shape[0]
        ng = (nb + dq_group - 1) // dq_group
        offset = np.float32(amax.astype(np.float64).mean())
        cen = amax.astype(np.float64) - float(offset)
        pad = np.zeros(ng * dq_group)
        pad[:nb] = np.abs(cen)
        scale2 = pad.reshape(ng, dq_group).max(axis=1).astype(np.float32)
        s_rep = np.repeat(scale2, dq_group)[:nb].astype(np.float64)
        x = np.where(s_rep > 0, cen / np.where(s_rep > 0, s_rep, 1.0), 0.0)
        amap = float8_map().astype(np.float64)
        order = np.argsort(amap, kind="stable")
        sv = amap[order]
        j = np.clip(np.searchsorted(sv, x), 1, 255)
        pick = np.where(np.abs(x - sv[j - 1]) <= np.abs(sv[j] - x), j - 1, j)
        code = order[pick].astype(np.uint8)
        out["absmax_q"] = code.view(np.int8)
        out["absmax_scale"] = scale2
        out["absmax_map"] = amap.astype(np.float32)
        out["absmax_offset"] = float(offset)
        out["dq_group"] = dq_group
    elif double_quant:
        nb = amax.shape[0]
        ng = (nb + dq_group - 1) // dq_group
        pad = np.zeros(ng * dq_group, dtype=np.float32)
        pad[:nb] = amax
        gmax = pad.reshape(ng, dq_group).max(axis=1)
        scale2 = (gmax / np.float32(127.0)).astype(np.float32)
        s_rep = np.repeat(scale2, dq_group)[:nb]
        safe = np.where(s_rep > 0, s_rep, np.float32(1.0))
        q = np.rint((amax / safe).astype(np.float32))  # rint = ties to even
        q = np.clip(q, 0, 127)
        q[s_rep == 0] = 0
        out["absmax_q"] = q.astype(np.int8)
        out["absmax_scale"] = scale2
        out["dq_group"] = dq_group
    else:
        out["absmax"] = amax
    return out


def _round_half_away(x: np.ndarray) -> np.ndarray:
    return np.sign(x) * np.floor(np.abs(x) + 0.5)


def pack_q4_0(w: np.ndarray) -> Dict[str, np.ndarray]:
    """GGUF Q4_0: blocks of 32 along K, each {fp16 d, uint8 qs[16]} = 18 B.

    m = the element of largest magnitude (first one on ties);
    d = fp16(m / -8); nib = clamp(round_half_away(w/d) + 8, 0, 15); element
    i < 16 sits in the low nibble of qs[i], element i+16 in its high nibble.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % 32 == 0
    b = w.reshape(-1, 32).astype(np.float64)
    idx = np.argmax(np.abs(b), axis=1)
    m = b[np.arange(b.shape[0]), idx]
    d16 = (m.astype(np.float32) / np.float32(-8.0)).astype(np.float16)
    d = d16.astype(np.float64)
    safe = np.where(d != 0, d, 1.0)
    nib = np.clip(_round_half_away(b / safe[:, None]) + 8, 0, 15)
    nib[d == 0] = 8
    nib = nib.astype(np.uint8)
    qs = (nib[:, :16] | (nib[:, 16:] << 4)).astype(np.uint8)
    rec = np.empty((b.shape[0], 18), dtype=np.uint8)
    rec[:, 0:2] = d16.view(np.uint8).reshape(-1, 2)
    rec[:, 2:] = qs
    return {"fmt": "q4_0", "N": N, "K": K, "data": rec.reshape(-1)}


def pack_q8_0(w: np.ndarray) -> Dict[str, np.ndarray]:
    """GGUF Q8_0: blocks of 32 along K, each {fp16 d, int8 qs[32]} = 34 B.

    d = fp16(max|w| / 127); q = clamp(round_half_away(w/d), -127, 127).
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % 32 == 0
    b = w.reshape(-1, 32).astype(np.float64)
    amax = np.abs(b).max(axis=1)
    d16 = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float16)
    d = d16.astype(np.float64)
    safe = np.where(d != 0, d, 1.0)
    q = np.clip(_round_half_away(b / safe[:, None]), -127, 127)
    q[d == 0] = 0
    rec = np.empty((b.shape[0], 34), dtype=np.uint8)
    rec[:, 0:2] = d16.view(np.uint8).reshape(-1, 2)
    rec[:, 2:] = q.astype(np.int8).view(np.uint8)
    return {"fmt": "q8_0", "N": N, "K": K, "data": rec.reshape(-1)}


def pack_q4_k(w: np.ndarray) -> Dict[str, np.ndarray]:
    """GGUF Q4_K: super-blocks of 256 along K, 144 bytes each: fp16 d, fp16
    dmin, 12 bytes of eight 6-bit (scale, min) pairs, 128 bytes of codes.

    Sub-block j (32 elements): lo = min(0, min w), hi = max w,
    scale_j = (hi - lo)/15, min_j = -lo.  d = fp16(max scale_j / 63),
    dmin = fp16(max min_j / 63); sc_j = clamp(rint(scale_j/d), 0, 63),
    m_j = clamp(rint(min_j/dmin), 0, 63); q = clamp(rint((w + dmin m_j) /
    (d sc_j)), 0, 15).  Chunk c of 64 elements takes bytes 32c..32c+31 of the
    codes: sub-block 2c in the low nibbles, 2c+1 in the high nibbles.
    Scale bytes: sub-blocks 0..3 in the low 6 bits of bytes j (scale) and
    j+4 (min); sub-blocks 4..7 keep their low 4 bits in byte j+4 (scale low
    nibble, min high nibble) and their top 2 bits in the top bits of bytes
    j-4 (scale) and j (min).
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % 256 == 0
    sb = w.reshape(-1, 8, 32).astype(np.float64)
    lo = np.minimum(sb.min(axis=2), 0.0)
    hi = sb.max(axis=2)
    scale = (hi - lo) / 15.0
    mins = -lo
    d16 = (scale.max(axis=1) / 63.0).astype(np.float16)
    m16 = (mins.max(axis=1) / 63.0).astype(np.float16)
    d, dm = d16.astype(np.float64), m16.astype(np.float64)
    sc = np.clip(np.rint(scale / np.where(d > 0, d, 1.0)[:, None]), 0, 63).astype(np.int64)
    mn = np.clip(np.rint(mins / np.where(dm > 0, dm, 1.0)[:, None]), 0, 63).astype(np.int64)
    sc[d == 0] = 0
    mn[dm == 0] = 0
    step = d[:, None] * sc
    q = np.rint((sb + (dm[:, None] * mn)[:, :, None]) / np.where(step > 0, step, 1.0)[:, :, None])
    q = np.clip(q, 0, 15)
    q[np.broadcast_to((step == 0)[:, :, None], q.shape)] = 0
    q = q.astype(np.uint8)
    nsb = sb.shape[0]
    rec = np.zeros((nsb, 144), dtype=np.uint8)
    rec[:, 0:2] = d16.view(np.uint8).reshape(-1, 2)
    rec[:, 2:4] = m16.view(np.uint8).reshape(-1, 2)
    b = np.zeros((nsb, 12), dtype=np.int64)
    for j in range(4):
        b[:, j] = sc[:, j] | ((sc[:, j + 4] >> 4) << 6)
        b[:, j + 4] = mn[:, j] | ((mn[:, j + 4] >> 4) << 6)
        b[:, j + 8] = (sc[:, j + 4] & 0x0F) | ((mn[:, j + 4] & 0x0F) << 4)
    rec[:, 4:16] = b.astype(np.uint8)
    qc = q.reshape(nsb, 4, 2, 32)
    rec[:, 16:] = (qc[:, :, 0, :] | (qc[:, :, 1, :] << 4)).reshape(nsb, 128)
    return {"fmt": "q4_k", "N": N, "K": K, "data": rec.reshape(-1)}


def _to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Round to E4M3 codes (nearest, ties to even; saturated to +-448) with
    PyTorch's conversion."""
    import torch

    t = torch.from_numpy(np.clip(np.ascontiguousarray(x, dtype=np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def _e4m3_codes_to_f32(c: np.ndarray) -> np.ndarray:
    import torch

    return torch.from_numpy(np.ascontiguousarray(c, dtype=np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def pack_fp8_e4m3(w: np.ndarray) -> Dict[str, np.ndarray]:
    """FP8 E4M3 codes with one fp32 scale for the tensor: scale =
    max|w| / 448 (1 if the tensor is zero), code = E4M3(w / scale)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    amax = np.float32(np.abs(w).max()) if w.size else np.float32(0)
    scale = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
    codes = _to_e4m3_codes((w / scale).astype(np.float32))
    return {"fmt": "fp8_e4m3", "N": N, "K": K, "data": codes.reshape(-1),
            "tensor_scale": np.array([scale], dtype=np.float32)}


_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def pack_nvfp4(w: np.ndarray) -> Dict[str, np.ndarray]:
    """NVFP4: E2M1 codes in blocks of 16 along K, an E4M3 scale per block
    and one fp32 scale for the tensor.  scale = max|w| / (6 * 448);
    block scale = E4M3(max|w in block| / 6 / scale); with the block factor
    b = f32(E4M3 value) * scale, each element takes the E2M1 magnitude
    nearest to |w| / b (lower one on ties) and the sign of w.  Element 2j in
    the low nibble of byte j."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % 16 == 0
    amax = np.float32(np.abs(w).max()) if w.size else np.float32(0)
    ts = np.float32(amax / np.float32(6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    blk = w.reshape(-1, 16)
    bmax = np.abs(blk).max(axis=1).astype(np.float32)
    sc = _to_e4m3_codes((bmax / np.float32(6.0) / ts).astype(np.float32))
    b = (_e4m3_codes_to_f32(sc) * ts).astype(np.float32).astype(np.float64)
    x = np.abs(blk.astype(np.float64)) / np.where(b > 0, b, 1.0)[:, None]
    mid = (_E2M1_MAG[:-1] + _E2M1_MAG[1:]) / 2
    mag = np.searchsorted(mid, x, side="left")
    mag[np.broadcast_to((b == 0)[:, None], mag.shape)] = 0
    code = (mag | np.where(blk < 0, 8, 0)).astype(np.uint8).reshape(-1)
    packed = (code[0::2] | (code[1::2] << 4)).astype(np.uint8)
    return {"fmt": "nvfp4", "N": N, "K": K, "data": packed, "block_scale": sc.reshape(-1),
            "tensor_scale": np.array([ts], dtype=np.float32)}


def pack(w_f32: np.ndarray, fmt: str, double_quant: bool = False) -> Dict[str, np.ndarray]:
    if fmt == "bf16":
        N, K = w_f32.shape
        return {"fmt": "bf16", "N": N, "K": K, "data": f32_to_bf16_bits(w_f32).reshape(-1)}
    if fmt == "nf4":
        return pack_nf4(w_f32, double_quant)
    if fmt == "q8_0":
        return pack_q8_0(w_f32)
    if fmt == "q4_0":
        return pack_q4_0(w_f32)
    if fmt == "q4_k":
        return pack_q4_k(w_f32)
    if fmt == "fp8_e4m3":
        return pack_fp8_e4m3(w_f32)
    if fmt == "nvfp4":
        return pack_nvfp4(w_f32)
    if fmt == "nf4_dqmap":
        return pack_nf4(w_f32, True, dq_map=True)
    raise ValueError(fmt)


def weight_nbytes(qw: Dict) -> int:
    n = qw["data"].nbytes
    for k in ("absmax", "absmax_q", "absmax_scale", "absmax_map", "block_scale", "tensor_scale"):
        if k in qw:
            n += qw[k].nbytes
    return n


# ----------------------------------------------------------------------------
# Workloads (layer shapes from the configurations named in the pages'
# benchmark and model tables: Qwen3-0.6B, Llama-3.1-8B, Qwen3-8B, a Qwen3-MoE
# style expert layer).
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Linear:
    name: str
    K: int
    N: int


@dataclasses.dataclass
class Workload:
    name: str
    fmt: str
    double_quant: bool
    M: int
    rank: int
    alpha: float
    linears: List[Linear]
    w_std: float = 0.02
    a_std: Optional[float] = None  # None -> 1/sqrt(K)
    b_std: float = 0.01


def _decoder(hidden, q_out, kv_out, inter):
    return [
        Linear("q_proj", hidden, q_out),
        Linear("k_proj", hidden, kv_out),
        Linear("v_proj", hidden, kv_out),
        Linear("o_proj", q_out, hidden),
        Linear("gate_proj", hidden, inter),
        Linear("up_proj", hidden, inter),
        Linear("down_proj", inter, hidden),
    ]


WORKLOADS: Dict[str, Workload] = {
    "tiny_nf4": Workload("tiny_nf4", "nf4", False, 64, 8, 16.0, [Linear("tiny", 256, 256)],
                         a_std=1.0 / 16.0),
    "qwen3_0p6b_bf16": Workload("qwen3_0p6b_bf16", "bf16", False, 8192, 16, 32.0,
                                _decoder(1024, 2048, 1024, 3072)),
    "llama31_8b_nf4dq": Workload("llama31_8b_nf4dq", "nf4", True, 4096, 16, 16.0,
                                 _decoder(4096, 4096, 1024, 14336)),
    "qwen3_8b_q4_0": Workload("qwen3_8b_q4_0", "q4_0", False, 8192, 32, 64.0,
                              _decoder(4096, 4096, 1024, 12288)),
    "qwen3_8b_q8_0": Workload("qwen3_8b_q8_0", "q8_0", False, 8192, 32, 64.0,
                              _decoder(4096, 4096, 1024, 12288)),
}


def linear_flops(M: int, K: int, N: int, r: int) -> int:
    """Algorithmic fwd+bwd flops of one LoRA linear over a frozen base:
    base fwd 2MKN + base dX 2MKN + LoRA 6Mr(K+N)."""
    return 4 * M * K * N + 6 * M * r * (K + N)


def make_linear_inputs(wl: Workload, lin_idx: int, seed: int = 0, layer: int = 0,
                       M: Optional[int] = None, fmt: Optional[str] = None,
                       with_w_f32: bool = False) -> Dict[str, object]:
    """All inputs of one linear: X, dY, A, B (bf16 bits) and the packed base."""
    lin = wl.linears[lin_idx]
    M = wl.M if M is None else M
    fmt = wl.fmt if fmt is None else fmt
    K, N, r = lin.K, lin.N, wl.rank
    a_std = wl.a_std if wl.a_std is not None else 1.0 / math.sqrt(K)
    X = normal_bf16(rng_for(seed, layer, lin_idx, S_X), (M, K), 1.0)
    w = normal_f32(rng_for(seed, layer, lin_idx, S_W), (N, K), wl.w_std)
    A = normal_bf16(rng_for(seed, layer, lin_idx, S_A), (r, K), a_std)
    B = normal_bf16(rng_for(seed, layer, lin_idx, S_B), (N, r), wl.b_std)
    dY = normal_bf16(rng_for(seed, layer, lin_idx, S_DY), (M, N), 1.0)
    out = {"X": X, "A": A, "B": B, "dY": dY, "W": pack(w, fmt, wl.double_quant),
           "M": M, "K": K, "N": N, "rank": r, "alpha": wl.alpha}
    if with_w_f32:
        out["w_f32"] = w
    return out


# ----------------------------------------------------------------------------
# MoE routing for the grouped workload: 4096 tokens, 128 experts, top-8.
# Router logits are Zipf-skewed: logit[t, e] = -(s/tau) ln(rank(e)) + Gumbel,
# with s = 1.1, tau = 4.5, ranks a seeded permutation of 1..E, and the 4
# lowest-ranked experts masked out so that empty experts occur.
# ----------------------------------------------------------------------------
def moe_routing(tokens: int = 4096, experts: int = 128, top_k: int = 8, seed: int = 0,
                zipf_s: float = 1.1, tau: float = 4.5, n_masked: int = 4
                ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Returns (offsets[E+1] int32, token_of_row[R] int32, counts[E] int64)
    with rows sorted by expert (stable by token index)."""
    rng = rng_for(seed, 0, 0, S_ROUTER)
    rank = rng.permutation(experts) + 1
    base = -(zipf_s / tau) * np.log(rank.astype(np.float64))
    g = rng.gumbel(size=(tokens, experts))
    logits = base[None, :] + g
    masked = np.argsort(-rank)[:n_masked]
    logits[:, masked] = -np.inf
    top = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    tok = np.repeat(np.arange(tokens), top_k)
    exp = top.reshape(-1)
    order = np.lexsort((tok, exp))
    counts = np.bincount(exp, minlength=experts)
    offsets = np.zeros(experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return offsets, tok[order].astype(np.int32), counts


@dataclasses.dataclass
class MoEWorkload:
    name: str = "moe_q8_0"
    fmt: str = "q8_0"
    tokens: int = 4096
    experts: int = 128
    top_k: int = 8
    hidden: int = 2048
    inter: int = 768
    rank: int = 16
    alpha: float = 32.0
    w_std: float = 0.02
    b_std: float = 0.01


MOE = MoEWorkload()


def moe_linears(mw: MoEWorkload) -> List[Linear]:
    return [Linear("gate_proj", mw.hidden, mw.inter), Linear("up_proj", mw.hidden, mw.inter),
            Linear("down_proj", mw.inter, mw.hidden)]


def make_moe_linear_inputs(mw: MoEWorkload, lin_idx: int, offsets: np.ndarray, seed: int = 0,
                           experts: Optional[Sequence[int]] = None) -> Dict[str, object]:
    """Per-expert packed bases, stacked adapters and expert-sorted X/dY rows."""
    lin = moe_linears(mw)[lin_idx]
    K, N, r, E = lin.K, lin.N, mw.rank, mw.experts
    R = int(offsets[-1])
    X = normal_bf16(rng_for(seed, 1000, lin_idx, S_X), (R, K), 1.0)
    dY = normal_bf16(rng_for(seed, 1000, lin_idx, S_DY), (R, N), 1.0)
    A = normal_bf16(rng_for(seed, 1000, lin_idx, S_A), (E, r, K), 1.0 / math.sqrt(K))
    B = normal_bf16(rng_for(seed, 1000, lin_idx, S_B), (E, N, r), mw.b_std)
    ws = []
    for e in range(E) if experts is None else experts:
        w = normal_f32(rng_for(seed, 1000 + e, lin_idx, S_W), (N, K), mw.w_std)
        ws.append(pack(w, mw.fmt))
    return {"X": X, "dY": dY, "A": A, "B": B, "W": ws, "K": K, "N": N, "rank": r,
            "alpha": mw.alpha, "offsets": offsets, "R": R}
