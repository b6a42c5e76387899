"""Python binding of the GB300 quantised-base LoRA linear library (libqlora.so).

Argument marshalling only: every computation runs in the CUDA library.  PyTorch
provides device memory and streams.  If the compiled library is missing, every
call raises; there is no fallback path.

    import quantized_base_lora_block_gb300 as q
    w = q.DeviceWeight.from_packed(packed)          # frozen base on the GPU
    Y, T = q.linear_fwd(w, X, A, B, alpha)
    dX, dA, dB = q.linear_bwd(w, X, A, B, T, dY, alpha)
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqlora.so")

FMT = {"bf16": 0, "nf4": 1, "q8_0": 2, "q4_0": 3, "q4_k": 4, "fp8_e4m3": 5, "nvfp4": 6}

STATUS = {
    0: "ok", -1: "invalid argument", -2: "unsupported", -3: "pointer not 16-byte aligned",
    -4: "CUDA error", -5: "device wait timed out", -6: "workspace missing or too small",
    -7: "streaming pool used out of order",
}


QLORA_OK, QLORA_ERR_INVALID, QLORA_ERR_UNSUPPORTED, QLORA_ERR_ALIGN = 0, -1, -2, -3
QLORA_ERR_CUDA, QLORA_ERR_TIMEOUT, QLORA_ERR_WORKSPACE, QLORA_ERR_STATE = -4, -5, -6, -7


class QloraError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({status})")
        self.status = status


class AdapterDesc(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("alpha", ctypes.c_float), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p)]


class WeightDesc(ctypes.Structure):
    _fields_ = [
        ("fmt", ctypes.c_int32),
        ("dq_group", ctypes.c_int32),
        ("N", ctypes.c_int64),
        ("K", ctypes.c_int64),
        ("data", ctypes.c_void_p),
        ("absmax", ctypes.c_void_p),
        ("absmax_q", ctypes.c_void_p),
        ("absmax_scale", ctypes.c_void_p),
        ("absmax_map", ctypes.c_void_p),
        ("tensor_scale", ctypes.c_void_p),
        ("block_scale", ctypes.c_void_p),
        ("absmax_offset", ctypes.c_float),
        ("reserved", ctypes.c_int32),
    ]


_lib: Optional[ctypes.CDLL] = None

# name -> (restype, argtypes)
_P, _I32, _I64, _F32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_WD = ctypes.POINTER(WeightDesc)
_AD = ctypes.POINTER(AdapterDesc)
_PP = ctypes.POINTER(ctypes.c_void_p)
SIGNATURES = {
    "qlora_status_string": (ctypes.c_char_p, [_I32]),
    "qlora_version": (_I32, []),
    "qlora_workspace_bytes": (_SZ, [_WD, _I64, _I32]),
    "dequant_blocks": (_I32, [_WD, _P, _P]),
    "qlora_linear_fwd": (_I32, [_WD, _I64, _I32, _F32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "qlora_linear_bwd": (_I32, [_WD, _I64, _I32, _F32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "qlora_grouped_workspace_bytes": (_SZ, [_WD, _I32, _I64, _I32]),
    "grouped_moe_qlora_fwd": (_I32, [_WD, _I32, _P, _I64, _I32, _F32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "grouped_moe_qlora_bwd": (_I32, [_WD, _I32, _P, _I64, _I32, _F32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                     _P]),
    "qlora_stream_create": (_I32, [_I32, _SZ, ctypes.POINTER(ctypes.c_void_p)]),
    "qlora_stream_prefetch": (_I32, [_P, _I32, _P, _SZ]),
    "qlora_stream_acquire": (_I32, [_P, _I32, _P, ctypes.POINTER(ctypes.c_void_p)]),
    "qlora_stream_release": (_I32, [_P, _I32, _P]),
    "qlora_stream_destroy": (_I32, [_P]),
    "qlora_device_error": (_I32, [_I32]),
    "qlora_last_device_error": (_I32, [_P, _I32]),
    "qlora_selftest_bounded_wait": (_I32, [_I64, _P]),
    "qlora_launch_count": (_I64, []),
    "qlora_linear_fwd_noalloc": (_I32, [_WD, _I64, _I32, _F32, _P, _P, _P, _P, _P, _P]),
    "qlora_stacked_workspace_bytes": (_SZ, [_WD, _I64, _I32, _AD]),
    "qlora_stacked_linear_fwd": (_I32, [_WD, _I64, _I32, _AD, _P, _P, _P, _P, _SZ, _P]),
    "qlora_stacked_linear_bwd": (_I32, [_WD, _I64, _I32, _AD, _P, _P, _P, _P, _PP, _PP, _P, _SZ, _P]),
    "qlora_multi_workspace_bytes": (_SZ, [_WD, _I32, ctypes.POINTER(ctypes.c_int64), _I64, _I32]),
    "qlora_multi_linear_fwd": (_I32, [_WD, _I32, ctypes.POINTER(ctypes.c_int64), _I64, _I32, _F32, _P, _P, _P, _P,
                                      _P, _P, _SZ, _P]),
    "qlora_multi_linear_bwd": (_I32, [_WD, _I32, ctypes.POINTER(ctypes.c_int64), _I64, _I32, _F32, _P, _P, _P, _P,
                                      _P, _P, _P, _P, _P, _SZ, _P]),
    "qlora_noalloc_scratch_bytes": (_SZ, []),
    "qlora_swiglu_workspace_bytes": (_SZ, [_WD, _I64, _I32]),
    "qlora_swiglu_fwd": (_I32, [_WD, _I64, _I32, _F32, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "qlora_swiglu_bwd": (_I32, [_WD, _I64, _I32, _F32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "qlora_forward_workspace_bytes": (_SZ, [_WD, _I64, _I32]),
    "qlora_debug_linear_fwd_f32": (_I32, [_WD, _I64, _I32, _F32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "qlora_debug_linear_bwd_f32": (_I32, [_WD, _I64, _I32, _F32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "qlora_profile_gemm": (_I32, [_I32]),
    "qlora_profile_gemm_read": (_I32, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64),
                                       ctypes.POINTER(ctypes.c_double)]),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqlora.so (built by ``build.py``).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m quantized_base_lora_block_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise QloraError(fn, status)


def _torch():
    import torch

    return torch


def _stream_ptr(stream=None) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


# ---------------------------------------------------------------------------
# host <-> device helpers (torch only as an allocator)
# ---------------------------------------------------------------------------
def bf16_from_bits(bits: np.ndarray, device="cuda"):
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def bits_from_bf16(t) -> np.ndarray:
    torch = _torch()
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _bytes_to_device(a: np.ndarray, device="cuda"):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).to(device)


class DeviceWeight:
    """A frozen base weight resident on the GPU plus its C descriptor."""

    def __init__(self, fmt: str, N: int, K: int, data, absmax=None, absmax_q=None, absmax_scale=None,
                 dq_group: int = 0, absmax_map=None, absmax_offset: float = 0.0, tensor_scale=None,
                 block_scale=None):
        self.fmt, self.N, self.K = fmt, int(N), int(K)
        self.data, self.absmax, self.absmax_q, self.absmax_scale = data, absmax, absmax_q, absmax_scale
        self.absmax_map, self.tensor_scale, self.block_scale = absmax_map, tensor_scale, block_scale
        self.desc = WeightDesc(FMT[fmt], int(dq_group), self.N, self.K, _ptr(data), _ptr(absmax), _ptr(absmax_q),
                               _ptr(absmax_scale), _ptr(absmax_map), _ptr(tensor_scale), _ptr(block_scale),
                               float(absmax_offset), 0)

    @classmethod
    def from_packed(cls, p: Dict, device="cuda") -> "DeviceWeight":
        torch = _torch()

        def f32(key):
            return torch.from_numpy(np.ascontiguousarray(p[key], np.float32).reshape(-1)).to(device)

        data = _bytes_to_device(p["data"], device)
        kw = {}
        if p["fmt"] == "nf4":
            if "absmax" in p:
                kw["absmax"] = f32("absmax")
            else:
                kw["absmax_q"] = torch.from_numpy(np.ascontiguousarray(p["absmax_q"]).view(np.int8)).to(device)
                kw["absmax_scale"] = f32("absmax_scale")
                if p.get("absmax_map") is not None:
                    kw["absmax_map"] = f32("absmax_map")
                    kw["absmax_offset"] = float(p["absmax_offset"])
        if p["fmt"] in ("fp8_e4m3", "nvfp4"):
            kw["tensor_scale"] = f32("tensor_scale")
        if p["fmt"] == "nvfp4":
            kw["block_scale"] = _bytes_to_device(p["block_scale"], device)
        return cls(p["fmt"], p["N"], p["K"], data, dq_group=p.get("dq_group", 0), **kw)

    @classmethod
    def from_pointers(cls, fmt: str, N: int, K: int, data: int, absmax: int = 0, absmax_q: int = 0,
                      absmax_scale: int = 0, dq_group: int = 0, keepalive=None) -> "DeviceWeight":
        """Descriptor over raw device addresses (e.g. a streaming-pool slot)."""
        self = cls.__new__(cls)
        self.fmt, self.N, self.K = fmt, int(N), int(K)
        self.data = self.absmax = self.absmax_q = self.absmax_scale = None
        self._keepalive = keepalive
        self.absmax_map = self.tensor_scale = self.block_scale = None
        self.desc = WeightDesc(FMT[fmt], int(dq_group), self.N, self.K, data or None, absmax or None,
                               absmax_q or None, absmax_scale or None, None, None, None, 0.0, 0)
        return self

    def nbytes(self) -> int:
        n = 0
        for t in (self.data, self.absmax, self.absmax_q, self.absmax_scale, self.absmax_map, self.tensor_scale,
                  self.block_scale):
            if t is not None:
                n += t.numel() * t.element_size()
        return n


# ---------------------------------------------------------------------------
# calls
# ---------------------------------------------------------------------------
def workspace_bytes(w: DeviceWeight, M: int, rank: int) -> int:
    return int(load().qlora_workspace_bytes(ctypes.byref(w.desc), int(M), int(rank)))


def alloc_workspace(nbytes: int, device="cuda"):
    torch = _torch()
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def debug_linear_fwd_f32(w: DeviceWeight, X, A, B, alpha: float, workspace=None, stream=None):
    """The forward with Y returned as the fp32 accumulator values (tests)."""
    torch = _torch()
    M, r = X.shape[0], A.shape[0]
    Y = torch.empty((M, w.N), dtype=torch.float32, device=X.device)
    T = torch.empty((M, r), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(workspace_bytes(w, M, r), X.device)
    st = load().qlora_debug_linear_fwd_f32(ctypes.byref(w.desc), M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B),
                                           _ptr(Y), _ptr(T), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check("qlora_debug_linear_fwd_f32", st)
    return Y, T


def debug_linear_bwd_f32(w: DeviceWeight, X, A, B, T, dY, alpha: float, workspace=None, stream=None):
    """The backward with dX returned as the fp32 accumulator values (tests)."""
    torch = _torch()
    M, r = X.shape[0], A.shape[0]
    dX = torch.empty((M, w.K), dtype=torch.float32, device=X.device)
    dA = torch.empty((r, w.K), dtype=torch.float32, device=X.device)
    dB = torch.empty((w.N, r), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(workspace_bytes(w, M, r), X.device)
    st = load().qlora_debug_linear_bwd_f32(ctypes.byref(w.desc), M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B),
                                           _ptr(T), _ptr(dY), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(workspace),
                                           workspace.numel(), _stream_ptr(stream))
    _check("qlora_debug_linear_bwd_f32", st)
    return dX, dA, dB


def swiglu_workspace_bytes(w: DeviceWeight, M: int, rank: int) -> int:
    return int(load().qlora_swiglu_workspace_bytes(ctypes.byref(w.desc), int(M), int(rank)))


def swiglu_fwd(w: DeviceWeight, X, A, B, alpha: float, H=None, GU=None, T=None, workspace=None, stream=None):
    """Gate / up with SwiGLU over w = [gate rows; up rows]; A [2, r, K], B
    [2I, r].  Returns (H [M, I], GU [M, 2I], T_save [M, 2r])."""
    torch = _torch()
    M, r, I = X.shape[0], A.shape[-2], w.N // 2
    if H is None:
        H = torch.empty((M, I), dtype=torch.bfloat16, device=X.device)
    if GU is None:
        GU = torch.empty((M, 2 * I), dtype=torch.bfloat16, device=X.device)
    if T is None:
        T = torch.empty((M, 2 * r), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(swiglu_workspace_bytes(w, M, r), X.device)
    st = load().qlora_swiglu_fwd(ctypes.byref(w.desc), M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B), _ptr(H),
                                 _ptr(GU), _ptr(T), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check("qlora_swiglu_fwd", st)
    return H, GU, T


def swiglu_bwd(w: DeviceWeight, X, A, B, T, GU, dH, alpha: float, dX=None, dA=None, dB=None, workspace=None,
               stream=None, want_dx: bool = True):
    """Returns (dX [M, K] (summed over gate and up), dA [2, r, K], dB [2I, r])."""
    torch = _torch()
    M, r = X.shape[0], A.shape[-2]
    if dX is None and want_dx:
        dX = torch.empty((M, w.K), dtype=torch.bfloat16, device=X.device)
    if dA is None:
        dA = torch.empty((2, r, w.K), dtype=torch.float32, device=X.device)
    if dB is None:
        dB = torch.empty((w.N, r), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(swiglu_workspace_bytes(w, M, r), X.device)
    st = load().qlora_swiglu_bwd(ctypes.byref(w.desc), M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B), _ptr(T),
                                 _ptr(GU), _ptr(dH), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(workspace),
                                 workspace.numel(), _stream_ptr(stream))
    _check("qlora_swiglu_bwd", st)
    return dX, dA, dB


def dequant_blocks(w: DeviceWeight, out=None, stream=None):
    torch = _torch()
    if out is None:
        out = torch.empty((w.N, w.K), dtype=torch.bfloat16, device=w.data.device)
    _check("dequant_blocks", load().dequant_blocks(ctypes.byref(w.desc), _ptr(out), _stream_ptr(stream)))
    return out


def linear_fwd(w: DeviceWeight, X, A, B, alpha: float, Y=None, T=None, workspace=None, stream=None):
    """Y = X deq(W)^T + (alpha/r) (X A^T) B^T; returns (Y, T_save)."""
    torch = _torch()
    M, r = X.shape[0], A.shape[0]
    if Y is None:
        Y = torch.empty((M, w.N), dtype=torch.bfloat16, device=X.device)
    if T is None:
        T = torch.empty((M, r), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(workspace_bytes(w, M, r), X.device)
    st = load().qlora_linear_fwd(ctypes.byref(w.desc), M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B), _ptr(Y),
                                 _ptr(T), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check("qlora_linear_fwd", st)
    return Y, T


def linear_fwd_noalloc(w: DeviceWeight, X, A, B, alpha: float, Y=None, T=None, stream=None):
    """Forward pass without a workspace argument, for callers that cannot
    allocate device memory: the library uses its own fixed device scratch
    (qlora_noalloc_scratch_bytes() bytes, shared by every such call on the
    device, so calls must not overlap on the GPU).  Y and T are still the
    caller's buffers.  Returns (Y, T_save)."""
    torch = _torch()
    M, r = X.shape[0], A.shape[0]
    if Y is None:
        Y = torch.empty((M, w.N), dtype=torch.bfloat16, device=X.device)
    if T is None:
        T = torch.empty((M, r), dtype=torch.float32, device=X.device)
    st = load().qlora_linear_fwd_noalloc(ctypes.byref(w.desc), M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B),
                                         _ptr(Y), _ptr(T), _stream_ptr(stream))
    _check("qlora_linear_fwd_noalloc", st)
    return Y, T


def linear_bwd(w: DeviceWeight, X, A, B, T, dY, alpha: float, dX=None, dA=None, dB=None, workspace=None,
               stream=None, want_dx: bool = True):
    """Returns (dX, dA, dB); dX is None when want_dx is False."""
    torch = _torch()
    M, r = X.shape[0], A.shape[0]
    if dX is None and want_dx:
        dX = torch.empty((M, w.K), dtype=torch.bfloat16, device=X.device)
    if dA is None:
        dA = torch.empty((r, w.K), dtype=torch.float32, device=X.device)
    if dB is None:
        dB = torch.empty((w.N, r), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(workspace_bytes(w, M, r), X.device)
    st = load().qlora_linear_bwd(ctypes.byref(w.desc), M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B), _ptr(T),
                                 _ptr(dY), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(workspace), workspace.numel(),
                                 _stream_ptr(stream))
    _check("qlora_linear_bwd", st)
    return dX, dA, dB


# ---------------------------------------------------------------------------
# stacked adapters on one base
# ---------------------------------------------------------------------------
def _adapters(As, Bs, alphas):
    n = len(As)
    arr = (AdapterDesc * n)(*[AdapterDesc(int(A.shape[0]), float(al), _ptr(A), _ptr(B))
                              for A, B, al in zip(As, Bs, alphas)])
    return n, arr


def stacked_workspace_bytes(w: DeviceWeight, M: int, As, Bs, alphas) -> int:
    n, arr = _adapters(As, Bs, alphas)
    return int(load().qlora_stacked_workspace_bytes(ctypes.byref(w.desc), int(M), n, arr))


def stacked_linear_fwd(w: DeviceWeight, X, As, Bs, alphas, Y=None, T=None, workspace=None, stream=None):
    """Adapters i = 0.. with A_i [r_i, K], B_i [N, r_i], alpha_i.  Returns (Y, T_save [M, sum r_i])."""
    torch = _torch()
    n, arr = _adapters(As, Bs, alphas)
    M = X.shape[0]
    Q = sum(int(A.shape[0]) for A in As)
    if Y is None:
        Y = torch.empty((M, w.N), dtype=torch.bfloat16, device=X.device)
    if T is None:
        T = torch.empty((M, Q), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(stacked_workspace_bytes(w, M, As, Bs, alphas), X.device)
    st = load().qlora_stacked_linear_fwd(ctypes.byref(w.desc), M, n, arr, _ptr(X), _ptr(Y), _ptr(T), _ptr(workspace),
                                         workspace.numel(), _stream_ptr(stream))
    _check("qlora_stacked_linear_fwd", st)
    return Y, T


def stacked_linear_bwd(w: DeviceWeight, X, As, Bs, alphas, T, dY, trainable=None, dX=None, workspace=None,
                       stream=None, want_dx: bool = True):
    """Returns (dX, [dA_i or None], [dB_i or None]); trainable[i] False leaves
    adapter i without gradient."""
    torch = _torch()
    n, arr = _adapters(As, Bs, alphas)
    M = X.shape[0]
    trainable = [True] * n if trainable is None else list(trainable)
    dAs = [torch.empty((int(A.shape[0]), w.K), dtype=torch.float32, device=X.device) if t else None
           for A, t in zip(As, trainable)]
    dBs = [torch.empty((w.N, int(A.shape[0])), dtype=torch.float32, device=X.device) if t else None
           for A, t in zip(As, trainable)]
    pa = (ctypes.c_void_p * n)(*[_ptr(t) for t in dAs])
    pb = (ctypes.c_void_p * n)(*[_ptr(t) for t in dBs])
    if dX is None and want_dx:
        dX = torch.empty((M, w.K), dtype=torch.bfloat16, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(stacked_workspace_bytes(w, M, As, Bs, alphas), X.device)
    st = load().qlora_stacked_linear_bwd(ctypes.byref(w.desc), M, n, arr, _ptr(X), _ptr(T), _ptr(dY), _ptr(dX), pa, pb,
                                         _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check("qlora_stacked_linear_bwd", st)
    return dX, dAs, dBs


# ---------------------------------------------------------------------------
# fused projections sharing one input
# ---------------------------------------------------------------------------
def _split(n_split: Sequence[int]):
    arr = (ctypes.c_int64 * len(n_split))(*[int(n) for n in n_split])
    return len(n_split), arr


def stack_weights(packed: Sequence[Dict]) -> Dict:
    """Host-side stacking of P packed base weights with the same K into one
    [sum N_p x K] weight in the same format (rows of projection p after those
    of projections < p).  Double-quantised NF4 groups must not span two
    projections (each N_p K / 64 a multiple of the group)."""
    fmt = packed[0]["fmt"]
    K = packed[0]["K"]
    out = {"fmt": fmt, "N": sum(p["N"] for p in packed), "K": K,
           "data": np.concatenate([np.asarray(p["data"]).reshape(-1) for p in packed])}
    for k in ("absmax", "absmax_q", "absmax_scale", "block_scale"):
        if k in packed[0]:
            out[k] = np.concatenate([np.asarray(p[k]).reshape(-1) for p in packed])
    # per-tensor constants must agree to describe the stack with one set
    for k in ("absmax_map", "absmax_offset", "tensor_scale"):
        if packed[0].get(k) is not None:
            v = np.asarray(packed[0][k])
            if not all(np.array_equal(np.asarray(p[k]), v) for p in packed):
                raise ValueError(f"stacked weights need the same {k}")
            out[k] = packed[0][k]
    if "dq_group" in packed[0]:
        g = packed[0]["dq_group"]
        assert all((p["N"] * K // 64) % g == 0 for p in packed), "a quantisation group spans two projections"
        out["dq_group"] = g
    return out


def multi_workspace_bytes(w: DeviceWeight, n_split: Sequence[int], M: int, rank: int) -> int:
    P, arr = _split(n_split)
    return int(load().qlora_multi_workspace_bytes(ctypes.byref(w.desc), P, arr, int(M), int(rank)))


def multi_linear_fwd(w: DeviceWeight, n_split: Sequence[int], X, A, B, alpha: float, Y=None, T=None,
                     workspace=None, stream=None):
    """A [P, r, K], B [N, r].  Returns (Y [M, N], T_save [M, P r])."""
    torch = _torch()
    P, arr = _split(n_split)
    M, r = X.shape[0], A.shape[1]
    if Y is None:
        Y = torch.empty((M, w.N), dtype=torch.bfloat16, device=X.device)
    if T is None:
        T = torch.empty((M, P * r), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(multi_workspace_bytes(w, n_split, M, r), X.device)
    st = load().qlora_multi_linear_fwd(ctypes.byref(w.desc), P, arr, M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B),
                                       _ptr(Y), _ptr(T), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check("qlora_multi_linear_fwd", st)
    return Y, T


def multi_linear_bwd(w: DeviceWeight, n_split: Sequence[int], X, A, B, T, dY, alpha: float, dX=None, dA=None,
                     dB=None, workspace=None, stream=None, want_dx: bool = True):
    """Returns (dX summed over projections, dA [P, r, K], dB [N, r])."""
    torch = _torch()
    P, arr = _split(n_split)
    M, r = X.shape[0], A.shape[1]
    if dX is None and want_dx:
        dX = torch.empty((M, w.K), dtype=torch.bfloat16, device=X.device)
    if dA is None:
        dA = torch.empty((P, r, w.K), dtype=torch.float32, device=X.device)
    if dB is None:
        dB = torch.empty((w.N, r), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(multi_workspace_bytes(w, n_split, M, r), X.device)
    st = load().qlora_multi_linear_bwd(ctypes.byref(w.desc), P, arr, M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B),
                                       _ptr(T), _ptr(dY), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(workspace),
                                       workspace.numel(), _stream_ptr(stream))
    _check("qlora_multi_linear_bwd", st)
    return dX, dA, dB


# ---------------------------------------------------------------------------
# grouped (mixture-of-experts)
# ---------------------------------------------------------------------------
def _grouped_descs(weights: Sequence[DeviceWeight]):
    E = len(weights)
    return E, (WeightDesc * E)(*[w.desc for w in weights])


def device_offsets(offsets, device="cuda"):
    """Expert row offsets [E+1] as a device int32 tensor (the grouped calls
    read them on the device only)."""
    torch = _torch()
    if isinstance(offsets, torch.Tensor) and offsets.is_cuda:
        if offsets.dtype != torch.int32 or not offsets.is_contiguous():
            raise ValueError("device offsets must be a contiguous int32 tensor")
        return offsets
    return torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.int32)).to(device)


def _offsets_for_call(offsets, X, E, stream):
    off = device_offsets(offsets, X.device)
    if off.numel() != E + 1:
        raise ValueError(f"offsets must have E + 1 = {E + 1} entries, got {off.numel()}")
    if stream is not None and off is not offsets:
        off.record_stream(stream)  # a copy made here stays alive until the call's work ran
    return off


def grouped_workspace_bytes(weights: Sequence[DeviceWeight], M_total: int, rank: int) -> int:
    E, descs = _grouped_descs(weights)
    return int(load().qlora_grouped_workspace_bytes(descs, E, int(M_total), int(rank)))


def grouped_fwd(weights: Sequence[DeviceWeight], offsets, X, A, B, alpha: float, Y=None, T=None, workspace=None,
                stream=None):
    """Rows of X [M_total, K] sorted by expert; offsets [E+1] (a device int32
    tensor, or host values copied to the device); A [E, r, K], B [E, N, r].
    Returns (Y, T_save)."""
    torch = _torch()
    E, descs = _grouped_descs(weights)
    M = int(X.shape[0])
    off = _offsets_for_call(offsets, X, E, stream)
    r, N = A.shape[1], weights[0].N
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    if T is None:
        T = torch.empty((M, r), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(grouped_workspace_bytes(weights, M, r), X.device)
    st = load().grouped_moe_qlora_fwd(descs, E, _ptr(off), M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B), _ptr(Y),
                                      _ptr(T), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check("grouped_moe_qlora_fwd", st)
    return Y, T


def grouped_bwd(weights: Sequence[DeviceWeight], offsets, X, A, B, T, dY, alpha: float, dX=None, dA=None, dB=None,
                workspace=None, stream=None, want_dx: bool = True):
    """Returns (dX, dA [E, r, K], dB [E, N, r])."""
    torch = _torch()
    E, descs = _grouped_descs(weights)
    M = int(X.shape[0])
    off = _offsets_for_call(offsets, X, E, stream)
    r, N, K = A.shape[1], weights[0].N, weights[0].K
    if dX is None and want_dx:
        dX = torch.empty((M, K), dtype=torch.bfloat16, device=X.device)
    if dA is None:
        dA = torch.empty((E, r, K), dtype=torch.float32, device=X.device)
    if dB is None:
        dB = torch.empty((E, N, r), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(grouped_workspace_bytes(weights, M, r), X.device)
    st = load().grouped_moe_qlora_bwd(descs, E, _ptr(off), M, r, float(alpha), _ptr(X), _ptr(A), _ptr(B), _ptr(T),
                                      _ptr(dY), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(workspace), workspace.numel(),
                                      _stream_ptr(stream))
    _check("grouped_moe_qlora_bwd", st)
    return dX, dA, dB


def upload_experts(weights: Sequence[Dict], device="cuda") -> List[DeviceWeight]:
    """Expert bases with their bytes back to back in one device array
    [E][N][row bytes] (grouped calls read such a stack through one 3-D tensor
    map: required for bf16 bases, the fast path for quantised ones); each
    expert's other arrays (absmax, scales) are uploaded on their own.
    Returns per-expert descriptors over views of the stack."""
    big = _bytes_to_device(np.concatenate([np.ascontiguousarray(w["data"]).view(np.uint8).reshape(-1)
                                           for w in weights]), device)
    per = big.numel() // len(weights)
    out = []
    for e, w in enumerate(weights):
        one = DeviceWeight.from_packed(dict(w, data=np.zeros(16, np.uint8)), device)
        one.data = big[e * per:(e + 1) * per]
        one.desc.data = one.data.data_ptr()
        out.append(one)
    out[0]._stack = big
    return out


def device_error(clear: bool = True) -> int:
    return int(load().qlora_device_error(1 if clear else 0))


def last_device_error(stream=None, clear: bool = True) -> int:
    """The device error word as of the end of `stream`'s enqueued work (waits
    for that stream only)."""
    return int(load().qlora_last_device_error(_stream_ptr(stream), 1 if clear else 0))


def selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Launch the diagnostic wait that runs out after limit_ns (see qlora.h)."""
    _check("qlora_selftest_bounded_wait", load().qlora_selftest_bounded_wait(int(limit_ns), _stream_ptr(stream)))


def launch_count() -> int:
    return int(load().qlora_launch_count())


def profile_gemm(enable: bool) -> None:
    _check("qlora_profile_gemm", load().qlora_profile_gemm(1 if enable else 0))


def profile_gemm_read() -> Tuple[float, int, float]:
    """(summed device ms, launches, summed algorithmic flops) of the fused GEMM."""
    ms, n, fl = ctypes.c_double(), ctypes.c_int64(), ctypes.c_double()
    _check("qlora_profile_gemm_read", load().qlora_profile_gemm_read(ctypes.byref(ms), ctypes.byref(n),
                                                                     ctypes.byref(fl)))
    return ms.value, n.value, fl.value


# ---------------------------------------------------------------------------
# layer streaming
# ---------------------------------------------------------------------------
def pack_weight_blob(p: Dict) -> Tuple[np.ndarray, Dict[str, int]]:
    """One contiguous byte blob per packed base weight (sections 256-byte
    aligned): the unit the streaming pool copies.  Returns (blob, offsets)."""
    parts = [("data", np.ascontiguousarray(p["data"]).view(np.uint8).reshape(-1))]
    for k in ("absmax", "absmax_q", "absmax_scale"):
        if k in p and p[k] is not None:
            parts.append((k, np.ascontiguousarray(p[k]).view(np.uint8).reshape(-1)))
    offs, o = {}, 0
    for k, a in parts:
        offs[k] = o
        o = (o + a.nbytes + 255) // 256 * 256
    blob = np.zeros(o, dtype=np.uint8)
    for k, a in parts:
        blob[offs[k]:offs[k] + a.nbytes] = a
    return blob, offs


def weight_in_slot(p: Dict, offs: Dict[str, int], base: int) -> DeviceWeight:
    """Descriptor of a packed weight whose blob sits at device address base."""
    g = lambda k: (base + offs[k]) if k in offs else 0  # noqa: E731
    return DeviceWeight.from_pointers(p["fmt"], p["N"], p["K"], g("data"), g("absmax"), g("absmax_q"),
                                      g("absmax_scale"), p.get("dq_group", 0))
class LayerStream:
    """Pool of device slots fed from pinned host memory one layer ahead."""

    def __init__(self, slots: int, slot_bytes: int):
        h = ctypes.c_void_p()
        _check("qlora_stream_create", load().qlora_stream_create(int(slots), int(slot_bytes), ctypes.byref(h)))
        self.h = h

    def prefetch(self, layer: int, host_pinned) -> None:
        nbytes = host_pinned.numel() * host_pinned.element_size()
        _check("qlora_stream_prefetch", load().qlora_stream_prefetch(self.h, int(layer), _ptr(host_pinned), nbytes))

    def acquire(self, layer: int, stream=None) -> int:
        p = ctypes.c_void_p()
        _check("qlora_stream_acquire",
               load().qlora_stream_acquire(self.h, int(layer), _stream_ptr(stream), ctypes.byref(p)))
        return int(p.value)

    def release(self, layer: int, stream=None) -> None:
        _check("qlora_stream_release", load().qlora_stream_release(self.h, int(layer), _stream_ptr(stream)))

    def close(self) -> None:
        if self.h is not None and self.h.value:
            _check("qlora_stream_destroy", load().qlora_stream_destroy(self.h))
        self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
