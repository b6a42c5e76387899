"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every
entry point declared in include/qlora.h, and rejects invalid arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import quantized_base_lora_block_gb300 as q
from quantized_base_lora_block_gb300 import build as qbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "qlora.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(", text, re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return q.load()


def test_header_declares_the_api():
    names = header_functions()
    for n in ("dequant_blocks", "qlora_linear_fwd", "qlora_linear_bwd", "grouped_moe_qlora_fwd",
              "grouped_moe_qlora_bwd", "qlora_stream_create", "qlora_workspace_bytes"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in header_functions():
        assert hasattr(lib, n), n
        assert n in q.SIGNATURES, n


def test_status_strings(lib):
    for s in range(-7, 1):
        assert lib.qlora_status_string(s).decode() == q.STATUS[s]
    assert lib.qlora_version() == 200


def _desc(fmt="nf4", N=256, K=256, data=0x1000, absmax=0x2000):
    return q.WeightDesc(q.FMT[fmt], 0, N, K, data, absmax, None, None)


def test_validation_rejects_before_any_launch(lib):
    d = _desc()
    bufs = [0x10000 * (i + 1) for i in range(8)]
    ws = 1 << 30
    f = lib.qlora_linear_fwd
    # bad rank (not a multiple of 8 / too large / zero)
    for r in (0, 7, 12, 72):
        assert f(ctypes.byref(d), 64, r, 16.0, *bufs[:5], bufs[5], ws, None) == -1
    # misaligned activation pointer
    assert f(ctypes.byref(d), 64, 8, 16.0, bufs[0] + 2, *bufs[1:5], bufs[5], ws, None) == -3
    # N or K not a multiple of 64
    for bad in (_desc(N=200), _desc(K=96), _desc(N=0)):
        assert f(ctypes.byref(bad), 64, 8, 16.0, *bufs[:5], bufs[5], ws, None) == -1
    # NF4 without any absmax
    nd = q.WeightDesc(q.FMT["nf4"], 0, 256, 256, 0x1000, None, None, None)
    assert f(ctypes.byref(nd), 64, 8, 16.0, *bufs[:5], bufs[5], ws, None) == -1
    # unknown format
    bf = q.WeightDesc(9, 0, 256, 256, 0x1000, None, None, None)
    assert f(ctypes.byref(bf), 64, 8, 16.0, *bufs[:5], bufs[5], ws, None) == -1
    # workspace too small
    assert f(ctypes.byref(d), 64, 8, 16.0, *bufs[:5], bufs[5], 16, None) == -6
    # non-finite alpha
    assert f(ctypes.byref(d), 64, 8, float("nan"), *bufs[:5], bufs[5], ws, None) == -1
    # M == 0 is a no-op
    assert f(ctypes.byref(d), 0, 8, 16.0, *bufs[:5], bufs[5], ws, None) == 0
    # backward needs dA and dB
    b = lib.qlora_linear_bwd
    assert b(ctypes.byref(d), 64, 8, 16.0, *bufs[:5], bufs[5], None, None, bufs[6], ws, None) == -1


def test_descriptor_fields_of_each_format_checked(lib):
    """Per-format descriptor fields: required ones present and aligned,
    fields of other formats NULL, reserved zero (all checked before any
    launch; the pointers here are never dereferenced)."""
    bufs = [0x10000 * (i + 1) for i in range(8)]
    f = lib.qlora_linear_fwd

    def call(d):
        return f(ctypes.byref(d), 64, 8, 16.0, *bufs[:5], bufs[5], 1 << 30, None)

    def desc(fmt, K=256, **kw):
        d = q.WeightDesc(q.FMT[fmt], kw.pop("dq_group", 0), 256, K, 0x1000)
        for k, v in kw.items():
            setattr(d, k, v)
        return d

    # FP8 / NVFP4 need their scales
    assert call(desc("fp8_e4m3")) == -1
    assert call(desc("nvfp4", tensor_scale=0x3000)) == -1
    assert call(desc("fp8_e4m3", tensor_scale=0x3002)) == -3
    assert call(desc("nvfp4", tensor_scale=0x3000, block_scale=0x4008)) == -3
    # scales of another format
    assert call(desc("q8_0", tensor_scale=0x3000)) == -1
    assert call(desc("fp8_e4m3", tensor_scale=0x3000, block_scale=0x4000)) == -1
    assert call(desc("q4_0", absmax=0x2000)) == -1
    # Q4_K super-blocks need K % 256 == 0
    assert call(desc("q4_k", K=192)) == -1
    # the map variant of NF4 needs a finite offset; reserved must stay 0
    nan_off = desc("nf4", absmax_q=0x2000, absmax_scale=0x3000, absmax_map=0x4000, dq_group=256,
                   absmax_offset=float("nan"))
    assert call(nan_off) == -1
    assert call(desc("q8_0", reserved=1)) == -1
    # workspace queries agree (0 on an invalid descriptor)
    assert lib.qlora_workspace_bytes(ctypes.byref(desc("q4_k", K=192)), 64, 8) == 0
    assert lib.qlora_workspace_bytes(ctypes.byref(desc("nvfp4", tensor_scale=0x3000, block_scale=0x4000)),
                                     64, 8) > 0


def test_workspace_size_is_deterministic(lib):
    d = _desc(N=14336, K=4096)
    a = lib.qlora_workspace_bytes(ctypes.byref(d), 4096, 16)
    b = lib.qlora_workspace_bytes(ctypes.byref(d), 4096, 16)
    assert a == b and a > 4096 * 16 * 2
    assert lib.qlora_workspace_bytes(ctypes.byref(d), 4096, 7) == 0


def test_stream_api_rejects_bad_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.qlora_stream_create(0, 1024, ctypes.byref(h)) == -1
    assert lib.qlora_stream_create(2, 0, ctypes.byref(h)) == -1
    assert lib.qlora_stream_prefetch(None, 0, 0x1000, 16) == -1
    assert lib.qlora_stream_release(None, 0, None) == -1
    assert lib.qlora_stream_destroy(None) == -1
