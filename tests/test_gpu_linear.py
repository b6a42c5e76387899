"""qlora_linear_fwd / qlora_linear_bwd on the GPU against the fp64 oracle.

Tolerance: max|err| <= 1e-2 * RMS(ref) per tensor for the fp32 gradients dA,
dB; for the bf16 outputs Y, dX, T additionally half a bf16 ulp of |ref|
elementwise (a bf16 output cannot be closer than its own rounding).
"""
import numpy as np
import pytest

import oracle
import qlora_synth as syn
from gpu_helpers import check_bf16, check_f32, oracle_layer, run_layer, sample_rows

pytestmark = pytest.mark.gpu


def make(M, K, N, r, fmt, dq=False, alpha=None, seed=0, b_std=0.01):
    wl = syn.Workload("t", fmt, dq, M, r, float(alpha if alpha is not None else 2 * r),
                      [syn.Linear("t", K, N)], b_std=b_std)
    return syn.make_linear_inputs(wl, 0, seed=seed)


def check_all(inp, got, ref):
    check_bf16(got["Y"], ref["Y"], "Y")
    check_f32(got["T"], ref["T"], "T")
    check_bf16(got["dX"], ref["dX"], "dX")
    check_f32(got["dA"], ref["dA"], "dA")
    check_f32(got["dB"], ref["dB"], "dB")


def test_tiny_config_nf4(lib):
    """64 x 256 -> 256, NF4 bs64 fp32 absmax, rank 8, alpha 16, seed 0."""
    inp = syn.make_linear_inputs(syn.WORKLOADS["tiny_nf4"], 0, seed=0)
    check_all(inp, run_layer(inp), oracle_layer(inp))


SHAPES = [
    # M, K, N, r
    (64, 256, 256, 8),
    (200, 512, 320, 16),    # ragged M, N not a multiple of the 256-wide tile
    (1, 128, 64, 32),       # a single row
    (384, 1024, 768, 64),   # largest rank
    (130, 192, 448, 24),    # odd multiple-of-8 rank, ragged everything
    (257, 640, 512, 16),    # one row past a tile
]


@pytest.mark.parametrize("fmt,dq", [("bf16", False), ("nf4", False), ("nf4", True), ("q8_0", False),
                                    ("q4_0", False), ("fp8_e4m3", False), ("nvfp4", False),
                                    ("nf4_dqmap", False)])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_formats_and_shapes(lib, fmt, dq, shape):
    M, K, N, r = shape
    inp = make(M, K, N, r, fmt, dq, seed=M + K + N + r)
    check_all(inp, run_layer(inp), oracle_layer(inp))


# Q4_K needs K % 256 == 0
Q4_K_SHAPES = [(64, 256, 256, 8), (200, 512, 320, 16), (1, 256, 64, 32), (300, 1024, 768, 64),
               (130, 768, 448, 24), (600, 512, 1280, 16)]


@pytest.mark.parametrize("shape", Q4_K_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_q4_k_shapes(lib, shape):
    M, K, N, r = shape
    inp = make(M, K, N, r, "q4_k", False, seed=M + K + N + r)
    check_all(inp, run_layer(inp), oracle_layer(inp))


# Shapes whose launches take the 512 x 256 pair tiles (the NF4 code-byte ring
# and the forward absmax cache): forward with a ragged last column block
# (10048 = 39 x 256 + 64, one CTA of the pair without weight rows), forward
# with whole blocks, and dX with the absmax / group-scale ring (groups
# spanning weight rows); all ragged in M.  The last case also has a long
# reduction (K = 14336, as the down projection) with a ragged column block.
@pytest.mark.parametrize("shape", [(600, 1024, 10048, 16), (600, 1024, 9728, 16), (600, 10240, 1088, 16),
                                   (1100, 14336, 4160, 16)],
                         ids=["fwd_ragged", "fwd", "dx", "fwd_long_ragged"])
def test_nf4dq_wide_tiles(lib, shape):
    M, K, N, r = shape
    inp = make(M, K, N, r, "nf4", True, seed=M + K + N)
    check_all(inp, run_layer(inp), oracle_layer(inp))


def test_b_zero_gives_base_product_and_zero_dA(lib):
    inp = make(160, 512, 256, 16, "nf4", b_std=0.0)
    assert np.all(syn.bf16_bits_to_f32(inp["B"]) == 0.0)  # +0 and -0 entries
    got = run_layer(inp)
    ref = oracle_layer(inp)
    Wd = oracle.dequant(inp["W"])
    base = oracle.bf16_bits_to_f64(inp["X"]) @ Wd.T
    assert np.array_equal(ref["Y"], base)
    check_bf16(got["Y"], base, "Y(B=0)")
    assert np.all(got["dA"] == 0.0)
    check_f32(got["dB"], ref["dB"], "dB")


def test_alpha_scales_adapter_terms(lib):
    a = make(128, 256, 256, 16, "q8_0", alpha=16.0, seed=5)
    b = dict(a)
    b["alpha"] = 32.0
    ga, gb = run_layer(a), run_layer(b)
    check_f32(gb["dA"], 2 * ga["dA"].astype(np.float64), "dA scale", rel=2e-2)
    check_f32(gb["dB"], 2 * ga["dB"].astype(np.float64), "dB scale", rel=2e-2)


def test_bitwise_deterministic(lib):
    inp = make(300, 512, 512, 16, "nf4", dq=True, seed=7)
    g1, g2 = run_layer(inp), run_layer(inp)
    for k in g1:
        assert np.array_equal(g1[k], g2[k]), k


def test_backward_without_dx(lib):
    inp = make(96, 256, 320, 16, "q4_0", seed=9)
    got = run_layer(inp, want_dx=False)
    ref = oracle_layer(inp)
    check_f32(got["dA"], ref["dA"], "dA")
    check_f32(got["dB"], ref["dB"], "dB")


@pytest.mark.slow
@pytest.mark.parametrize("wl_name,lin", [("llama31_8b_nf4dq", 4), ("llama31_8b_nf4dq", 6), ("llama31_8b_nf4dq", 1),
                                         ("qwen3_0p6b_bf16", 0), ("qwen3_8b_q4_0", 3), ("qwen3_8b_q8_0", 6)])
def test_full_size_layer_sampled_rows(lib, wl_name, lin):
    """Full-size linears of the benchmark layers: Y and dX on sampled rows,
    T, dA and dB in full."""
    wl = syn.WORKLOADS[wl_name]
    inp = syn.make_linear_inputs(wl, lin, seed=0)
    got = run_layer(inp)
    rows = sample_rows(inp["M"], 256)
    ref = oracle_layer(inp, rows=rows)
    M = inp["M"]
    check_bf16(got["Y"].reshape(M, -1)[rows], ref["Y"], "Y")
    check_bf16(got["dX"].reshape(M, -1)[rows], ref["dX"], "dX")
    check_f32(got["T"], ref["T_all"], "T")
    check_f32(got["dA"], ref["dA"], "dA")
    check_f32(got["dB"], ref["dB"], "dB")


@pytest.mark.parametrize("shape", [(128, 64, 64, 8), (129, 64, 64, 8), (513, 128, 192, 8), (1, 64, 64, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_edge_shapes(lib, shape):
    """Smallest K and N (one decode line, one 64-wide chunk), the last size of
    the one-CTA path (128 rows) and the first of the pair path (129), one row
    past a 512-row pair tile, a single row at the largest rank."""
    M, K, N, r = shape
    inp = make(M, K, N, r, "nf4", True, seed=M + K + N + r)
    check_all(inp, run_layer(inp), oracle_layer(inp))


def test_zero_rows(lib):
    """M = 0: the forward writes nothing; the backward sets dA and dB to zero."""
    import torch

    inp = make(64, 256, 320, 16, "q8_0", seed=3)
    d = {k: lib.bf16_from_bits(inp[k]) for k in ("A", "B")}
    w = lib.DeviceWeight.from_packed(inp["W"])
    X = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    dY = torch.empty((0, 320), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((0, 320), dtype=torch.bfloat16, device="cuda")
    T = torch.empty((0, 16), dtype=torch.float32, device="cuda")
    lib.linear_fwd(w, X, d["A"], d["B"], inp["alpha"], Y=Y, T=T)
    dA = torch.full((16, 256), 5.0, device="cuda")
    dB = torch.full((320, 16), 5.0, device="cuda")
    lib.linear_bwd(w, X, d["A"], d["B"], T, dY, inp["alpha"], dA=dA, dB=dB, want_dx=False)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert float(dA.abs().max()) == 0.0 and float(dB.abs().max()) == 0.0
