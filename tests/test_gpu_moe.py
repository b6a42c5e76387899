"""grouped_moe_qlora_fwd / _bwd (rows sorted by expert, offsets in device
memory) against the oracle's per-expert loop; empty experts must get exactly
zero adapter gradients; offsets that do not partition the rows are reported
through the device error word."""
import numpy as np
import pytest

import oracle
import qlora_synth as syn
from gpu_helpers import check_bf16, check_f32

pytestmark = pytest.mark.gpu


def _moe_inputs(counts, K, N, r, fmt, seed=0, alpha=None):
    E = len(counts)
    off = np.zeros(E + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    R = int(off[-1])
    rng = lambda s: syn.rng_for(seed, 77, 0, s)  # noqa: E731
    X = syn.normal_bf16(rng(syn.S_X), (R, K), 1.0)
    dY = syn.normal_bf16(rng(syn.S_DY), (R, N), 1.0)
    A = syn.normal_bf16(rng(syn.S_A), (E, r, K), 1.0 / np.sqrt(K))
    B = syn.normal_bf16(rng(syn.S_B), (E, N, r), 0.01)
    W = [syn.pack(syn.normal_f32(syn.rng_for(seed, 78 + e, 0, syn.S_W), (N, K), 0.02), fmt,
                  double_quant=(fmt in ("nf4", "nf4_dqmap"))) for e in range(E)]
    return {"X": X, "dY": dY, "A": A, "B": B, "W": W, "off": off, "alpha": float(alpha or 2 * r), "r": r}


def _run(lib, d, stacked=True):
    """stacked: expert bases back to back in one array (the tensor-map path);
    else each expert uploaded on its own (per-thread loads; bf16 bases must
    be stacked)."""
    if stacked or d["W"][0]["fmt"] == "bf16":
        ws = lib.upload_experts(d["W"])
    else:
        ws = [lib.DeviceWeight.from_packed(w) for w in d["W"]]
    X, dY = lib.bf16_from_bits(d["X"]), lib.bf16_from_bits(d["dY"])
    A, B = lib.bf16_from_bits(d["A"]), lib.bf16_from_bits(d["B"])
    off = lib.device_offsets(d["off"])  # device int32 [E+1], as a router leaves them
    Y, T = lib.grouped_fwd(ws, off, X, A, B, d["alpha"])
    dX, dA, dB = lib.grouped_bwd(ws, off, X, A, B, T, dY, d["alpha"])
    assert lib.last_device_error() == 0
    return {"Y": lib.bits_from_bf16(Y), "T": T.cpu().numpy(), "dX": lib.bits_from_bf16(dX),
            "dA": dA.cpu().numpy(), "dB": dB.cpu().numpy()}


def _oracle(d):
    Wds = [oracle.dequant(w) for w in d["W"]]
    A = oracle.bf16_bits_to_f64(d["A"])
    B = oracle.bf16_bits_to_f64(d["B"])
    Y, T = oracle.grouped_fwd(d["X"], Wds, A, B, d["off"], d["alpha"])
    g = oracle.grouped_bwd(d["X"], Wds, A, B, d["dY"], d["off"], d["alpha"])
    return {"Y": Y, "T": T, **g}


def _check(d, got, ref):
    off = d["off"]
    check_bf16(got["Y"], ref["Y"], "Y")
    check_f32(got["T"], ref["T"], "T")
    check_bf16(got["dX"], ref["dX"], "dX")
    for e in range(len(off) - 1):
        if off[e + 1] == off[e]:
            assert np.all(got["dA"][e] == 0) and np.all(got["dB"][e] == 0), f"expert {e} has no rows"
        else:
            check_f32(got["dA"][e], ref["dA"][e], f"dA[{e}]")
            check_f32(got["dB"][e], ref["dB"][e], f"dB[{e}]")


@pytest.mark.parametrize("stacked", [True, False], ids=["stacked", "separate"])
@pytest.mark.parametrize("fmt", ["q8_0", "nf4", "q4_0", "bf16", "q4_k", "fp8_e4m3", "nvfp4", "nf4_dqmap"])
def test_grouped_mixed_counts(lib, fmt, stacked):
    if fmt == "bf16" and not stacked:
        pytest.skip("bf16 expert bases are always stacked")
    d = _moe_inputs([0, 5, 130, 1, 0, 260, 64], K=256, N=320, r=16, fmt=fmt, seed=3)
    _check(d, _run(lib, d, stacked), _oracle(d))


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0", "nf4", "q4_k"])
def test_grouped_wide_and_ragged(lib, fmt):
    """More column blocks than one (N = 1280 forward, K = 768 dX), K whose
    Q8_0 / Q4_0 rows are not a multiple of 16 bytes (raw ring off) where
    the format allows it, and an expert spanning several row tiles."""
    K = 768 if fmt == "q4_k" else 832
    d = _moe_inputs([700, 3, 0, 300], K=K, N=1280, r=8, fmt=fmt, seed=12)
    _check(d, _run(lib, d), _oracle(d))


def test_grouped_all_experts_empty(lib):
    import torch

    d = _moe_inputs([0, 0, 0], K=128, N=128, r=8, fmt="q8_0")
    ws = [lib.DeviceWeight.from_packed(w) for w in d["W"]]
    X = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    dY = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    A, B = lib.bf16_from_bits(d["A"]), lib.bf16_from_bits(d["B"])
    T = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    dA = torch.full((3, 8, 128), 7.0, device="cuda")
    dB = torch.full((3, 128, 8), 7.0, device="cuda")
    lib.grouped_bwd(ws, d["off"], X, A, B, T, dY, d["alpha"], dA=dA, dB=dB, want_dx=False)
    torch.cuda.synchronize()
    assert float(dA.abs().max()) == 0.0 and float(dB.abs().max()) == 0.0


def _close_ulps(a_bits, b_bits, name, ulps=2):
    """Elementwise |a - b| <= ulps bf16 ulps of |a| (the two calls round the
    same sums after different split / tile orders)."""
    a = oracle.bf16_bits_to_f64(a_bits)
    b = oracle.bf16_bits_to_f64(b_bits.reshape(a_bits.shape))
    tol = ulps * np.maximum(np.abs(a), 1e-30) * 2.0 ** -7
    assert np.all(np.abs(a - b) <= tol), f"{name}: max diff {np.abs(a - b).max():.3g}"


@pytest.mark.parametrize("rows", [100, 700])
def test_one_expert_equals_dense(lib, rows):
    """E = 1 computes the dense layer over the same rows (different tile
    shapes and split orders, so compared within rounding)."""
    d = _moe_inputs([rows], K=256, N=512, r=16, fmt="nf4", seed=5)
    got = _run(lib, d)
    inp = {"X": d["X"], "A": d["A"][0], "B": d["B"][0], "dY": d["dY"], "W": d["W"][0], "alpha": d["alpha"]}
    from gpu_helpers import run_layer

    dense = run_layer(inp)
    _close_ulps(got["Y"], dense["Y"], "Y")
    _close_ulps(got["dX"], dense["dX"], "dX")
    check_f32(got["T"], dense["T"].astype(np.float64), "T vs dense", rel=1e-5)
    check_f32(got["dA"][0], dense["dA"].astype(np.float64), "dA vs dense", rel=1e-5)
    check_f32(got["dB"][0], dense["dB"].astype(np.float64), "dB vs dense", rel=1e-5)


@pytest.mark.parametrize("bad", [[0, 40, 30, 100], [0, 40, 70, 90], [5, 40, 70, 100], [0, 40, 70, 130]])
def test_invalid_offsets_reported(lib, bad):
    """Offsets that are not a partition of [0, M_total) (decreasing, short,
    not starting at 0, past the end) make both calls do no GEMM work and
    record QLORA_ERR_INVALID in the device error word; the offsets are never
    read on the host."""
    import torch

    d = _moe_inputs([40, 30, 30], K=128, N=256, r=8, fmt="q8_0", seed=9)
    ws = [lib.DeviceWeight.from_packed(w) for w in d["W"]]
    X, dY = lib.bf16_from_bits(d["X"]), lib.bf16_from_bits(d["dY"])
    A, B = lib.bf16_from_bits(d["A"]), lib.bf16_from_bits(d["B"])
    off = torch.tensor(bad, dtype=torch.int32, device="cuda")
    assert lib.last_device_error() == 0
    Y = torch.zeros((100, 256), dtype=torch.bfloat16, device="cuda")
    _, T = lib.grouped_fwd(ws, off, X, A, B, d["alpha"], Y=Y)
    assert lib.last_device_error() == lib.QLORA_ERR_INVALID
    assert float(Y.float().abs().max()) == 0.0  # no tile was scheduled
    dX = torch.zeros((100, 128), dtype=torch.bfloat16, device="cuda")
    T.zero_()
    lib.grouped_bwd(ws, off, X, A, B, T, dY, d["alpha"], dX=dX)
    assert lib.last_device_error() == lib.QLORA_ERR_INVALID
    assert float(dX.float().abs().max()) == 0.0
    assert lib.last_device_error() == 0  # cleared by the read


def test_offsets_written_on_device(lib):
    """Offsets produced by a device computation (a prefix sum of per-expert
    counts) feed the call directly."""
    import torch

    counts = [3, 0, 77, 200, 1]
    d = _moe_inputs(counts, K=192, N=256, r=24, fmt="q4_0", seed=11)
    c = torch.tensor(counts, dtype=torch.int32, device="cuda")
    off = torch.zeros(len(counts) + 1, dtype=torch.int32, device="cuda")
    off[1:] = torch.cumsum(c, 0).to(torch.int32)
    ws = [lib.DeviceWeight.from_packed(w) for w in d["W"]]
    X, dY = lib.bf16_from_bits(d["X"]), lib.bf16_from_bits(d["dY"])
    A, B = lib.bf16_from_bits(d["A"]), lib.bf16_from_bits(d["B"])
    Y, T = lib.grouped_fwd(ws, off, X, A, B, d["alpha"])
    dX, dA, dB = lib.grouped_bwd(ws, off, X, A, B, T, dY, d["alpha"])
    assert lib.last_device_error() == 0
    got = {"Y": lib.bits_from_bf16(Y), "T": T.cpu().numpy(), "dX": lib.bits_from_bf16(dX),
           "dA": dA.cpu().numpy(), "dB": dB.cpu().numpy()}
    _check(d, got, _oracle(d))


@pytest.mark.slow
@pytest.mark.parametrize("lin", [0, 2], ids=["gate_2048x768", "down_768x2048"])
def test_moe_workload(lib, lin):
    """128 experts, top-8 Zipf-skewed routing of 4096 tokens (32,768 rows,
    4 experts empty), Q8_0 bases, rank 16: the gate projection 2048 -> 768
    and the down projection 768 -> 2048, at full size."""
    mw = syn.MOE
    off, _, counts = syn.moe_routing()
    assert counts.min() == 0
    d = syn.make_moe_linear_inputs(mw, lin, off, seed=0)
    dd = {"X": d["X"], "dY": d["dY"], "A": d["A"], "B": d["B"], "W": d["W"], "off": off, "alpha": d["alpha"],
          "r": d["rank"]}
    _check(dd, _run(lib, dd), _oracle(dd))


def test_largest_expert_count(lib):
    """256 experts (the limit), most with a handful of rows, some empty; 257
    experts are rejected before anything is launched."""
    import ctypes

    rng = np.random.default_rng(21)
    counts = rng.integers(0, 12, size=256)
    counts[::17] = 0
    d = _moe_inputs(list(counts), K=128, N=192, r=8, fmt="q4_0", seed=21)
    _check(d, _run(lib, d), _oracle(d))
    ws = [lib.DeviceWeight.from_packed(w) for w in d["W"]]
    descs = (lib.WeightDesc * 257)(*([w.desc for w in ws] + [ws[0].desc]))
    assert lib.load().qlora_grouped_workspace_bytes(descs, 257, int(counts.sum()), 8) == 0
