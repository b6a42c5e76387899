"""Fused projections sharing one input (qlora_multi_linear_fwd / _bwd) on the
GPU against the oracle's per-projection layer with the input gradients summed.
Each projection's base is packed on its own and the packed weights are stacked
by rows; the oracle decodes each projection's own bytes."""
import numpy as np
import pytest

import oracle
import qlora_synth as syn
from gpu_helpers import check_bf16, check_f32, sample_rows

pytestmark = pytest.mark.gpu


def make_multi(M, K, Ns, r, fmt, dq, seed):
    wl = syn.Workload("multi", fmt, dq, M, r, float(2 * r), [syn.Linear(f"p{i}", K, n) for i, n in enumerate(Ns)])
    ins = [syn.make_linear_inputs(wl, i, seed=seed) for i in range(len(Ns))]
    return {"ins": ins, "X": ins[0]["X"], "A": np.stack([i["A"] for i in ins]),
            "B": np.concatenate([i["B"] for i in ins], axis=0),
            "dY": np.concatenate([i["dY"] for i in ins], axis=1), "Ns": Ns, "r": r, "alpha": wl.alpha, "M": M, "K": K}


def run_multi(lib, d):
    import torch

    w = lib.DeviceWeight.from_packed(lib.stack_weights([i["W"] for i in d["ins"]]))
    X, dY = lib.bf16_from_bits(d["X"]), lib.bf16_from_bits(d["dY"])
    A, B = lib.bf16_from_bits(d["A"]), lib.bf16_from_bits(d["B"])
    Y, T = lib.multi_linear_fwd(w, d["Ns"], X, A, B, d["alpha"])
    dX, dA, dB = lib.multi_linear_bwd(w, d["Ns"], X, A, B, T, dY, d["alpha"])
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    return {"Y": lib.bits_from_bf16(Y), "T": T.cpu().numpy(), "dX": lib.bits_from_bf16(dX), "dA": dA.cpu().numpy(),
            "dB": dB.cpu().numpy()}


def oracle_multi(d, rows=None):
    Wds = [oracle.dequant(i["W"]) for i in d["ins"]]
    As = [oracle.bf16_bits_to_f64(a) for a in d["A"]]
    Bs = np.split(oracle.bf16_bits_to_f64(d["B"]), np.cumsum(d["Ns"])[:-1], axis=0)
    X = d["X"] if rows is None else d["X"][rows]
    dYr = d["dY"] if rows is None else d["dY"][rows]
    Y, T = oracle.multi_linear_fwd(X, Wds, As, Bs, d["alpha"])
    g_rows = oracle.multi_linear_bwd(X, Wds, As, Bs, dYr, d["alpha"])
    if rows is None:
        g = g_rows
    else:  # adapter gradients over every row: only T and U are needed
        Xa = oracle.bf16_bits_to_f64(d["X"])
        dYa = oracle.bf16_bits_to_f64(d["dY"])
        s = d["alpha"] / d["r"]
        offs = np.cumsum([0] + list(d["Ns"]))
        Ts = [Xa @ A.T for A in As]
        Us = [dYa[:, offs[p]:offs[p + 1]] @ Bs[p] for p in range(len(As))]
        g = {"dA": np.stack([s * U.T @ Xa for U in Us]),
             "dB": np.concatenate([s * dYa[:, offs[p]:offs[p + 1]].T @ Ts[p] for p in range(len(As))]),
             "T": np.concatenate(Ts, axis=1)}
    return {"Y": Y, "T": T if rows is None else g["T"], "dX": g_rows["dX"], "dA": g["dA"], "dB": g["dB"]}


@pytest.mark.parametrize("fmt,dq", [("nf4", True), ("q8_0", False), ("bf16", False), ("q4_0", False)])
@pytest.mark.parametrize("M", [64, 300])
def test_three_projections(lib, fmt, dq, M):
    d = make_multi(M, 256, [256, 512, 256], 16, fmt, dq, seed=M)
    got, ref = run_multi(lib, d), oracle_multi(d)
    check_bf16(got["Y"], ref["Y"], "Y")
    check_f32(got["T"], ref["T"], "T")
    check_bf16(got["dX"], ref["dX"], "dX")
    check_f32(got["dA"], ref["dA"], "dA")
    check_f32(got["dB"], ref["dB"], "dB")


@pytest.mark.parametrize("Ns,r", [([256, 512, 256], 8), ([256, 256], 24), ([512, 256], 32), ([256, 256, 256], 16)])
def test_projection_windows(lib, Ns, r):
    """dB of each projection uses only that projection's columns of T: ranks
    whose windows are not aligned to 16 columns (8, 24) and adapter chunks of
    up to 64 columns, on 64-column tiles of dY."""
    d = make_multi(300, 256, Ns, r, "q8_0", False, seed=r)
    got, ref = run_multi(lib, d), oracle_multi(d)
    check_bf16(got["dX"], ref["dX"], "dX")
    check_f32(got["dA"], ref["dA"], "dA")
    check_f32(got["dB"], ref["dB"], "dB")


def test_one_projection_is_the_single_linear(lib):
    """P = 1 runs the same kernels as qlora_linear_fwd / _bwd: bitwise equal."""
    from gpu_helpers import run_layer

    d = make_multi(200, 512, [320], 16, "nf4", False, seed=4)
    got = run_multi(lib, d)
    i = d["ins"][0]
    single = run_layer(i)
    for k in got:
        assert np.array_equal(got[k].reshape(-1), single[k].reshape(-1)), k


def test_rejects_bad_splits(lib):
    import torch

    d = make_multi(64, 256, [256, 256], 16, "q8_0", False, seed=1)
    w = lib.DeviceWeight.from_packed(lib.stack_weights([i["W"] for i in d["ins"]]))
    X = lib.bf16_from_bits(d["X"])
    A, B = lib.bf16_from_bits(d["A"]), lib.bf16_from_bits(d["B"])
    # widths not summing to N; a width not a multiple of 256; no projection
    for ns, status in (([256, 512], -1), ([128, 384], -2), ([], -1)):
        with pytest.raises(lib.QloraError) as e:
            lib.multi_linear_fwd(w, ns, X, A, B, 32.0, workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
        assert e.value.status == status, ns


@pytest.mark.slow
@pytest.mark.parametrize("which", ["qkv", "gate_up"])
def test_llama_fused_projections(lib, which):
    """Llama-3.1-8B-shaped fused launches (NF4 + double-quantised absmax,
    M 4096, rank 16): q|k|v 4096 -> 4096 + 1024 + 1024 and gate|up 4096 ->
    14336 + 14336.  Y and dX on sampled rows, T, dA, dB in full."""
    Ns = [4096, 1024, 1024] if which == "qkv" else [14336, 14336]
    d = make_multi(4096, 4096, Ns, 16, "nf4", True, seed=11)
    got = run_multi(lib, d)
    rows = sample_rows(4096, 192)
    ref = oracle_multi(d, rows=rows)
    M, N = 4096, sum(Ns)
    check_bf16(got["Y"].reshape(M, N)[rows], ref["Y"], "Y")
    check_bf16(got["dX"].reshape(M, 4096)[rows], ref["dX"], "dX")
    check_f32(got["T"], ref["T"], "T")
    check_f32(got["dA"], ref["dA"], "dA")
    check_f32(got["dB"], ref["dB"], "dB")
