"""Stacked adapters (qlora_stacked_linear_fwd / _bwd) on the GPU against the
oracle: several LoRA pairs of different ranks and scales on one frozen base,
applied together; a frozen adapter gets no gradient."""
import numpy as np
import pytest

import oracle
import qlora_synth as syn
from gpu_helpers import check_bf16, check_f32

pytestmark = pytest.mark.gpu


def make(M, K, N, ranks, alphas, fmt, dq, seed):
    wl = syn.Workload("stk", fmt, dq, M, ranks[0], alphas[0], [syn.Linear("t", K, N)])
    inp = syn.make_linear_inputs(wl, 0, seed=seed)
    As = [syn.normal_bf16(syn.rng_for(seed, 50 + i, 0, syn.S_A), (r, K), 1.0 / np.sqrt(K)) for i, r in enumerate(ranks)]
    Bs = [syn.normal_bf16(syn.rng_for(seed, 50 + i, 0, syn.S_B), (N, r), 0.01) for i, r in enumerate(ranks)]
    return {"X": inp["X"], "dY": inp["dY"], "W": inp["W"], "As": As, "Bs": Bs, "alphas": alphas, "M": M, "K": K,
            "N": N}


def run(lib, d, trainable=None):
    import torch

    w = lib.DeviceWeight.from_packed(d["W"])
    X, dY = lib.bf16_from_bits(d["X"]), lib.bf16_from_bits(d["dY"])
    As = [lib.bf16_from_bits(a) for a in d["As"]]
    Bs = [lib.bf16_from_bits(b) for b in d["Bs"]]
    Y, T = lib.stacked_linear_fwd(w, X, As, Bs, d["alphas"])
    dX, dAs, dBs = lib.stacked_linear_bwd(w, X, As, Bs, d["alphas"], T, dY, trainable=trainable)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    return {"Y": lib.bits_from_bf16(Y), "T": T.cpu().numpy(), "dX": lib.bits_from_bf16(dX),
            "dA": [None if a is None else a.cpu().numpy() for a in dAs],
            "dB": [None if b is None else b.cpu().numpy() for b in dBs]}


def ref(d):
    Wd = oracle.dequant(d["W"])
    As = [oracle.bf16_bits_to_f64(a) for a in d["As"]]
    Bs = [oracle.bf16_bits_to_f64(b) for b in d["Bs"]]
    Y, T = oracle.stacked_linear_fwd(d["X"], Wd, As, Bs, d["alphas"])
    g = oracle.stacked_linear_bwd(d["X"], Wd, As, Bs, d["dY"], d["alphas"])
    return {"Y": Y, "T": T, **g}


@pytest.mark.parametrize("fmt,dq", [("nf4", True), ("q8_0", False), ("bf16", False)])
@pytest.mark.parametrize("M", [64, 300])
def test_two_stacked_adapters(lib, fmt, dq, M):
    d = make(M, 512, 384, [8, 16], [16.0, 8.0], fmt, dq, seed=M + 3)
    got, r = run(lib, d), ref(d)
    check_bf16(got["Y"], r["Y"], "Y")
    check_f32(got["T"], r["T"], "T")
    check_bf16(got["dX"], r["dX"], "dX")
    for i in range(2):
        check_f32(got["dA"][i], r["dA"][i], f"dA[{i}]")
        check_f32(got["dB"][i], r["dB"][i], f"dB[{i}]")


def test_frozen_lower_adapter_and_three_adapters(lib):
    d = make(200, 256, 320, [8, 16, 8], [8.0, 32.0, 4.0], "nf4", False, seed=9)
    got, r = run(lib, d, trainable=[False, True, True]), ref(d)
    check_bf16(got["Y"], r["Y"], "Y")
    check_bf16(got["dX"], r["dX"], "dX")
    assert got["dA"][0] is None and got["dB"][0] is None
    for i in (1, 2):
        check_f32(got["dA"][i], r["dA"][i], f"dA[{i}]")
        check_f32(got["dB"][i], r["dB"][i], f"dB[{i}]")


def test_one_stacked_adapter_is_the_single_linear(lib):
    """n_adapters = 1 computes the single adapter's layer: same results as
    qlora_linear_fwd / _bwd within the tolerance (same kernels; the adapter is
    read from its packed copy)."""
    from gpu_helpers import run_layer

    d = make(300, 512, 256, [16], [32.0], "nf4", True, seed=5)
    got = run(lib, d)
    single = run_layer({"X": d["X"], "A": d["As"][0], "B": d["Bs"][0], "dY": d["dY"], "W": d["W"], "alpha": 32.0})
    for k in ("Y", "dX", "T"):
        assert np.array_equal(got[k].reshape(-1), single[k].reshape(-1)), k
    assert np.array_equal(got["dA"][0], single["dA"]) and np.array_equal(got["dB"][0], single["dB"])
