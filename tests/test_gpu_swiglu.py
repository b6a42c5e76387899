"""Gate / up projections with the SwiGLU activation (qlora_swiglu_fwd /
_bwd) on the GPU against the oracle.  Forward: the pre-activations G | U,
T, and H = silu(G) U computed from G and U as stored.  Backward: dX (summed
over gate and up), per-projection dA and dB from dH and a given G | U (the
stored pre-activations are an input of the backward, so the backward is
checked on seeded G | U, and the chained forward + backward through the
layer's own G | U)."""
import ctypes

import numpy as np
import pytest

import oracle
import qlora_synth as syn
from gpu_helpers import bf16_ulp, check_bf16, check_f32
from test_gpu_multi import make_multi

pytestmark = pytest.mark.gpu


def _split(d):
    Wg, Wu = (oracle.dequant(i["W"]) for i in d["ins"])
    Ag, Au = (oracle.bf16_bits_to_f64(a) for a in d["A"])
    Bg, Bu = np.split(oracle.bf16_bits_to_f64(d["B"]), 2, axis=0)
    return Wg, Wu, Ag, Au, Bg, Bu


def _device(lib, d):
    w = lib.DeviceWeight.from_packed(lib.stack_weights([i["W"] for i in d["ins"]]))
    return w, lib.bf16_from_bits(d["X"]), lib.bf16_from_bits(d["A"]), lib.bf16_from_bits(d["B"])


def check_h(got_bits, G, U, T, d, name="H"):
    """H from the stored G, U: each is the exact value moved by the
    forward's arithmetic — fp32 accumulation over the K + r bf16 products
    (the sequential bound (K + r) 2^-24 of the absolute-value products, times
    4 for the tensor core's own summation order and alignment), the adapter
    operand s T rounded to bf16 (2^-9 of |s T| |B|^T) and the bf16 rounding
    of the result (one ulp allowed).  H moves by |dH/dG| and |dH/dU| times
    those, and is rounded once more."""
    Wg, Wu, _, _, Bg, Bu = _split(d)
    r, sc = d["r"], d["alpha"] / d["r"]
    acc = 4.0 * (d["K"] + r) * 2.0 ** -24
    aX, aT = np.abs(oracle.bf16_bits_to_f64(d["X"])), np.abs(T)
    aBg, aBu = np.abs(Bg).T, np.abs(Bu).T
    eG = (2.0 ** -9 + acc) * (sc * aT[:, :r]) @ aBg + acc * aX @ np.abs(Wg).T + bf16_ulp(G)
    eU = (2.0 ** -9 + acc) * (sc * aT[:, r:]) @ aBu + acc * aX @ np.abs(Wu).T + bf16_ulp(U)
    s = 1.0 / (1.0 + np.exp(-G))
    H = G * s * U
    tol = np.abs(U * s * (1.0 + G * (1.0 - s))) * eG + np.abs(G * s) * eU + 0.5 * eG * eU + bf16_ulp(H)
    got = oracle.bf16_bits_to_f64(got_bits).reshape(H.shape)
    err = np.abs(got - H)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} of {err.size} out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {H[i]!r} tol {tol[i]:.3g}")


def _inputs(M, I, K, r, fmt, dq, seed):
    d = make_multi(M, K, [I, I], r, fmt, dq, seed=seed)
    dH = syn.normal_bf16(syn.rng_for(seed, 99, 0, syn.S_DY), (M, I), 1.0)
    # seeded pre-activations for the backward, wide enough to reach the
    # saturated ends of silu
    GU = syn.normal_bf16(syn.rng_for(seed, 99, 1, syn.S_X), (M, 2 * I), 2.0)
    return d, dH, GU


@pytest.mark.parametrize("fmt,dq", [("nf4", True), ("q8_0", False), ("bf16", False), ("q4_k", False)])
@pytest.mark.parametrize("M", [96, 300, 1030])
def test_swiglu_layer(lib, fmt, dq, M):
    """96 rows: the one-CTA GEMM and the elementwise activation pass; 300 and
    1030 rows: the activation in the pair kernel's epilogue."""
    import torch

    I, K, r = 512, 512, 16
    d, dH_bits, GU_bits = _inputs(M, I, K, r, fmt, dq, seed=M + 5)
    Wg, Wu, Ag, Au, Bg, Bu = _split(d)
    w, X, A, B = _device(lib, d)
    H, GU, T = lib.swiglu_fwd(w, X, A, B, d["alpha"])
    dX, dA, dB = lib.swiglu_bwd(w, X, A, B, T, lib.bf16_from_bits(GU_bits), lib.bf16_from_bits(dH_bits), d["alpha"])
    torch.cuda.synchronize()
    assert lib.device_error() == 0

    Hr, Gr, Ur, Tr = oracle.swiglu_fwd(d["X"], Wg, Wu, Ag, Au, Bg, Bu, d["alpha"])
    check_bf16(lib.bits_from_bf16(GU), np.concatenate([Gr, Ur], axis=1), "G | U")
    check_f32(T.cpu().numpy(), Tr, "T")
    check_h(lib.bits_from_bf16(H), Gr, Ur, Tr, d)

    Gs, Us = np.split(oracle.bf16_bits_to_f64(GU_bits), 2, axis=1)
    g = oracle.swiglu_bwd(d["X"], Wg, Wu, Ag, Au, Bg, Bu, dH_bits, d["alpha"], G=Gs, U=Us)
    check_bf16(lib.bits_from_bf16(dX), g["dX"], "dX")
    check_f32(dA.cpu().numpy(), g["dA"], "dA")
    check_f32(dB.cpu().numpy(), g["dB"], "dB")


def test_swiglu_chained(lib):
    """Forward, then the backward from the forward's own G | U, on one
    workspace.  The stored G | U differ from the exact ones by the forward's
    rounding, which silu' and silu'' carry into every row of dY, so the
    gradients are held to the oracle's chain at the RMS level (1e-2)."""
    import torch

    M, I, K, r = 640, 768, 256, 8
    d, dH_bits, _ = _inputs(M, I, K, r, "nf4", True, seed=3)
    w, X, A, B = _device(lib, d)
    ws = lib.alloc_workspace(lib.swiglu_workspace_bytes(w, M, r))
    H, GU, T = lib.swiglu_fwd(w, X, A, B, d["alpha"], workspace=ws)
    dX, dA, dB = lib.swiglu_bwd(w, X, A, B, T, GU, lib.bf16_from_bits(dH_bits), d["alpha"], workspace=ws)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    Hr, Gr, Ur, Tr = oracle.swiglu_fwd(d["X"], *_split(d), d["alpha"])
    check_h(lib.bits_from_bf16(H), Gr, Ur, Tr, d)
    Wg, Wu, Ag, Au, Bg, Bu = _split(d)
    g = oracle.swiglu_bwd(d["X"], Wg, Wu, Ag, Au, Bg, Bu, dH_bits, d["alpha"], G=Gr, U=Ur)
    for name, got, ref in (("dX", oracle.bf16_bits_to_f64(lib.bits_from_bf16(dX)), g["dX"]),
                           ("dA", dA.cpu().numpy(), g["dA"]), ("dB", dB.cpu().numpy(), g["dB"])):
        rms = np.sqrt(np.mean(ref * ref))
        assert np.sqrt(np.mean((got.reshape(ref.shape) - ref) ** 2)) <= 1e-2 * rms, name


@pytest.mark.parametrize("M", [100, 640])
def test_h_is_the_activation_of_the_stored_g_u(lib, M):
    """With 100 rows H comes from the elementwise pass, with 640 from the
    GEMM epilogue; both take G and U as stored, so H is silu(G) U of the
    returned bf16 G | U rounded once (fp32 arithmetic: 1e-5 relative)."""
    import torch

    I, K, r = 768, 256, 8
    d, _, _ = _inputs(M, I, K, r, "nf4", True, seed=2)
    w, X, A, B = _device(lib, d)
    H, GU, _ = lib.swiglu_fwd(w, X, A, B, d["alpha"])
    torch.cuda.synchronize()
    gu = oracle.bf16_bits_to_f64(lib.bits_from_bf16(GU)).reshape(M, 2 * I)
    G, U = gu[:, :I], gu[:, I:]
    ref = G / (1 + np.exp(-G)) * U
    h = oracle.bf16_bits_to_f64(lib.bits_from_bf16(H)).reshape(M, I)
    assert np.all(np.abs(h - ref) <= 0.5 * bf16_ulp(ref) + 1e-5 * np.abs(ref))


def test_swiglu_zero_rows(lib):
    """M = 0: the forward writes nothing; the backward sets dA and dB to zero."""
    import torch

    d, _, _ = _inputs(64, 256, 256, 8, "q8_0", False, seed=4)
    w, X, A, B = _device(lib, d)
    H, GU, T = lib.swiglu_fwd(w, X[:0].contiguous(), A, B, d["alpha"])
    assert H.shape == (0, 256) and GU.shape == (0, 512) and T.shape == (0, 16)
    dA = torch.full((2, 8, 256), 5.0, device="cuda")
    dB = torch.full((512, 8), 5.0, device="cuda")
    lib.swiglu_bwd(w, X[:0].contiguous(), A, B, T, GU, H, d["alpha"], dA=dA, dB=dB, want_dx=False)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert float(dA.abs().max()) == 0.0 and float(dB.abs().max()) == 0.0


def test_swiglu_rejects_shapes(lib):
    d = make_multi(64, 256, [384, 384], 16, "q8_0", False, seed=1)   # I % 256 != 0
    w = lib.DeviceWeight.from_packed(lib.stack_weights([i["W"] for i in d["ins"]]))
    assert lib.load().qlora_swiglu_workspace_bytes(ctypes.byref(w.desc), 64, 16) == 0
    d = make_multi(64, 256, [256, 256], 40, "q8_0", False, seed=1)   # 2 rank > 64
    w = lib.DeviceWeight.from_packed(lib.stack_weights([i["W"] for i in d["ins"]]))
    assert lib.load().qlora_swiglu_workspace_bytes(ctypes.byref(w.desc), 64, 40) == 0
