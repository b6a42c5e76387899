"""Shared helpers of the GPU parity tests: device upload, tolerance checks."""
from __future__ import annotations

import numpy as np

import oracle
import qlora_synth as syn


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values around |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def check_bf16(got_bits: np.ndarray, ref: np.ndarray, name: str, rel: float = 1e-2) -> float:
    """max|err| <= rel*RMS(ref) + 1/2 ulp_bf16(|ref|), elementwise."""
    got = oracle.bf16_bits_to_f64(got_bits).reshape(ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(got - ref)
    tol = rel * rms + 0.5 * bf16_ulp(ref)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} of {err.size} out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} tol {tol[i]:.3g} (rms {rms:.3g})")
    return float(err.max() / rms) if rms > 0 else 0.0


def check_f32(got: np.ndarray, ref: np.ndarray, name: str, rel: float = 1e-2) -> float:
    """max|err| <= rel*RMS(ref)."""
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    assert err <= rel * rms, f"{name}: max err {err:.4g} > {rel} * rms {rms:.4g}"
    return err / rms if rms > 0 else 0.0


def to_device(inp):
    import quantized_base_lora_block_gb300 as q

    d = {k: q.bf16_from_bits(inp[k]) for k in ("X", "A", "B", "dY")}
    d["W"] = q.DeviceWeight.from_packed(inp["W"])
    return d


def run_layer(inp, want_dx=True):
    """fwd + bwd through the C ABI; returns host arrays."""
    import torch

    import quantized_base_lora_block_gb300 as q

    d = to_device(inp)
    Y, T = q.linear_fwd(d["W"], d["X"], d["A"], d["B"], inp["alpha"])
    dX, dA, dB = q.linear_bwd(d["W"], d["X"], d["A"], d["B"], T, d["dY"], inp["alpha"], want_dx=want_dx)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    out = {"Y": q.bits_from_bf16(Y), "T": T.cpu().numpy(), "dA": dA.cpu().numpy(), "dB": dB.cpu().numpy()}
    if dX is not None:
        out["dX"] = q.bits_from_bf16(dX)
    return out


def oracle_layer(inp, rows=None):
    """Oracle on all rows (rows=None) or on a row sample for Y / dX."""
    Wd = oracle.dequant(inp["W"])
    X, A, B, dY = inp["X"], inp["A"], inp["B"], inp["dY"]
    alpha = inp["alpha"]
    g = oracle.linear_bwd_adapter_grads(X, A, B, dY, alpha)
    if rows is None:
        Y, T = oracle.linear_fwd(X, Wd, A, B, alpha)
        dX = oracle.linear_bwd_rows(dY, Wd, A, B, alpha)
    else:
        Y, T = oracle.linear_fwd_rows(X[rows], Wd, A, B, alpha)
        dX = oracle.linear_bwd_rows(dY[rows], Wd, A, B, alpha)
    return {"Y": Y, "T": T, "dX": dX, "dA": g["dA"], "dB": g["dB"], "T_all": g["T"]}


def sample_rows(M: int, n: int = 256, seed: int = 0, tile: int = 128) -> np.ndarray:
    """Seeded row sample including the first/last row of every tile boundary
    region near the start and end, plus random rows."""
    rng = np.random.default_rng(seed)
    edge = [0, 1, M - 1, M - 2]
    for t in range(tile, M, tile):
        if len(edge) > n // 2:
            break
        edge += [t - 1, t]
    rest = rng.choice(M, size=min(M, n), replace=False)
    rows = np.unique(np.clip(np.array(edge + list(rest)), 0, M - 1))
    return rows[:n] if rows.size > n else rows
