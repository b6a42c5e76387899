"""Seeded random sweep of the plain layer call over formats, shapes and
ranks (M from 1 to 700 rows, K and N multiples of 64 up to 1152, rank a
multiple of 8 up to 64), each against the oracle at the stated tolerance;
it reaches tile and launch choices the structured cases do not list one by
one (one-CTA and pair kernels, 512 x 128 and 512 x 256 tiles, ragged row
and column blocks)."""
import numpy as np
import pytest

from gpu_helpers import oracle_layer, run_layer
from test_gpu_linear import check_all, make

pytestmark = pytest.mark.gpu

FORMATS = [("bf16", False), ("nf4", False), ("nf4", True), ("q8_0", False), ("q4_0", False), ("q4_k", False),
           ("fp8_e4m3", False), ("nvfp4", False), ("nf4_dqmap", False)]


def _cases(n=36, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        fmt, dq = FORMATS[i % len(FORMATS)]
        kq = 256 if fmt == "q4_k" else 64
        M = int(rng.choice([1, 7, 64, 127, 128, 129, 200, 255, 256, 257, 384, 511, 513, 700]))
        K = int(rng.integers(1, 1152 // kq + 1)) * kq
        N = int(rng.integers(1, 1152 // 64 + 1)) * 64
        r = int(rng.integers(1, 9)) * 8
        out.append((fmt, dq, M, K, N, r, 1000 + i))
    return out


@pytest.mark.parametrize("fmt,dq,M,K,N,r,seed", _cases(),
                         ids=lambda v: str(v) if not isinstance(v, bool) else ("dq" if v else "-"))
def test_random_shape(lib, fmt, dq, M, K, N, r, seed):
    inp = make(M, K, N, r, fmt, dq, seed=seed)
    check_all(inp, run_layer(inp), oracle_layer(inp))


def _grouped_cases(n=12, seed=20261204):
    rng = np.random.default_rng(seed)
    fmts = ["q8_0", "nf4", "q4_0", "bf16", "q4_k", "fp8_e4m3"]
    out = []
    for i in range(n):
        fmt = fmts[i % len(fmts)]
        kq = 256 if fmt == "q4_k" else 64
        E = int(rng.integers(1, 9))
        counts = [int(c) if rng.random() > 0.2 else 0 for c in rng.integers(1, 400, size=E)]
        K = int(rng.integers(1, 768 // kq + 1)) * kq
        N = int(rng.integers(1, 768 // 64 + 1)) * 64
        r = int(rng.integers(1, 5)) * 8
        out.append((fmt, tuple(counts), K, N, r, 2000 + i))
    return out


@pytest.mark.parametrize("fmt,counts,K,N,r,seed", _grouped_cases(), ids=str)
def test_random_grouped(lib, fmt, counts, K, N, r, seed):
    from test_gpu_moe import _check, _moe_inputs, _oracle, _run

    d = _moe_inputs(list(counts), K, N, r, fmt, seed=seed)
    _check(d, _run(lib, d), _oracle(d))


def _multi_cases(n=8, seed=20261205):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        P = int(rng.integers(2, 4))
        r = int(rng.choice([8, 16]))
        Ns = [int(x) * 256 for x in rng.integers(1, 4, size=P)]
        M = int(rng.choice([64, 130, 300, 600]))
        K = int(rng.integers(1, 9)) * 64
        fmt = ["nf4", "q8_0", "bf16", "q4_0"][i % 4]
        out.append((fmt, M, K, tuple(Ns), r, 3000 + i))
    return out


@pytest.mark.parametrize("fmt,M,K,Ns,r,seed", _multi_cases(), ids=str)
def test_random_fused_projections(lib, fmt, M, K, Ns, r, seed):
    from gpu_helpers import check_bf16, check_f32
    from test_gpu_multi import make_multi, oracle_multi, run_multi

    d = make_multi(M, K, list(Ns), r, fmt, fmt == "nf4", seed=seed)
    got, ref = run_multi(lib, d), oracle_multi(d)
    check_bf16(got["Y"], ref["Y"], "Y")
    check_f32(got["T"], ref["T"], "T")
    check_bf16(got["dX"], ref["dX"], "dX")
    check_f32(got["dA"], ref["dA"], "dA")
    check_f32(got["dB"], ref["dB"], "dB")
