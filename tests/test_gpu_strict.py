"""The strict bound on the GEMM outputs, without the bf16 output rounding:
the debug forms of the calls return Y and dX as their fp32 accumulator
values, which must meet max|err| <= 1e-2 * RMS(ref) against the oracle with
no half-ulp allowance; rounding them to bf16 must give exactly the regular
calls' outputs."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check_f32, oracle_layer, run_layer, to_device
from test_gpu_linear import make

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,dq,shape", [
    ("nf4", True, (300, 512, 768, 16)),     # pair kernel, ragged rows
    ("q8_0", False, (96, 256, 320, 8)),     # one-CTA kernel (M <= 128)
    ("q4_k", False, (640, 1024, 512, 32)),
    ("nvfp4", False, (257, 640, 512, 16)),
    ("bf16", False, (200, 512, 320, 64)),
])
def test_fp32_outputs_meet_the_strict_bound(lib, fmt, dq, shape):
    import torch

    M, K, N, r = shape
    inp = make(M, K, N, r, fmt, dq, seed=M + 3 * K + N)
    ref = oracle_layer(inp)
    d = to_device(inp)
    Y32, T = lib.debug_linear_fwd_f32(d["W"], d["X"], d["A"], d["B"], inp["alpha"])
    dX32, dA, dB = lib.debug_linear_bwd_f32(d["W"], d["X"], d["A"], d["B"], T, d["dY"], inp["alpha"])
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    check_f32(Y32.cpu().numpy(), ref["Y"], "Y (fp32)")
    check_f32(dX32.cpu().numpy(), ref["dX"], "dX (fp32)")
    # the regular calls store exactly the bf16 rounding of these values
    got = run_layer(inp)
    y16 = oracle.bf16_round_f32(Y32.cpu().numpy()).view(np.uint32) >> 16
    dx16 = oracle.bf16_round_f32(dX32.cpu().numpy()).view(np.uint32) >> 16
    assert np.array_equal(y16.astype(np.uint16).reshape(-1), got["Y"].reshape(-1))
    assert np.array_equal(dx16.astype(np.uint16).reshape(-1), got["dX"].reshape(-1))
