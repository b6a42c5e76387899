"""The forward entry point that allocates nothing: qlora_linear_fwd_noalloc.

It exists for callers that cannot allocate device memory themselves (a
plug-in that only receives its host application's buffers, or a loop that
must not call cudaMalloc because it can synchronise the device).  It takes no
workspace and uses the library's fixed device scratch instead.  Here it is
called through the C ABI, twice in a row with different problems, and its
outputs are compared with those of qlora_linear_fwd on the same inputs.
"""
import ctypes

import numpy as np
import pytest

import oracle
import qlora_synth as syn
from gpu_helpers import check_bf16, check_f32, to_device

pytestmark = pytest.mark.gpu


def _inputs(M, K, N, r, fmt, dq, seed):
    wl = syn.Workload("noalloc", fmt, dq, M, r, float(2 * r), [syn.Linear("t", K, N)])
    return syn.make_linear_inputs(wl, 0, seed=seed)


def test_noalloc_forward_matches_regular_forward_two_calls(lib):
    import torch

    c = lib.load()
    for M, K, N, r, fmt, dq, seed in [(300, 512, 768, 16, "nf4", True, 11), (96, 256, 320, 8, "q8_0", False, 12)]:
        inp = _inputs(M, K, N, r, fmt, dq, seed)
        d = to_device(inp)
        w = d["W"]
        Y_ref, T_ref = lib.linear_fwd(w, d["X"], d["A"], d["B"], inp["alpha"])
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        T = torch.full((M, r), float("nan"), dtype=torch.float32, device="cuda")
        st = c.qlora_linear_fwd_noalloc(ctypes.byref(w.desc), M, r, inp["alpha"], d["X"].data_ptr(),
                                        d["A"].data_ptr(), d["B"].data_ptr(), Y.data_ptr(), T.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
        assert st == 0, lib.STATUS.get(st, st)
        torch.cuda.synchronize()
        assert lib.device_error() == 0
        y_ref = oracle.bf16_bits_to_f64(lib.bits_from_bf16(Y_ref)).reshape(M, N)
        check_bf16(lib.bits_from_bf16(Y), y_ref, "Y (no-alloc vs regular)")
        check_f32(T.cpu().numpy(), T_ref.cpu().numpy().astype(np.float64), "T (no-alloc vs regular)")


def test_noalloc_rejects_problems_larger_than_its_scratch(lib):
    import torch

    c = lib.load()
    cap = c.qlora_noalloc_scratch_bytes()
    assert cap == 16 << 20
    # a Llama-sized gate projection over 1,048,576 tokens: its forward needs
    # 32 MiB of scaled activation, more than the 16 MiB array
    desc = lib.WeightDesc(lib.FMT["nf4"], 0, 14336, 4096, 0x1000, 0x2000, None, None)
    assert c.qlora_forward_workspace_bytes(ctypes.byref(desc), 1 << 20, 16) > cap
    n0 = c.qlora_launch_count()
    st = c.qlora_linear_fwd_noalloc(ctypes.byref(desc), 1 << 20, 16, 16.0, 0x10000, 0x20000, 0x30000, 0x40000,
                                    0x50000, None)
    assert st == -6  # QLORA_ERR_WORKSPACE, nothing launched
    assert c.qlora_launch_count() == n0


def test_noalloc_serves_forwards_whose_backward_workspace_is_larger(lib):
    """131,072 rows at rank 16: the forward needs 4 MiB (fits the array), the
    forward+backward layout 20 MiB (does not)."""
    import torch

    c = lib.load()
    M, K, N, r = 131072, 256, 256, 16
    inp = _inputs(M, K, N, r, "q8_0", False, 13)
    d = to_device(inp)
    w = d["W"]
    assert c.qlora_forward_workspace_bytes(ctypes.byref(w.desc), M, r) <= c.qlora_noalloc_scratch_bytes()
    assert c.qlora_workspace_bytes(ctypes.byref(w.desc), M, r) > c.qlora_noalloc_scratch_bytes()
    Y_ref, T_ref = lib.linear_fwd(w, d["X"], d["A"], d["B"], inp["alpha"])
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    T = torch.empty((M, r), dtype=torch.float32, device="cuda")
    st = c.qlora_linear_fwd_noalloc(ctypes.byref(w.desc), M, r, inp["alpha"], d["X"].data_ptr(), d["A"].data_ptr(),
                                    d["B"].data_ptr(), Y.data_ptr(), T.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.STATUS.get(st, st)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert torch.equal(Y, Y_ref) and torch.equal(T, T_ref)

