"""The calls can be captured in a CUDA graph: a forward + backward of fused
projections, a grouped (MoE) forward + backward and gate|up with SwiGLU,
each captured once on its own stream and replayed, give the same bits as
the same calls run eagerly.  Nothing in a call synchronises, allocates or
reads device memory on the host, and the backward's side-stream work joins
the capture through its fork / join events."""
import numpy as np
import pytest

import qlora_synth as syn
from test_gpu_moe import _moe_inputs
from test_gpu_multi import make_multi

pytestmark = pytest.mark.gpu


def _capture_and_compare(run, outputs):
    """run(stream) enqueues the calls; outputs() returns the result tensors."""
    import torch

    cur = torch.cuda.current_stream()
    run(cur)
    torch.cuda.synchronize()
    eager = [t.clone() for t in outputs()]
    for t in outputs():
        t.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(s)
    for t in outputs():  # capture launches nothing: replay writes them
        t.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outputs()):
        assert torch.equal(a, b)


def test_graph_fused_projections(lib):
    import torch

    d = make_multi(520, 512, [512, 256, 256], 16, "nf4", True, seed=21)
    w = lib.DeviceWeight.from_packed(lib.stack_weights([i["W"] for i in d["ins"]]))
    X, dY = lib.bf16_from_bits(d["X"]), lib.bf16_from_bits(d["dY"])
    A, B = lib.bf16_from_bits(d["A"]), lib.bf16_from_bits(d["B"])
    M, K, N, r, Ns = d["M"], d["K"], sum(d["Ns"]), d["r"], d["Ns"]
    ws = lib.alloc_workspace(lib.multi_workspace_bytes(w, Ns, M, r))
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    T = torch.empty((M, len(Ns) * r), dtype=torch.float32, device="cuda")
    dX = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dA = torch.empty((len(Ns), r, K), dtype=torch.float32, device="cuda")
    dB = torch.empty((N, r), dtype=torch.float32, device="cuda")

    def run(st):
        lib.multi_linear_fwd(w, Ns, X, A, B, d["alpha"], Y=Y, T=T, workspace=ws, stream=st)
        lib.multi_linear_bwd(w, Ns, X, A, B, T, dY, d["alpha"], dX=dX, dA=dA, dB=dB, workspace=ws, stream=st)

    _capture_and_compare(run, lambda: [Y, T, dX, dA, dB])
    assert lib.device_error() == 0


def test_graph_grouped(lib):
    import torch

    d = _moe_inputs([70, 0, 300, 5, 256], 256, 512, 16, "q8_0", seed=4)
    ws_e = lib.upload_experts(d["W"])
    X, dY = lib.bf16_from_bits(d["X"]), lib.bf16_from_bits(d["dY"])
    A, B = lib.bf16_from_bits(d["A"]), lib.bf16_from_bits(d["B"])
    off = lib.device_offsets(d["off"])
    R, E, r = int(d["off"][-1]), len(d["W"]), d["r"]
    K, N = 256, 512
    ws = lib.alloc_workspace(lib.grouped_workspace_bytes(ws_e, R, r))
    Y = torch.empty((R, N), dtype=torch.bfloat16, device="cuda")
    T = torch.empty((R, r), dtype=torch.float32, device="cuda")
    dX = torch.empty((R, K), dtype=torch.bfloat16, device="cuda")
    dA = torch.empty((E, r, K), dtype=torch.float32, device="cuda")
    dB = torch.empty((E, N, r), dtype=torch.float32, device="cuda")

    def run(st):
        lib.grouped_fwd(ws_e, off, X, A, B, d["alpha"], Y=Y, T=T, workspace=ws, stream=st)
        lib.grouped_bwd(ws_e, off, X, A, B, T, dY, d["alpha"], dX=dX, dA=dA, dB=dB, workspace=ws, stream=st)

    _capture_and_compare(run, lambda: [Y, T, dX, dA, dB])
    assert lib.device_error() == 0


def test_graph_swiglu(lib):
    import torch

    M, I, K, r = 300, 512, 256, 8
    d = make_multi(M, K, [I, I], r, "q4_0", False, seed=6)
    dH = lib.bf16_from_bits(syn.normal_bf16(syn.rng_for(6, 99, 0, syn.S_DY), (M, I), 1.0))
    w = lib.DeviceWeight.from_packed(lib.stack_weights([i["W"] for i in d["ins"]]))
    X, A, B = lib.bf16_from_bits(d["X"]), lib.bf16_from_bits(d["A"]), lib.bf16_from_bits(d["B"])
    ws = lib.alloc_workspace(lib.swiglu_workspace_bytes(w, M, r))
    H = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    GU = torch.empty((M, 2 * I), dtype=torch.bfloat16, device="cuda")
    T = torch.empty((M, 2 * r), dtype=torch.float32, device="cuda")
    dX = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dA = torch.empty((2, r, K), dtype=torch.float32, device="cuda")
    dB = torch.empty((2 * I, r), dtype=torch.float32, device="cuda")

    def run(st):
        lib.swiglu_fwd(w, X, A, B, d["alpha"], H=H, GU=GU, T=T, workspace=ws, stream=st)
        lib.swiglu_bwd(w, X, A, B, T, GU, dH, d["alpha"], dX=dX, dA=dA, dB=dB, workspace=ws, stream=st)

    _capture_and_compare(run, lambda: [H, GU, T, dX, dA, dB])
    assert lib.device_error() == 0
