#!/usr/bin/env python
"""Throughput of the LoRA linear over a frozen block-quantised base, fwd+bwd.

One step = forward of the 7 LoRA-adapted linears of one decoder layer (q, k,
v, o, gate, up, down), then their backward in reverse order, through the C ABI
(qlora_linear_fwd / qlora_linear_bwd).  Default workload: Llama-3.1-8B layer
shapes, NF4 base with double-quantised absmax, M = 4096 tokens, rank 16,
alpha 16; inputs synthetic and seeded.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica on its own GPU (the layer needs no exchange between replicas).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import qlora_synth as syn  # noqa: E402

METRIC = "QLoRA linear fwd+bwd tokens/s and TFLOP/s vs GB300 dense BF16 roofline"
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0
CPU_SAMPLE_ROWS = 64


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="llama31_8b_nf4dq", choices=sorted(syn.WORKLOADS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--stream-layers", type=int, default=32,
                   help="layers for the streamed leg (0 = skip); Llama workload only")
    p.add_argument("--no-moe", action="store_true", help="skip the grouped MoE leg")
    p.add_argument("--no-context", action="store_true",
                   help="skip the dequant_blocks GB/s and library-composition baseline legs")
    p.add_argument("--case", default=None, choices=["gemm_m128", "dequant", "linear_m4096", "swiglu"],
                   help="run one small case of a kernel family --steps times and print its time (for profiling): "
                        "gemm_m128 = Llama gate fwd+bwd at 128 rows (one-CTA GEMM), dequant = dequant_blocks of "
                        "the Llama gate base, linear_m4096 = Llama gate fwd+bwd at 4096 rows (reductions and pair "
                        "GEMM), swiglu = Llama gate|up with SwiGLU fwd+bwd at 4096 rows")
    p.add_argument("--only-moe", action="store_true",
                   help="run the grouped MoE leg alone and print its result (for profiling)")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the layer legs of the other configurations (Qwen3-0.6B bf16, Qwen3-8B Q4_0 / Q8_0)")
    return p.parse_args()


def captured_traffic(wl):
    """DRAM bytes per fused-GEMM launch from the committed ncu capture, or
    None when the kernel sources changed since it was taken (or for another
    workload)."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "qgemm_traffic_llama8b_nf4dq.json")
    if wl.name != "llama31_8b_nf4dq" or not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    h = hashlib.sha256()
    for src in d["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return d["traffic_bytes_per_launch"] if h.hexdigest() == d["sources_sha256"] else None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16": float(d["bf16_tflops"]), "bf16_sustained": float(d["bf16_tflops_sustained"]),
                "hbm": float(d["hbm_gbs"]), "source": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark(self, which: str):
        """Wall-clock bounds of the timed region (samples outside are dropped)."""
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t0", None), getattr(self, "t1", None)
        import datetime

        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            if ts is not None and t0 is not None and t1 is not None and not (t0 - 0.05 <= ts <= t1 + 0.05):
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# distributed plumbing (replicas)
# ----------------------------------------------------------------------------
def dist_init(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU oracle timing (baseline only; never part of the GPU path)
# ----------------------------------------------------------------------------
def oracle_step(inputs, rows: int):
    import oracle

    for inp in inputs:
        Wd = oracle.dequant(inp["W"])
        X, dY = inp["X"][:rows], inp["dY"][:rows]
        oracle.linear_fwd(X, Wd, inp["A"], inp["B"], inp["alpha"])
        oracle.linear_bwd(X, Wd, inp["A"], inp["B"], dY, inp["alpha"])


def cpu_threads() -> int:
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    return os.cpu_count() or 1


def time_oracle(inputs, rows: int, reps: int = 1) -> float:
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(inputs, rows)
    return (time.perf_counter() - t0) / reps


# ----------------------------------------------------------------------------
# streamed leg: L layers of the same shapes, bases in pinned host memory,
# one layer per pool slot, prefetched one layer ahead
# ----------------------------------------------------------------------------
def stream_leg(q, torch, inputs, L_dev, wl, n_layers, steps, stream, resident_ms_per_layer):
    blobs = [q.pack_weight_blob(inp["W"]) for inp in inputs]
    offs, o = [], 0
    for b, _ in blobs:
        offs.append(o)
        o = (o + b.nbytes + 255) // 256 * 256
    layer_bytes = o
    one = np.zeros(layer_bytes, dtype=np.uint8)
    for (b, _), off in zip(blobs, offs):
        one[off:off + b.nbytes] = b
    src = torch.from_numpy(one)
    hosts = []
    for _ in range(n_layers):
        h = torch.empty(layer_bytes, dtype=torch.uint8).pin_memory()
        h.copy_(src)
        hosts.append(h)
    pool = q.LayerStream(2, layer_bytes)
    M, r, alpha = wl.M, wl.rank, wl.alpha

    def views(base):
        return [q.weight_in_slot(inp["W"], bo, base + off) for inp, (_, bo), off in zip(inputs, blobs, offs)]

    def one_pass():
        pool.prefetch(0, hosts[0])
        for i in range(n_layers):
            if i + 1 < n_layers:
                pool.prefetch(i + 1, hosts[i + 1])
            ws = views(pool.acquire(i, stream))
            for d, w in zip(L_dev, ws):
                q.linear_fwd(w, d["X"], d["A"], d["B"], alpha, Y=d["Y"], T=d["T"], workspace=d["ws"], stream=stream)
            pool.release(i, stream)
        for i in reversed(range(n_layers)):
            pool.prefetch(i, hosts[i])
            if i > 0:
                pool.prefetch(i - 1, hosts[i - 1])
            ws = views(pool.acquire(i, stream))
            for d, w in zip(reversed(L_dev), reversed(ws)):
                q.linear_bwd(w, d["X"], d["A"], d["B"], d["T"], d["dY"], alpha, dX=d["dX"], dA=d["dA"], dB=d["dB"],
                             workspace=d["ws"], stream=stream)
            pool.release(i, stream)

    one_pass()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one_pass()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    pool.close()
    # one layer's copy alone, for context
    dst = torch.empty(layer_bytes, dtype=torch.uint8, device="cuda")
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for h in hosts[:4]:
        dst.copy_(h, non_blocking=True)
    c1.record(stream)
    torch.cuda.synchronize()
    alone = 4 * layer_bytes / (c0.elapsed_time(c1) / 1e3) / 1e9
    del dst
    # every layer is copied for the forward pass and again for the backward
    # pass, except the two the forward pass leaves resident
    h2d = (2 * n_layers - 2) * layer_bytes
    return {"layers": n_layers, "slots": 2, "layer_bytes": layer_bytes, "ms_per_pass": ms,
            "value": M / (ms / n_layers / 1e3), "unit": "tokens/s per layer (fwd+bwd)",
            "h2d_bytes_per_pass": h2d, "h2d_GBps": h2d / (ms / 1e3) / 1e9, "h2d_alone_GBps": alone,
            "streamed_over_resident": ms / (n_layers * resident_ms_per_layer),
            "note": "pinned host -> 2-slot device pool, one layer ahead on the library's copy stream; "
                    "fwd 0..L-1 then bwd L-1..0; each layer's 7 bases in one blob"}


def moe_leg(q, torch, steps, stream):
    mw = syn.MOE
    off, _, counts = syn.moe_routing(seed=0)
    lins = syn.moe_linears(mw)
    data = [syn.make_moe_linear_inputs(mw, i, off, seed=0) for i in range(len(lins))]
    rows = int(off[-1])
    off_dev = q.device_offsets(off)  # the router's offsets stay on the device
    dev = []
    for d in data:
        ws = q.upload_experts(d["W"])  # expert bases back to back (one tensor map)
        X, dY = q.bf16_from_bits(d["X"]), q.bf16_from_bits(d["dY"])
        A, B = q.bf16_from_bits(d["A"]), q.bf16_from_bits(d["B"])
        nb = q.grouped_workspace_bytes(ws, rows, mw.rank)
        dev.append({"W": ws, "X": X, "dY": dY, "A": A, "B": B, "alpha": d["alpha"], "ws": q.alloc_workspace(nb)})

    def step():
        Ts = []
        for d in dev:
            _, T = q.grouped_fwd(d["W"], off_dev, d["X"], d["A"], d["B"], d["alpha"], workspace=d["ws"],
                                 stream=stream)
            Ts.append(T)
        for d, T in zip(reversed(dev), reversed(Ts)):
            q.grouped_bwd(d["W"], off_dev, d["X"], d["A"], d["B"], T, d["dY"], d["alpha"], workspace=d["ws"],
                          stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # a second pass with every grouped GEMM launch bracketed by events
    q.profile_gemm(True)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    q.profile_gemm(False)
    gemm_ms, gemm_n, gemm_flops = q.profile_gemm_read()
    flops = sum(syn.linear_flops(rows, l.K, l.N, mw.rank) for l in lins)
    return {"workload": "moe_q8_0: 128 experts, top-8 of 4096 tokens (32768 rows, Zipf-skewed, "
                        f"{int((counts == 0).sum())} experts empty), gate/up 2048->768, down 768->2048, rank 16",
            "ms_per_step": ms, "tokens_per_s": mw.tokens / (ms / 1e3), "rows_per_s": rows / (ms / 1e3),
            "tflops": flops / (ms / 1e3) / 1e12,
            "gemm": {"ms_per_step": gemm_ms / steps, "launches_per_step": gemm_n / steps,
                     "tflops": gemm_flops / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None,
                     "kernel": "qgemm_pair_kernel grouped (256x256 tiles, Q8_0 decode in the producer)"}}


def dequant_leg(q, torch, L, wl, peaks, reps=20):
    """dequant_blocks on every distinct base weight of the layer: the
    standalone block decode to bf16 in HBM (HBM-bound): bytes read (codes
    and scales) + bytes written (bf16), per second."""
    out, seen = [], set()
    stream = torch.cuda.current_stream()
    for lin, d in zip(wl.linears, L):
        key = (d["N"], d["K"])
        if key in seen:
            continue
        seen.add(key)
        w = d["W"]
        Wd = torch.empty((w.N, w.K), dtype=torch.bfloat16, device=w.data.device)
        # L2 (129 MB) is emptied before each timed launch by reading a larger
        # buffer (a read leaves no dirty lines whose write-back would share
        # the timed launch's DRAM bandwidth)
        flush = torch.ones(256 << 20, dtype=torch.uint8, device=w.data.device)
        for _ in range(3):
            q.dequant_blocks(w, out=Wd, stream=stream)
        ts = []
        for _ in range(reps):
            flush.max()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            q.dequant_blocks(w, out=Wd, stream=stream)
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        ms = sorted(ts)[len(ts) // 2]
        nbytes = w.nbytes() + Wd.numel() * 2
        gbs = nbytes / (ms / 1e3) / 1e9
        out.append({"linear": lin.name, "N": w.N, "K": w.K, "us": ms * 1e3, "bytes": nbytes, "GBps": gbs,
                    "frac_of_measured_hbm": gbs / peaks["hbm"]})
    return {"kernel": "dequant_kernel (dequant_blocks)", "format": wl.fmt + ("+dq" if wl.double_quant else ""),
            "l2": "emptied before each timed launch (256 MB read)", "per_weight": out,
            "note": "the traffic is 79 % writes (bf16 out) against a copy-measured peak (half reads, half writes)"}


def library_leg(q, torch, L, wl, steps):
    """Context baseline: the same layer composed from library pieces, as a
    framework without fused kernels would run it: each linear decodes its
    base to bf16 in HBM with dequant_blocks (forward and again for dX), then
    cuBLAS bf16 GEMMs (torch.matmul) and PyTorch ops for the adapter terms
    and gradients."""
    M, r, alpha = wl.M, wl.rank, wl.alpha
    s = alpha / r
    stream = torch.cuda.current_stream()
    Wd = torch.empty(max(d["N"] * d["K"] for d in L), dtype=torch.bfloat16, device=L[0]["X"].device)

    def step():
        for d in L:
            w = q.dequant_blocks(d["W"], out=Wd[: d["N"] * d["K"]].view(d["N"], d["K"]), stream=stream)
            T = d["X"] @ d["A"].t()
            d["Y"].copy_(d["X"] @ w.t() + (s * T) @ d["B"].t())
            d["T"].copy_(T.float())
        for d in reversed(L):
            w = q.dequant_blocks(d["W"], out=Wd[: d["N"] * d["K"]].view(d["N"], d["K"]), stream=stream)
            U = d["dY"] @ d["B"]
            d["dX"].copy_(d["dY"] @ w + (s * U) @ d["A"])
            d["dA"].copy_(s * (U.t().float() @ d["X"].float()))
            d["dB"].copy_(s * (d["dY"].t().float() @ d["T"]))

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    flops = sum(syn.linear_flops(M, l.K, l.N, r) for l in wl.linears)
    return {"ms_per_step": ms, "value": M / (ms / 1e3), "unit": "tokens/s", "tflops": flops / (ms / 1e3) / 1e12,
            "kind": "context (library composition, not the product path)",
            "note": "dequant_blocks to bf16 in HBM + torch.matmul (cuBLAS bf16) + PyTorch adapter ops; dA, dB "
                    "in fp32"}


def run_case(args):
    """One small case of a kernel family, --steps times (for ncu captures)."""
    import torch

    import quantized_base_lora_block_gb300 as q

    q.load()
    wl = syn.WORKLOADS["llama31_8b_nf4dq"]
    M = {"gemm_m128": 128, "dequant": 1, "linear_m4096": 4096, "swiglu": 4096}[args.case]
    gate = [i for i, l in enumerate(wl.linears) if l.name == "gate_proj"][0]
    inp = syn.make_linear_inputs(wl, gate, seed=0, M=M)
    w = q.DeviceWeight.from_packed(inp["W"])
    X, A, B, dY = (q.bf16_from_bits(inp[k]) for k in ("X", "A", "B", "dY"))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.case == "swiglu":
        up = [i for i, l in enumerate(wl.linears) if l.name == "up_proj"][0]
        inu = syn.make_linear_inputs(wl, up, seed=0, M=M)
        w = q.DeviceWeight.from_packed(q.stack_weights([inp["W"], inu["W"]]))
        A = q.bf16_from_bits(np.stack([inp["A"], inu["A"]]))
        B = q.bf16_from_bits(np.concatenate([inp["B"], inu["B"]], axis=0))
        ws = q.alloc_workspace(q.swiglu_workspace_bytes(w, M, wl.rank))
        H, GU, T = q.swiglu_fwd(w, X, A, B, wl.alpha, workspace=ws)

        def f():
            q.swiglu_fwd(w, X, A, B, wl.alpha, H=H, GU=GU, T=T, workspace=ws)
            q.swiglu_bwd(w, X, A, B, T, GU, dY, wl.alpha, workspace=ws)
    elif args.case == "dequant":
        out = torch.empty((w.N, w.K), dtype=torch.bfloat16, device="cuda")
        f = lambda: q.dequant_blocks(w, out=out)  # noqa: E731
    else:
        ws = q.alloc_workspace(q.workspace_bytes(w, M, wl.rank))
        Y, T = q.linear_fwd(w, X, A, B, wl.alpha, workspace=ws)

        def f():
            q.linear_fwd(w, X, A, B, wl.alpha, Y=Y, T=T, workspace=ws)
            q.linear_bwd(w, X, A, B, T, dY, wl.alpha, workspace=ws)
    f()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(args.steps):
        f()
    e1.record()
    torch.cuda.synchronize()
    assert q.device_error() == 0
    print(json.dumps({"case": args.case, "rows": M, "ms_per_iter": e0.elapsed_time(e1) / args.steps}))


def fused_groups(wl):
    """Linears of a decoder layer that share their input and run as one fused
    launch (q|k|v, gate|up), where the fused call supports them (widths
    multiples of 256, P rank <= 64); every other linear on its own."""
    names = [l.name for l in wl.linears]
    groups, done = [], set()
    for members in (("q_proj", "k_proj", "v_proj"), ("gate_proj", "up_proj")):
        idx = [names.index(n) for n in members if n in names]
        if (len(idx) == len(members) and len(idx) * wl.rank <= 64 and
                all(wl.linears[i].N % 256 == 0 for i in idx)):
            groups.append(idx)
            done.update(idx)
    for i in range(len(names)):
        if i not in done:
            groups.append([i])
    return sorted(groups, key=lambda g: g[0])


def make_units(q, torch, wl, inputs, dev, groups):
    """Device tensors of each launch unit: the stacked base, the shared input
    (the first member's X), stacked adapters, concatenated dY, outputs."""
    M, r = wl.M, wl.rank
    units = []
    for g in groups:
        ins = [inputs[i] for i in g]
        packed = q.stack_weights([i["W"] for i in ins]) if len(g) > 1 else ins[0]["W"]
        w = q.DeviceWeight.from_packed(packed, device=dev)
        Ns, K = [i["N"] for i in ins], ins[0]["K"]
        N = sum(Ns)
        u = {"W": w, "Ns": Ns, "K": K, "N": N, "name": "|".join(wl.linears[i].name for i in g),
             "X": q.bf16_from_bits(ins[0]["X"], device=dev),
             "A": q.bf16_from_bits(np.stack([i["A"] for i in ins]), device=dev),
             "B": q.bf16_from_bits(np.concatenate([i["B"] for i in ins], axis=0), device=dev),
             "dY": q.bf16_from_bits(np.concatenate([i["dY"] for i in ins], axis=1), device=dev)}
        u["Y"] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        u["T"] = torch.empty((M, len(g) * r), dtype=torch.float32, device=dev)
        u["dX"] = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        u["dA"] = torch.empty((len(g), r, K), dtype=torch.float32, device=dev)
        u["dB"] = torch.empty((N, r), dtype=torch.float32, device=dev)
        units.append(u)
    return units


def unit_of_linear(d):
    """A single linear's tensors as a one-projection unit (views, no copies)."""
    return {"W": d["W"], "Ns": [d["N"]], "K": d["K"], "N": d["N"], "X": d["X"], "A": d["A"].unsqueeze(0),
            "B": d["B"], "dY": d["dY"], "Y": d["Y"], "T": d["T"], "dX": d["dX"], "dA": d["dA"].unsqueeze(0),
            "dB": d["dB"]}


def swiglu_leg(q, torch, units, wl, steps, stream):
    """gate|up of the layer with the SwiGLU activation (H = silu(G) U in the
    GEMM epilogue, its derivative in an elementwise pass before the fused
    backward) against the same fused unit without it, on the same weights;
    dH is the gate block of the unit's dY.  Every launch on `stream`."""
    u = next((u for u in units if u["name"] == "gate_proj|up_proj"), None)
    if u is None or u["Ns"][0] != u["Ns"][1]:
        return None
    M, r, alpha, I = wl.M, wl.rank, wl.alpha, u["Ns"][0]
    ws = q.alloc_workspace(q.swiglu_workspace_bytes(u["W"], M, r), u["X"].device)
    H = torch.empty((M, I), dtype=torch.bfloat16, device=u["X"].device)
    GU, T = torch.empty_like(u["Y"]), torch.empty_like(u["T"])
    dH = u["dY"][:, :I].contiguous()

    def plain():
        q.multi_linear_fwd(u["W"], u["Ns"], u["X"], u["A"], u["B"], alpha, Y=u["Y"], T=u["T"], workspace=ws,
                           stream=stream)
        q.multi_linear_bwd(u["W"], u["Ns"], u["X"], u["A"], u["B"], u["T"], u["dY"], alpha, dX=u["dX"],
                           dA=u["dA"], dB=u["dB"], workspace=ws, stream=stream)

    def act():
        q.swiglu_fwd(u["W"], u["X"], u["A"], u["B"], alpha, H=H, GU=GU, T=T, workspace=ws, stream=stream)
        q.swiglu_bwd(u["W"], u["X"], u["A"], u["B"], T, GU, dH, alpha, dX=u["dX"], dA=u["dA"], dB=u["dB"],
                     workspace=ws, stream=stream)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms_plain, ms_act = timed(plain), timed(act)
    assert q.device_error() == 0, "device error in the SwiGLU leg"
    flops = sum(syn.linear_flops(M, u["K"], n, r) for n in u["Ns"])
    # elementwise derivative: reads G, U, dH, writes dG, dU (bf16); the
    # epilogue adds the H store
    grad_bytes = 10 * M * I
    return {"unit": "gate_proj|up_proj + SwiGLU", "M": M, "I": I, "K": u["K"], "rank": r,
            "ms_fwd_bwd": ms_act, "ms_fwd_bwd_without_activation": ms_plain,
            "tflops": flops / (ms_act / 1e3) / 1e12,
            "activation_overhead_us": 1e3 * (ms_act - ms_plain),
            "derivative_pass_bytes": grad_bytes,
            "note": "the overhead is the derivative pass plus the H store in the epilogue"}


def config_leg(q, torch, name, steps, dev):
    """The layer step of another configuration (fused launches where the
    fused call supports them), timed on its own: ms per step, tokens/s,
    algorithmic TFLOP/s and fractions of the peaks."""
    wl = syn.WORKLOADS[name]
    inputs = make_inputs(wl)
    M, r, alpha = wl.M, wl.rank, wl.alpha
    units = make_units(q, torch, wl, inputs, dev, fused_groups(wl))
    ws = q.alloc_workspace(max(q.multi_workspace_bytes(u["W"], u["Ns"], M, r) for u in units), dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        for u in units:
            q.multi_linear_fwd(u["W"], u["Ns"], u["X"], u["A"], u["B"], alpha, Y=u["Y"], T=u["T"], workspace=ws,
                               stream=stream)
        for u in reversed(units):
            q.multi_linear_bwd(u["W"], u["Ns"], u["X"], u["A"], u["B"], u["T"], u["dY"], alpha, dX=u["dX"],
                               dA=u["dA"], dB=u["dB"], workspace=ws, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    assert q.device_error() == 0, f"device error in the {name} leg"
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    flops = sum(syn.linear_flops(M, l.K, l.N, r) for l in wl.linears)
    peaks = measured_peaks()
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": f"{name}_layer", "format": wl.fmt, "M": M, "rank": r, "alpha": alpha,
            "launch_units": [u["name"] for u in units], "ms_per_step": ms, "tokens_per_s": M / (ms / 1e3),
            "tflops": tf, "frac_of_nominal_2250": tf / NOMINAL_BF16_TFLOPS, "frac_of_measured_burst": tf / peaks["bf16"]}


def make_inputs(wl):
    return [syn.make_linear_inputs(wl, i, seed=0) for i in range(len(wl.linears))]


def run_reference(args, wl):
    rank, world, _ = dist_init(args.gpus)
    if rank != 0:
        return
    inputs = make_inputs(wl)
    rows = 16
    for _ in range(args.warmup):
        oracle_step(inputs, rows)
    t = time_oracle(inputs, rows, reps=args.steps)
    value = rows / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"{rows} of {wl.M} rows per step, all {len(wl.linears)} linears fwd+bwd, "
                                   f"block decode of every base weight included"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(wl):
    return {"workload": f"{wl.name}_layer", "format": wl.fmt + ("+dq" if wl.double_quant else ""), "M": wl.M,
            "rank": wl.rank, "alpha": wl.alpha,
            "linears": [f"{l.name}:{l.K}->{l.N}" for l in wl.linears],
            "step": "fwd of the 7 linears, then bwd in reverse order; the projections that read the same input "
                    "(q|k|v, gate|up) run as one fused launch each way, and their input gradients come out summed, "
                    "as the decoder layer consumes them (see unfused_layer for every linear on its own)",
            "l2": "per-step working set (weights + activations) > 1 GB, larger than the 129 MB L2; no flush",
            "parallelism": "replicas"}


def main():
    args = parse_args()
    wl = syn.WORKLOADS[args.workload]
    if args.case:
        return run_case(args)
    if args.only_moe:
        import torch

        import quantized_base_lora_block_gb300 as q

        q.load()
        stream = torch.cuda.Stream()
        print(json.dumps(moe_leg(q, torch, args.steps, stream)))
        return
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch

    import quantized_base_lora_block_gb300 as q

    rank, world, local = dist_init(args.gpus)
    torch.cuda.set_device(local)
    q.load()
    dev = torch.device("cuda", local)
    inputs = make_inputs(wl)
    M, r, alpha = wl.M, wl.rank, wl.alpha
    L = []
    for inp in inputs:
        w = q.DeviceWeight.from_packed(inp["W"], device=dev)
        d = {"W": w, "K": inp["K"], "N": inp["N"]}
        for k in ("X", "A", "B", "dY"):
            d[k] = q.bf16_from_bits(inp[k], device=dev)
        d["Y"] = torch.empty((M, inp["N"]), dtype=torch.bfloat16, device=dev)
        d["T"] = torch.empty((M, r), dtype=torch.float32, device=dev)
        d["dX"] = torch.empty((M, inp["K"]), dtype=torch.bfloat16, device=dev)
        d["dA"] = torch.empty((r, inp["K"]), dtype=torch.float32, device=dev)
        d["dB"] = torch.empty((inp["N"], r), dtype=torch.float32, device=dev)
        L.append(d)
    # The step's units: fused launches for the projections that share an
    # input (q|k|v, gate|up), each other linear on its own; the unfused step
    # runs every linear on its own.
    units = make_units(q, torch, wl, inputs, dev, fused_groups(wl))
    units_u = [unit_of_linear(d) for d in L]
    ws_bytes = max(q.multi_workspace_bytes(u["W"], u["Ns"], M, r) for u in units + units_u)
    ws = q.alloc_workspace(ws_bytes, dev)
    for d in L:
        d["ws"] = ws
    stream = torch.cuda.current_stream(dev)

    def step_units_on(us, st):
        for u in us:
            q.multi_linear_fwd(u["W"], u["Ns"], u["X"], u["A"], u["B"], alpha, Y=u["Y"], T=u["T"], workspace=ws,
                               stream=st)
        for u in reversed(us):
            q.multi_linear_bwd(u["W"], u["Ns"], u["X"], u["A"], u["B"], u["T"], u["dY"], alpha, dX=u["dX"],
                               dA=u["dA"], dB=u["dB"], workspace=ws, stream=st)

    def step_units(us):
        step_units_on(us, stream)

    def step():
        step_units(units)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert q.device_error() == 0, "device error during warm-up"

    # --------------------------------------------------------- timed region
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(1.0)  # let the sampler start before the timed region
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark("t0")
    n0 = q.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = q.launch_count() - n0
    ms = e0.elapsed_time(e1)
    # The same step captured once as a CUDA graph (the calls enqueue only
    # device work, so they capture as they are) and replayed K times.
    graph_res = None
    try:
        cap = torch.cuda.Stream(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step_units_on(units, cap)
        g.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        ms_graph = g0.elapsed_time(g1) / args.steps
        graph_res = {"ms_per_step": ms_graph, "value": M / (ms_graph / 1e3) * world, "unit": "tokens/s",
                     "note": "the step's calls captured once as a CUDA graph and replayed (same kernels)"}
        del g
    except Exception as e:  # capture is an extra, the headline pass above stands
        graph_res = {"error": str(e)[:200]}
    # The same K steps again with CUDA events around every fused-GEMM launch
    # (on the stream it is launched on) for the kernel's own time.  Those
    # events lengthen a step by ~3.6%, so the headline pass above runs
    # without them.
    q.profile_gemm(True)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(args.steps):
        step()
    p1.record(stream)
    torch.cuda.synchronize()
    q.profile_gemm(False)
    ms_prof = p0.elapsed_time(p1)
    # the same layer with every linear launched on its own (input gradients
    # of q, k, v and of gate, up returned separately)
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    u0.record(stream)
    for _ in range(args.steps):
        step_units(units_u)
    u1.record(stream)
    torch.cuda.synchronize()
    ms_unfused = u0.elapsed_time(u1)
    if clocks:
        clocks.mark("t1")
    barrier(world)
    clk = clocks.stop() if clocks else None
    gemm_ms, gemm_n, gemm_flops = q.profile_gemm_read()
    assert q.device_error() == 0, "device error in the timed region"
    ms_max = max_over_ranks(ms, world)

    flops_step = sum(syn.linear_flops(M, l.K, l.N, r) for l in wl.linears)
    t_step = ms_max / args.steps / 1e3
    value = world * M / t_step
    peaks = measured_peaks()
    ach = gemm_flops / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else 0.0
    # The fused GEMM runs inside a region of tens of milliseconds at full
    # clock (see `clocks`), so the burst peak is its denominator; the
    # sustained peak was measured over seconds under the power cap.
    roofline = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16"], "traffic": captured_traffic(wl),
                "kernel": "qgemm_pair_kernel (fused decode + tcgen05 cta_group::2 GEMM + adapter chunk), fwd and dX "
                          "launches",
                "peak_kind": f"{peaks['source']} burst bf16 (of measured)",
                "frac_of_measured_sustained": ach / peaks["bf16_sustained"],
                "frac_of_nominal_2250": ach / NOMINAL_BF16_TFLOPS,
                "launches": gemm_n, "share_of_step": gemm_ms / ms_prof if ms_prof > 0 else None,
                "measured": "CUDA events around each fused-GEMM launch over a second pass of the same K steps"}

    # --------------------------------------------------------- end to end
    # Every step copies its inputs X and dY in from pinned host memory and
    # every result out to pinned host memory: Y after each linear's forward,
    # dX, dA and dB after its backward.  Inputs go on a copy stream into two
    # alternating sets of device buffers; results go out on a third stream as
    # soon as each is written.  A linear's compute waits only for its own
    # inputs and for the previous step's copy-out of the buffers it is about
    # to overwrite, so copies in both directions overlap the computation.
    e2e = None
    if not args.no_e2e:
        pin = lambda t, dt: torch.empty(t.shape, dtype=dt).pin_memory()  # noqa: E731
        U = units
        hX = [pin(u["X"], torch.bfloat16) for u in U]
        hdY = [pin(u["dY"], torch.bfloat16) for u in U]
        for h, u in zip(hX, U):
            h.copy_(u["X"])
        for h, u in zip(hdY, U):
            h.copy_(u["dY"])
        hY = [pin(u["Y"], torch.bfloat16) for u in U]
        hdX = [pin(u["dX"], torch.bfloat16) for u in U]
        hdA = [pin(u["dA"], torch.float32) for u in U]
        hdB = [pin(u["dB"], torch.float32) for u in U]
        nbytes = lambda hs: sum(h.numel() * h.element_size() for h in hs)  # noqa: E731
        h2d = nbytes(hX + hdY)
        d2h = nbytes(hY + hdX + hdA + hdB)
        sets = [[{"X": torch.empty_like(u["X"]), "dY": torch.empty_like(u["dY"])} for u in U] for _ in range(2)]
        copy_stream = torch.cuda.Stream(dev)
        out_stream = torch.cuda.Stream(dev)
        n = len(U)
        ev_x = [[torch.cuda.Event() for _ in range(n)] for _ in range(2)]
        ev_y = [[torch.cuda.Event() for _ in range(n)] for _ in range(2)]
        ev_f = [torch.cuda.Event() for _ in range(n)]     # Y of linear i written
        ev_fout = [torch.cuda.Event() for _ in range(n)]  # Y of linear i copied out
        ev_g = [torch.cuda.Event() for _ in range(n)]     # gradients of linear i written
        ev_out = [torch.cuda.Event() for _ in range(n)]   # gradients of linear i copied out
        used = {"fout": [False] * n, "out": [False] * n}
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_done_used = [False, False]

        def e2e_step(k):
            b = k % 2
            with torch.cuda.stream(copy_stream):
                if ev_done_used[b]:
                    copy_stream.wait_event(ev_done[b])  # step k-2 finished with this set
                for i in range(n):
                    sets[b][i]["X"].copy_(hX[i], non_blocking=True)
                    ev_x[b][i].record(copy_stream)
                for i in reversed(range(n)):
                    sets[b][i]["dY"].copy_(hdY[i], non_blocking=True)
                    ev_y[b][i].record(copy_stream)
            for i, d in enumerate(U):
                stream.wait_event(ev_x[b][i])
                if used["fout"][i]:
                    stream.wait_event(ev_fout[i])  # the previous step's Y of unit i is out
                q.multi_linear_fwd(d["W"], d["Ns"], sets[b][i]["X"], d["A"], d["B"], alpha, Y=d["Y"], T=d["T"],
                                   workspace=ws, stream=stream)
                ev_f[i].record(stream)
                with torch.cuda.stream(out_stream):
                    out_stream.wait_event(ev_f[i])
                    hY[i].copy_(d["Y"], non_blocking=True)
                    ev_fout[i].record(out_stream)
                    used["fout"][i] = True
            for i in reversed(range(n)):
                d = U[i]
                stream.wait_event(ev_y[b][i])
                if used["out"][i]:
                    stream.wait_event(ev_out[i])  # the previous step's dX, dA, dB of unit i are out
                q.multi_linear_bwd(d["W"], d["Ns"], sets[b][i]["X"], d["A"], d["B"], d["T"], sets[b][i]["dY"], alpha,
                                   dX=d["dX"], dA=d["dA"], dB=d["dB"], workspace=ws, stream=stream)
                ev_g[i].record(stream)
                with torch.cuda.stream(out_stream):
                    out_stream.wait_event(ev_g[i])
                    hdX[i].copy_(d["dX"], non_blocking=True)
                    hdA[i].copy_(d["dA"], non_blocking=True)
                    hdB[i].copy_(d["dB"], non_blocking=True)
                    ev_out[i].record(out_stream)
                    used["out"][i] = True
            ev_done[b].record(stream)
            ev_done_used[b] = True

        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize()
        barrier(world)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        g0.record(stream)
        for k in range(args.steps):
            e2e_step(k)
        g1.record(stream)
        t_issue = time.perf_counter() - t0
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(time.perf_counter() - t0, world)
        # one step's copies alone in each direction, for context
        c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        with torch.cuda.stream(copy_stream):
            c0.record(copy_stream)
            for i in range(n):
                sets[0][i]["X"].copy_(hX[i], non_blocking=True)
                sets[0][i]["dY"].copy_(hdY[i], non_blocking=True)
            c1.record(copy_stream)
            for i in range(n):
                hY[i].copy_(U[i]["Y"], non_blocking=True)
                hdX[i].copy_(U[i]["dX"], non_blocking=True)
            c2.record(copy_stream)
        torch.cuda.synchronize()
        e2e = {"value": world * M * args.steps / t_e2e, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "h2d_alone_GBps": h2d / (c0.elapsed_time(c1) / 1e3) / 1e9,
               "d2h_alone_GBps": nbytes(hY + hdX) / (c1.elapsed_time(c2) / 1e3) / 1e9,
               "host_issue_ms_per_step": 1e3 * t_issue / args.steps,
               "compute_stream_ms_per_step": g0.elapsed_time(g1) / args.steps,
               "note": "every step: pinned host X and dY copied in (copy stream, double-buffered), Y, dX, dA "
                       "and dB copied out to pinned host (third stream) as each is written; wall clock"}

    # --------------------------------------------------------- other legs
    stream_res = None
    if args.stream_layers > 0 and wl.name == "llama31_8b_nf4dq":
        stream_res = stream_leg(q, torch, inputs, L, wl, args.stream_layers, 2, stream, ms_max / args.steps)
    moe_res = None
    if not args.no_moe and rank == 0:
        moe_res = moe_leg(q, torch, 10, stream)
    deq_res = lib_res = None
    if rank == 0 and not args.no_context:
        deq_res = dequant_leg(q, torch, L, wl, peaks)
        lib_res = library_leg(q, torch, L, wl, 5)
    swiglu_res = None
    if rank == 0 and not args.no_context:
        swiglu_res = swiglu_leg(q, torch, units, wl, 10, stream)
    cfg_res = None
    if not args.no_configs and rank == 0:
        cfg_res = [config_leg(q, torch, name, 10, dev)
                   for name in ("qwen3_0p6b_bf16", "qwen3_8b_q4_0", "qwen3_8b_q8_0") if name != wl.name]

    # --------------------------------------------------------- CPU oracle
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows = CPU_SAMPLE_ROWS
        t = time_oracle(inputs, rows, reps=2)
        cpu = {"value": rows / t, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{rows} of {M} rows, all {len(wl.linears)} linears fwd+bwd, fp64, block decode of "
                         f"every base weight included; {2 * t:.1f} s for 2 repetitions"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(wl),
            "tflops": flops_step / t_step / 1e12 * world,
            "launch_units": [u["name"] for u in units],
            "unfused_layer": {"ms_per_step": ms_unfused / args.steps,
                              "value": M / (ms_unfused / args.steps / 1e3), "unit": "tokens/s",
                              "tflops": flops_step / (ms_unfused / args.steps / 1e3) / 1e12,
                              "note": "the same 7 linears, each launched on its own (q, k, v and gate, up input "
                                      "gradients returned separately)"},
            "frac_of_nominal_2250": flops_step / t_step / 1e12 / NOMINAL_BF16_TFLOPS,
            "frac_of_measured_burst": flops_step / t_step / 1e12 / peaks["bf16"],
            "frac_of_measured_sustained": flops_step / t_step / 1e12 / peaks["bf16_sustained"],
            "target": {"what": "whole fwd+bwd step >= 60% of 2.25 PFLOP/s dense bf16",
                       "needed_tflops": 0.6 * NOMINAL_BF16_TFLOPS,
                       "met": flops_step / t_step / 1e12 >= 0.6 * NOMINAL_BF16_TFLOPS},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clk, "stream": stream_res, "moe": moe_res, "configs": cfg_res,
            "dequant_blocks": deq_res, "library_baseline": lib_res, "swiglu": swiglu_res, "graph": graph_res,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
