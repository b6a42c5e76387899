"""Layer streaming: the frozen base of each layer lives in pinned host memory
and is copied into a 2-slot device pool one layer ahead on the library's copy
stream.  Streamed results must be bitwise equal to resident results of the
same kernels (the bit-exactness protocol of the Soup show post), forward over
layers 0..L-1, then backward L-1..0.  Misuse of the pool is rejected on the
host."""
import numpy as np
import pytest

import qlora_synth as syn

pytestmark = pytest.mark.gpu

L_LAYERS = 6


def _layers():
    wl = syn.Workload("stream", "nf4", True, 192, 16, 16.0, [syn.Linear("l", 512, 768)])
    return [syn.make_linear_inputs(wl, 0, seed=0, layer=i) for i in range(L_LAYERS)]


def _resident(lib, layers, X, A, B, dY):
    import torch

    out = []
    for i, inp in enumerate(layers):
        w = lib.DeviceWeight.from_packed(inp["W"])
        Y, T = lib.linear_fwd(w, X[i], A[i], B[i], inp["alpha"])
        out.append({"Y": Y, "T": T})
    for i in reversed(range(len(layers))):
        w = lib.DeviceWeight.from_packed(layers[i]["W"])
        dX, dA, dB = lib.linear_bwd(w, X[i], A[i], B[i], out[i]["T"], dY[i], layers[i]["alpha"])
        out[i].update(dX=dX, dA=dA, dB=dB)
    torch.cuda.synchronize()
    return out


def _streamed(lib, layers, X, A, B, dY):
    import torch

    blobs = [lib.pack_weight_blob(inp["W"]) for inp in layers]
    pinned = [torch.from_numpy(b).pin_memory() for b, _ in blobs]
    slot = max(b.nbytes for b, _ in blobs)
    pool = lib.LayerStream(2, slot)
    out = [dict() for _ in layers]
    n = len(layers)
    pool.prefetch(0, pinned[0])
    for i in range(n):                       # forward 0 .. n-1
        if i + 1 < n:
            pool.prefetch(i + 1, pinned[i + 1])
        base = pool.acquire(i)
        w = lib.weight_in_slot(layers[i]["W"], blobs[i][1], base)
        Y, T = lib.linear_fwd(w, X[i], A[i], B[i], layers[i]["alpha"])
        pool.release(i)
        out[i].update(Y=Y, T=T)
    for i in reversed(range(n)):             # backward n-1 .. 0
        pool.prefetch(i, pinned[i])          # resident already for the last two
        if i - 1 >= 0:
            pool.prefetch(i - 1, pinned[i - 1])
        base = pool.acquire(i)
        w = lib.weight_in_slot(layers[i]["W"], blobs[i][1], base)
        dX, dA, dB = lib.linear_bwd(w, X[i], A[i], B[i], out[i]["T"], dY[i], layers[i]["alpha"])
        pool.release(i)
        out[i].update(dX=dX, dA=dA, dB=dB)
    torch.cuda.synchronize()
    pool.close()
    return out


def test_streamed_equals_resident_bitwise(lib):
    layers = _layers()
    X = [lib.bf16_from_bits(l["X"]) for l in layers]
    A = [lib.bf16_from_bits(l["A"]) for l in layers]
    B = [lib.bf16_from_bits(l["B"]) for l in layers]
    dY = [lib.bf16_from_bits(l["dY"]) for l in layers]
    res = _resident(lib, layers, X, A, B, dY)
    st = _streamed(lib, layers, X, A, B, dY)
    assert lib.device_error() == 0
    import torch

    for i in range(len(layers)):
        for k in ("Y", "T", "dX", "dA", "dB"):
            a = res[i][k].contiguous().view(torch.uint8).cpu().numpy()
            b = st[i][k].contiguous().view(torch.uint8).cpu().numpy()
            assert np.array_equal(a, b), f"layer {i} {k}: streamed differs from resident"


def test_pool_rejects_misuse(lib):
    import torch

    pool = lib.LayerStream(2, 4096)
    buf = [torch.zeros(1024, dtype=torch.uint8).pin_memory() for _ in range(3)]
    with pytest.raises(lib.QloraError) as e:
        pool.acquire(5)                       # never prefetched
    assert e.value.status == -7
    pool.prefetch(0, buf[0])
    pool.prefetch(1, buf[1])
    pool.acquire(0)
    pool.acquire(1)
    with pytest.raises(lib.QloraError) as e:
        pool.prefetch(2, buf[2])              # both slots held by compute
    assert e.value.status == -7
    pool.release(0)
    pool.prefetch(2, buf[2])                  # slot of layer 0 is reused
    with pytest.raises(lib.QloraError) as e:
        pool.acquire(0)                       # layer 0 was overwritten
    assert e.value.status == -7
    with pytest.raises(lib.QloraError) as e:
        pool.release(9)
    assert e.value.status == -7
    big = torch.zeros(8192, dtype=torch.uint8).pin_memory()
    with pytest.raises(lib.QloraError) as e:
        pool.prefetch(3, big)                 # larger than a slot
    assert e.value.status == -1
    pool.release(1)
    torch.cuda.synchronize()
    pool.close()


def test_refill_waits_for_every_stream_that_released(lib):
    """One layer acquired on two unordered streams and released from both:
    the next refill of its slot must wait for the work of both releases,
    not only the last one.  The first stream's read of the slot is delayed
    by a device-side sleep, so a refill that waited only for the second
    stream would land before that read and change its result."""
    import torch

    wl = syn.Workload("refill", "q8_0", False, 64, 16, 32.0, [syn.Linear("l", 1024, 2048)])
    l0 = syn.make_linear_inputs(wl, 0, seed=1, layer=0)
    l1 = syn.make_linear_inputs(wl, 0, seed=2, layer=1)
    b0, o0 = lib.pack_weight_blob(l0["W"])
    b1, o1 = lib.pack_weight_blob(l1["W"])
    h0, h1 = torch.from_numpy(b0).pin_memory(), torch.from_numpy(b1).pin_memory()
    want = lib.dequant_blocks(lib.DeviceWeight.from_packed(l0["W"]))
    pool = lib.LayerStream(1, max(b0.nbytes, b1.nbytes))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    pool.prefetch(0, h0)
    base1 = pool.acquire(0, s1)
    base2 = pool.acquire(0, s2)
    w1 = lib.weight_in_slot(l0["W"], o0, base1)
    w2 = lib.weight_in_slot(l0["W"], o0, base2)
    out1 = torch.empty_like(want)
    out2 = torch.empty_like(want)
    with torch.cuda.stream(s1):
        torch.cuda._sleep(200_000_000)        # ~0.1 s of device time before the read
    lib.dequant_blocks(w1, out=out1, stream=s1)
    pool.release(0, s1)
    lib.dequant_blocks(w2, out=out2, stream=s2)
    pool.release(0, s2)
    pool.prefetch(1, h1)                      # refills the only slot
    base = pool.acquire(1)
    torch.cuda.current_stream().wait_stream(s1)
    torch.cuda.current_stream().wait_stream(s2)
    got1 = lib.dequant_blocks(lib.weight_in_slot(l1["W"], o1, base), out=torch.empty_like(want))
    pool.release(1)
    torch.cuda.synchronize()
    pool.close()
    assert torch.equal(out1.view(torch.int16), want.view(torch.int16)), "slow stream read the refilled slot"
    assert torch.equal(out2.view(torch.int16), want.view(torch.int16))
    assert torch.equal(got1.view(torch.int16),
                       lib.dequant_blocks(lib.DeviceWeight.from_packed(l1["W"])).view(torch.int16))
