"""The seeded input generator: determinism, shapes, and workload statistics."""
import numpy as np

import qlora_synth as syn


def test_same_seed_same_bytes():
    wl = syn.WORKLOADS["tiny_nf4"]
    a = syn.make_linear_inputs(wl, 0, seed=0)
    b = syn.make_linear_inputs(wl, 0, seed=0)
    for k in ("X", "A", "B", "dY"):
        assert np.array_equal(a[k], b[k])
    assert np.array_equal(a["W"]["data"], b["W"]["data"])
    c = syn.make_linear_inputs(wl, 0, seed=1)
    assert not np.array_equal(a["X"], c["X"])


def test_shapes_and_distributions():
    wl = syn.WORKLOADS["tiny_nf4"]
    d = syn.make_linear_inputs(wl, 0, seed=0, with_w_f32=True)
    assert d["X"].shape == (64, 256) and d["A"].shape == (8, 256) and d["B"].shape == (256, 8)
    x = syn.bf16_bits_to_f32(d["X"])
    assert abs(x.std() - 1.0) < 0.05
    assert abs(d["w_f32"].std() - 0.02) < 0.002
    a = syn.bf16_bits_to_f32(d["A"])
    assert abs(a.std() - 1 / 16) < 0.01
    w = d["W"]
    assert w["data"].size == 256 * 256 // 2 and w["absmax"].size == 256 * 256 // 64


def test_moe_routing_statistics():
    off, tok, counts = syn.moe_routing()
    assert off[-1] == 4096 * 8 and off.size == 129
    assert counts.min() == 0 and (counts == 0).sum() >= 4
    assert 400 <= counts.max() <= 800
    assert np.all(np.diff(off) >= 0)
    # rows of one expert are sorted by token index
    for e in range(128):
        t = tok[off[e]:off[e + 1]]
        assert np.all(np.diff(t) > 0)
