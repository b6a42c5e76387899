"""dequant_blocks on the GPU against the oracle's block decode: bit-exact."""
import numpy as np
import pytest

import oracle
import qlora_synth as syn

pytestmark = pytest.mark.gpu


def _gpu_dequant(lib, packed):
    w = lib.DeviceWeight.from_packed(packed)
    out = lib.dequant_blocks(w)
    import torch

    torch.cuda.synchronize()
    return lib.bits_from_bf16(out)


def _assert_bits_equal(got, want, name):
    got = got.reshape(want.shape)
    # compare by value so that -0 == +0 (bf16 bits 0x8000 vs 0x0000)
    gv = oracle.bf16_bits_to_f64(got)
    wv = oracle.bf16_bits_to_f64(want)
    bad = (gv != wv) & ~(np.isnan(gv) & np.isnan(wv))  # NaN codes decode to some NaN
    assert not bad.any(), f"{name}: {int(bad.sum())} mismatches, first at {np.argwhere(bad)[0]}"


def _nf4_all_codes(N=64, K=256, seed=0, dq=False):
    rng = np.random.default_rng(seed)
    codes = np.tile(np.arange(16, dtype=np.uint8), N * K // 16)
    rng.shuffle(codes)
    packed = ((codes[0::2] << 4) | codes[1::2]).astype(np.uint8)
    nb = N * K // 64
    p = {"fmt": "nf4", "N": N, "K": K, "data": packed}
    if dq:
        p["absmax_q"] = rng.integers(0, 128, nb).astype(np.int8)
        p["absmax_scale"] = (rng.random((nb + 255) // 256) * 0.01).astype(np.float32)
        p["dq_group"] = 256
    else:
        p["absmax"] = (rng.random(nb) * 0.1).astype(np.float32)
        p["absmax"][:3] = [0.0, 1.0, 3.0e-5]
    return p


@pytest.mark.parametrize("dq", [False, True])
def test_nf4_every_code_bit_exact(lib, dq):
    p = _nf4_all_codes(N=128, K=512, dq=dq)
    _assert_bits_equal(_gpu_dequant(lib, p), oracle.dequant_bf16_bits(p), "nf4")


def test_q4_0_every_nibble_bit_exact(lib):
    rng = np.random.default_rng(1)
    N, K = 64, 256
    nb = N * K // 32
    blocks = np.empty((nb, 18), dtype=np.uint8)
    d = (rng.standard_normal(nb) * 0.003).astype(np.float16)
    d[:4] = [0.0, -0.0, 1.0, 6.0e-5]  # zero scale, negative zero, a subnormal-ish fp16
    blocks[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    blocks[:, 2:] = rng.integers(0, 256, (nb, 16), dtype=np.uint8)
    blocks[0, 2:] = np.arange(16, dtype=np.uint8) * 17  # every nibble in both halves
    p = {"fmt": "q4_0", "N": N, "K": K, "data": blocks.reshape(-1)}
    _assert_bits_equal(_gpu_dequant(lib, p), oracle.dequant_bf16_bits(p), "q4_0")


def test_q8_0_every_code_bit_exact(lib):
    rng = np.random.default_rng(2)
    N, K = 64, 512
    nb = N * K // 32
    blocks = np.empty((nb, 34), dtype=np.uint8)
    d = (rng.standard_normal(nb) * 0.003).astype(np.float16)
    d[:3] = [0.0, 2.0 ** -24, -1.5]
    blocks[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    blocks[:, 2:] = rng.integers(0, 256, (nb, 32), dtype=np.uint8)
    codes = np.arange(256, dtype=np.uint8)  # all 256 int8 codes incl. -128
    blocks[8:16, 2:] = codes.reshape(8, 32)
    p = {"fmt": "q8_0", "N": N, "K": K, "data": blocks.reshape(-1)}
    _assert_bits_equal(_gpu_dequant(lib, p), oracle.dequant_bf16_bits(p), "q8_0")


def test_fp8_every_code_bit_exact(lib):
    """All 256 E4M3 codes (NaN included) under several tensor scales, one
    per launch: a normal, a power of two, a large and a tiny one."""
    rng = np.random.default_rng(5)
    N, K = 64, 512
    codes = np.tile(np.arange(256, dtype=np.uint8), N * K // 256)
    rng.shuffle(codes)
    for ts in (0.0173, 0.25, 3.0e4, 1.0e-30):
        p = {"fmt": "fp8_e4m3", "N": N, "K": K, "data": codes, "tensor_scale": np.array([ts], np.float32)}
        _assert_bits_equal(_gpu_dequant(lib, p), oracle.dequant_bf16_bits(p), f"fp8 scale {ts}")


def test_nvfp4_every_code_bit_exact(lib):
    """All 16 E2M1 codes in every block, block scales over every finite E4M3
    code of either sign (subnormals and zero included)."""
    rng = np.random.default_rng(6)
    N, K = 128, 512
    nblk = N * K // 16
    codes = np.tile(np.arange(16, dtype=np.uint8), N * K // 16)
    for b in range(nblk):
        rng.shuffle(codes[16 * b:16 * (b + 1)])
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    bsc = np.resize(finite, nblk)
    rng.shuffle(bsc)
    for ts in (1.0, 0.0123, 2.0 ** -100):
        p = {"fmt": "nvfp4", "N": N, "K": K, "data": (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8),
             "block_scale": bsc, "tensor_scale": np.array([ts], np.float32)}
        _assert_bits_equal(_gpu_dequant(lib, p), oracle.dequant_bf16_bits(p), f"nvfp4 scale {ts}")


def test_q4_k_random_bytes_bit_exact(lib):
    """Super-blocks of random bytes (every scale/min bit pattern and code)
    with finite fp16 d and dmin of either sign, zero and subnormal ones."""
    rng = np.random.default_rng(7)
    N, K = 64, 1024
    nsb = N * K // 256
    rec = rng.integers(0, 256, (nsb, 144), dtype=np.uint8)
    d = (rng.standard_normal((nsb, 2)) * 0.01).astype(np.float16)
    d[:4] = [[0.0, 0.0], [-0.0, 1.0], [6.0e-8, -3.0e-5], [65000.0, -0.5]]
    rec[:, 0:4] = d.view(np.uint8).reshape(nsb, 4)
    p = {"fmt": "q4_k", "N": N, "K": K, "data": rec.reshape(-1)}
    _assert_bits_equal(_gpu_dequant(lib, p), oracle.dequant_bf16_bits(p), "q4_k")


def test_nf4_absmax_map_bit_exact(lib):
    """NF4 with an 8-bit absmax map and offset: every absmax byte, every
    NF4 code."""
    rng = np.random.default_rng(8)
    p = _nf4_all_codes(N=128, K=512, dq=True)
    nb = 128 * 512 // 64
    p["absmax_q"] = np.resize(np.arange(256, dtype=np.uint8), nb).view(np.int8)
    p["absmax_map"] = (rng.standard_normal(256) * 0.5).astype(np.float32)
    p["absmax_offset"] = 0.0371
    _assert_bits_equal(_gpu_dequant(lib, p), oracle.dequant_bf16_bits(p), "nf4 map")


@pytest.mark.parametrize("fmt,dq", [("nf4", False), ("nf4", True), ("q4_0", False), ("q8_0", False),
                                    ("bf16", False), ("q4_k", False), ("fp8_e4m3", False), ("nvfp4", False),
                                    ("nf4_dqmap", False)])
def test_packed_normal_weights_bit_exact(lib, fmt, dq):
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((192, 1024)) * 0.02).astype(np.float32)
    w[5, :64] = 0.0  # an all-zero block
    p = syn.pack(w, fmt, double_quant=dq)
    _assert_bits_equal(_gpu_dequant(lib, p), oracle.dequant_bf16_bits(p), fmt)


@pytest.mark.slow
@pytest.mark.parametrize("fmt,dq,N,K", [("nf4", True, 14336, 4096), ("q4_0", False, 12288, 4096),
                                        ("q8_0", False, 4096, 12288), ("q4_k", False, 12288, 4096),
                                        ("fp8_e4m3", False, 14336, 4096), ("nvfp4", False, 4096, 14336)])
def test_full_size_layer_weight_bit_exact(lib, fmt, dq, N, K):
    """A full gate/down projection of the 8B-class layers."""
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    p = syn.pack(w, fmt, double_quant=dq)
    _assert_bits_equal(_gpu_dequant(lib, p), oracle.dequant_bf16_bits(p), fmt)
