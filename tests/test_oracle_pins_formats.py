"""Pins of the oracle's decoders for the further base formats: GGUF Q4_K,
FP8 E4M3 with a tensor scale, NVFP4 (E2M1 with E4M3 block scales and a tensor
scale) and NF4 with a QLoRA-style 8-bit absmax map.

Each decoder is tied to something other than itself: PyTorch's E4M3
conversion (a library routine), hand-worked blocks, the reduction of one
format to another already pinned one, and round trips through the input
generator's independently written packers.
"""
import numpy as np
import pytest

import oracle
import qlora_synth as syn

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------
# E4M3 and E2M1 value sets
# ---------------------------------------------------------------------------
def test_e4m3_matches_torch_for_every_code():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_value(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))  # -0 at 0x80


def test_e2m1_embeds_in_e4m3():
    """Every E2M1 value is the E4M3 value with the same sign, mantissa bit
    and unbiased exponent (bias 1 vs bias 7; the E2M1 subnormal 0.5 is the
    E4M3 normal 2^-1), read through PyTorch's E4M3 conversion."""
    torch = pytest.importorskip("torch")
    got = oracle.e2m1_value(np.arange(16, dtype=np.uint8))
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        if e == 0 and m == 0:
            want = -0.0 if s else 0.0
        else:
            ue = (e - 1) if e else -1  # unbiased exponent (subnormal 0.5 = 2^-1)
            e4 = (s << 7) | ((ue + 7) << 3) | ((m << 2) if e else 0)
            want = float(torch.tensor([e4], dtype=torch.uint8).view(torch.float8_e4m3fn).double()[0])
        assert got[c] == want and np.signbit(got[c]) == np.signbit(want), (c, got[c], want)
    assert sorted(set(np.abs(got).tolist())) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ---------------------------------------------------------------------------
# FP8 E4M3 with a tensor scale
# ---------------------------------------------------------------------------
def test_fp8_hand_worked():
    # codes: 1.0, 448, 2^-9 (smallest subnormal), -1.875, -0, 0.5
    codes = np.array([0x38, 0x7E, 0x01, 0xBF, 0x80, 0x30, 0x38, 0x38], dtype=np.uint8)
    w = {"fmt": "fp8_e4m3", "N": 1, "K": 8, "data": codes, "tensor_scale": np.array([0.75], np.float32)}
    got = oracle.dequant(w).reshape(-1)
    want = [0.75, 336.0, 0.75 * 2.0 ** -9, -1.40625, -0.0, 0.375, 0.75, 0.75]
    assert got.tolist() == want
    assert np.signbit(got[4])
    # fp32 product, then bf16: 1.875 * 1.1f = 2.0625000447 -> bf16 2.0625
    w["data"] = np.full(8, 0x3F, np.uint8)
    w["tensor_scale"] = np.array([1.1], np.float32)
    assert np.all(oracle.dequant(w) == 2.0625)


def test_fp8_round_trips_through_packer():
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]          # no NaN codes
    codes = codes[codes != 0x80]                      # -0 packs as +0
    codes = codes[:-1]                                # an even count (drops -448)
    w = {"fmt": "fp8_e4m3", "N": 2, "K": codes.size // 2, "data": codes,
         "tensor_scale": np.array([1.0], np.float32)}
    dec = oracle.dequant(w).astype(np.float32)       # every E4M3 value is a bf16 value
    re = syn.pack_fp8_e4m3(dec)
    assert re["tensor_scale"][0] == 1.0              # largest |value| is 448
    assert np.array_equal(re["data"], codes)


# ---------------------------------------------------------------------------
# NVFP4
# ---------------------------------------------------------------------------
def _nvfp4(codes, block_codes, ts):
    codes = np.asarray(codes, np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    return {"fmt": "nvfp4", "N": 1, "K": codes.size, "data": packed,
            "block_scale": np.asarray(block_codes, np.uint8), "tensor_scale": np.array([ts], np.float32)}


def test_nvfp4_hand_worked():
    # block 0: scale code 0x30 (0.5) x tensor scale 3 -> factor 1.5, codes 0..15
    # block 1: scale code 0x01 (2^-9, the smallest subnormal) x 3, codes 15..0
    codes = np.concatenate([np.arange(16), np.arange(15, -1, -1)]).astype(np.uint8)
    w = _nvfp4(codes, [0x30, 0x01], 3.0)
    got = oracle.dequant(w).reshape(-1)
    mags = np.array([0, 0.75, 1.5, 2.25, 3.0, 4.5, 6.0, 9.0])
    assert got[:16].tolist() == np.concatenate([mags, -mags]).tolist()
    assert np.signbit(got[8])                         # code 8 is -0
    f = 2.0 ** -9 * 3.0
    want1 = np.concatenate([mags / 1.5, -mags / 1.5])[::-1] * f
    assert got[16:].tolist() == want1.tolist()
    # nibble order: element 0 in the low nibble of byte 0
    assert (w["data"][0] & 0x0F) == 0 and (w["data"][0] >> 4) == 1


def test_nvfp4_round_trips_through_packer():
    rng = np.random.default_rng(5)
    nblk = 24
    codes = rng.integers(0, 16, size=(nblk, 16)).astype(np.uint8)
    codes[codes == 8] = 0                             # -0 packs as +0
    codes[:, 3] = 7                                   # each block holds +6 (its max)
    bsc = rng.integers(0x08, 0x7E, size=nblk).astype(np.uint8)   # positive normal scales
    bsc[0] = 0x7E                                     # 448: tensor max 6 * 448, tensor scale 1
    w = _nvfp4(codes.reshape(-1), bsc, 1.0)
    dec = oracle.dequant(w).astype(np.float32)
    re = syn.pack_nvfp4(dec)
    assert re["tensor_scale"][0] == 1.0
    assert np.array_equal(re["block_scale"], bsc)
    assert np.array_equal(re["data"], w["data"])


# ---------------------------------------------------------------------------
# Q4_K
# ---------------------------------------------------------------------------
def test_q4_k_scale_unpack_hand_worked():
    # sub-blocks 0..3: bytes 0..3 low 6 bits = scales 1, 2, 3, 4; bytes 4..7
    # low 6 bits = mins 5, 6, 7, 8.  Sub-blocks 4..7: low nibbles from bytes
    # 8..11 (scale | min << 4) and top bits from bytes 0..3 (scales) and 4..7
    # (mins): scale 4 = 0x9 | 1 << 4 = 25, min 4 = 0x2 | 3 << 4 = 50, ...
    b = np.array([[1 | (1 << 6), 2 | (0 << 6), 3 | (2 << 6), 4 | (3 << 6),
                   5 | (3 << 6), 6 | (1 << 6), 7 | (0 << 6), 8 | (2 << 6),
                   0x29, 0x5A, 0x6B, 0x7C]], dtype=np.uint8)
    sc, mn = oracle.q4_k_scale_min(b)
    assert sc[0].tolist() == [1, 2, 3, 4, 0x9 | (1 << 4), 0xA | (0 << 4), 0xB | (2 << 4), 0xC | (3 << 4)]
    assert mn[0].tolist() == [5, 6, 7, 8, 0x2 | (3 << 4), 0x5 | (1 << 4), 0x6 | (0 << 4), 0x7 | (2 << 4)]


def _q4_k_record(d, dmin, sc, mn, nib):
    """One super-block from its parts (nib: 256 codes in element order)."""
    rec = np.zeros(144, np.uint8)
    rec[0:2] = np.array([d], np.float16).view(np.uint8)
    rec[2:4] = np.array([dmin], np.float16).view(np.uint8)
    sc, mn = np.asarray(sc), np.asarray(mn)
    for j in range(4):
        rec[4 + j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        rec[8 + j] = mn[j] | ((mn[j + 4] >> 4) << 6)
        rec[12 + j] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    n = np.asarray(nib, np.uint8).reshape(4, 2, 32)
    rec[16:] = (n[:, 0, :] | (n[:, 1, :] << 4)).reshape(-1)
    return rec


def test_q4_k_hand_worked():
    d, dmin = 0.5, 0.25
    sc = [1, 2, 3, 4, 5, 6, 7, 7]      # small enough that every value is a bf16 value
    mn = [0, 1, 2, 3, 4, 5, 6, 7]
    nib = np.arange(256) % 16
    w = {"fmt": "q4_k", "N": 1, "K": 256, "data": _q4_k_record(d, dmin, sc, mn, nib)}
    got = oracle.dequant(w).reshape(-1)
    # element e is in sub-block e // 32 with code e % 16
    for e in (0, 15, 31, 32, 47, 100, 200, 224, 239, 255):
        j, q = e // 32, e % 16
        assert got[e] == d * sc[j] * q - dmin * mn[j], e
    assert got[255] == 50.75


def test_q4_k_reduces_to_q4_0():
    """With every sub-block scale 1 and min 8 and d = dmin = D, Q4_K decodes
    to (q - 8) D, which is Q4_0 with the same codes (in Q4_0's own byte
    order) and the same D."""
    rng = np.random.default_rng(2)
    D = np.float16(0.0137)
    nib = rng.integers(0, 16, size=256).astype(np.uint8)
    k = {"fmt": "q4_k", "N": 1, "K": 256,
         "data": _q4_k_record(D, D, [1] * 8, [8] * 8, nib)}
    blocks = np.zeros((8, 18), np.uint8)
    nb = nib.reshape(8, 32)
    blocks[:, 0:2] = np.full(8, D, np.float16).view(np.uint8).reshape(8, 2)
    blocks[:, 2:] = nb[:, :16] | (nb[:, 16:] << 4)
    q40 = {"fmt": "q4_0", "N": 1, "K": 256, "data": blocks.reshape(-1)}
    assert np.array_equal(oracle.dequant(k), oracle.dequant(q40))


def test_q4_k_decodes_parts_packed_independently():
    """Super-blocks built from known parts (d, dmin, 6-bit scales and mins
    up to 63, codes): the input generator's packer, given the exact values
    d sc q - dmin m, writes the same bytes as the test's record builder, and
    the oracle decodes those bytes to bf16 of the same exact values."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    recs, exact = [], []
    for _ in range(6):
        d = np.float16(2.0 ** -int(rng.integers(8, 12)))
        dmin = np.float16(2.0 ** -int(rng.integers(8, 12)))
        sc = rng.integers(1, 64, size=8)
        mn = rng.integers(0, 64, size=8)
        sc[rng.integers(0, 8)] = 63                  # largest scale / min pins d / dmin
        mn[rng.integers(0, 8)] = 63
        nib = rng.integers(0, 16, size=(8, 32))
        nib[:, 0], nib[:, 1] = 0, 15                 # every sub-block spans its range
        recs.append(_q4_k_record(d, dmin, sc, mn, nib.reshape(-1)))
        exact.append((float(d) * sc[:, None] * nib - float(dmin) * mn[:, None]).reshape(-1))
    data = np.concatenate(recs)
    x = np.concatenate(exact).reshape(2, 768)
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x)   # exact in fp32
    assert np.array_equal(syn.pack_q4_k(x.astype(np.float32))["data"], data)
    w = {"fmt": "q4_k", "N": 2, "K": 768, "data": data}
    want = torch.from_numpy(x.astype(np.float32)).bfloat16().double().numpy()
    assert np.array_equal(oracle.dequant(w), want)


def test_q4_k_pack_error_bound():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((4, 512)).astype(np.float32) * 0.02
    dec = oracle.dequant(syn.pack_q4_k(x))
    span = x.reshape(-1, 32).max(axis=1) - np.minimum(x.reshape(-1, 32).min(axis=1), 0)
    err = np.abs(dec - x).reshape(-1, 32).max(axis=1)
    assert np.all(err <= 0.1 * span + 1e-6)


# ---------------------------------------------------------------------------
# NF4 with a QLoRA-style 8-bit absmax map
# ---------------------------------------------------------------------------
def _nf4_codes_block(K):
    codes = np.full(K, 15, dtype=np.uint8)
    codes[1::2] = 0
    return ((codes[0::2] << 4) | codes[1::2]).astype(np.uint8)


def test_dq_map_linear_map_reduces_to_int8_dq():
    """The map i -> int8(i) with offset 0 is the plain int8 double
    quantisation (pinned separately)."""
    K = 64 * 512
    packed = _nf4_codes_block(K)
    q = (np.arange(512) % 128).astype(np.int8)
    scale2 = np.array([0.001, 0.25], dtype=np.float32)
    plain = {"fmt": "nf4", "N": 1, "K": K, "data": packed, "absmax_q": q, "absmax_scale": scale2,
             "dq_group": 256}
    lin = np.arange(256).astype(np.uint8).view(np.int8).astype(np.float32)
    mapped = dict(plain, absmax_map=lin, absmax_offset=0.0)
    assert np.array_equal(oracle.dequant(mapped), oracle.dequant(plain))


def test_dq_map_hand_worked():
    # map[5] = 0.5, map[200] = -0.25; scale2 = 3, offset = 0.25:
    # absmax' = 0.5 * 3 + 0.25 = 1.75 and -0.25 * 3 + 0.25 = -0.5
    K = 128
    amap = np.zeros(256, np.float32)
    amap[5], amap[200] = 0.5, -0.25
    w = {"fmt": "nf4", "N": 1, "K": K, "data": _nf4_codes_block(K),
         "absmax_q": np.array([5, 200], np.uint8).view(np.int8), "absmax_scale": np.array([3.0], np.float32),
         "dq_group": 256, "absmax_map": amap, "absmax_offset": 0.25}
    got = oracle.dequant(w).reshape(2, 64)
    assert got[0, 0] == 1.75 and got[0, 1] == -1.75      # codes 15 (+1) and 0 (-1)
    assert got[1, 0] == -0.5 and got[1, 1] == 0.5


def test_dq_map_pack_decode_error_bound():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 64 * 64)).astype(np.float32) * 0.02
    p = syn.pack_nf4(x, double_quant=True, dq_map=True)
    amax = np.abs(x.reshape(-1, 64)).max(axis=1)
    dec_amax = np.abs(oracle.dequant(dict(p, data=_nf4_codes_block(x.size))).reshape(-1, 64)[:, 0])
    # the E4M3 map has 3 mantissa bits (half a step: 1/16 of the centred
    # value), then the decoded value is read back through bf16 (2^-9)
    assert np.all(np.abs(dec_amax - amax) <= 0.07 * np.abs(amax - p["absmax_offset"]) + 2.0 ** -8 * amax)
    assert np.abs(oracle.dequant(p) - x).max() < 0.25 * amax.max()


# ---------------------------------------------------------------------------
# gate / up with SwiGLU
# ---------------------------------------------------------------------------
def test_swiglu_hand_worked():
    # G = [0, 2, -1], U = [3, 1, 2]: H = silu(G) U = [0, 2 s(2), -2 s(-1)]
    G = np.array([[0.0, 2.0, -1.0]])
    U = np.array([[3.0, 1.0, 2.0]])
    dH = np.array([[1.0, 1.0, 0.5]])
    dG, dU = oracle.swiglu_grad_gate_up(G, U, dH)
    s = lambda x: 1.0 / (1.0 + np.exp(-x))  # noqa: E731
    # d silu / dg at 0 is 1/2; at g: s(g) + g s(g) (1 - s(g))
    assert dG[0, 0] == 1.5
    assert np.isclose(dG[0, 1], 1.0 * (s(2.0) + 2.0 * s(2.0) * (1 - s(2.0))), rtol=1e-15)
    assert np.isclose(dG[0, 2], 0.5 * 2.0 * (s(-1.0) - s(-1.0) * (1 - s(-1.0))), rtol=1e-15)
    assert dU.tolist() == [[0.0, 2.0 * s(2.0), -0.5 * s(-1.0)]]


def test_swiglu_forward_hand_worked():
    # K = 1 and B = 0 (the adapters add nothing): G = X Wg^T = [0, 2, -1],
    # U = X Wu^T = [3, 1, 2], H = silu(G) U = [0, 2 s(2), -2 s(-1)], and
    # T = [X Ag^T | X Au^T] = [1 | 1]
    X = np.array([[1.0]])
    Wg = np.array([[0.0], [2.0], [-1.0]])
    Wu = np.array([[3.0], [1.0], [2.0]])
    A = np.array([[1.0]])
    Bz = np.zeros((3, 1))
    H, G, U, T = oracle.swiglu_fwd(X, Wg, Wu, A, A, Bz, Bz, 1.0)
    s = lambda x: 1.0 / (1.0 + np.exp(-x))  # noqa: E731
    assert G.tolist() == [[0.0, 2.0, -1.0]] and U.tolist() == [[3.0, 1.0, 2.0]] and T.tolist() == [[1.0, 1.0]]
    assert H[0, 0] == 0.0
    assert np.isclose(H[0, 1], 2.0 * s(2.0) * 1.0, rtol=1e-15)
    assert np.isclose(H[0, 2], -1.0 * s(-1.0) * 2.0, rtol=1e-15)


def test_swiglu_gradients_by_finite_differences():
    """<dH, H> is smooth in X, A, B: central differences (fp64) match the
    analytic gradients of the oracle to ~1e-7 relative."""
    rng = np.random.default_rng(14)
    M, K, I, r = 3, 64, 8, 8
    X = rng.standard_normal((M, K))
    Wg, Wu = rng.standard_normal((I, K)) * 0.1, rng.standard_normal((I, K)) * 0.1
    Ag, Au = rng.standard_normal((r, K)) * 0.1, rng.standard_normal((r, K)) * 0.1
    Bg, Bu = rng.standard_normal((I, r)) * 0.1, rng.standard_normal((I, r)) * 0.1
    dH = rng.standard_normal((M, I))
    alpha = 4.0
    g = oracle.swiglu_bwd(X, Wg, Wu, Ag, Au, Bg, Bu, dH, alpha)

    def loss(X_=X, Ag_=Ag, Bu_=Bu):
        H = oracle.swiglu_fwd(X_, Wg, Wu, Ag_, Au, Bg, Bu_, alpha)[0]
        return float(np.sum(dH * H))

    eps = 1e-5
    for (i, j) in [(0, 3), (2, 40), (1, 63)]:
        Xp, Xm = X.copy(), X.copy()
        Xp[i, j] += eps
        Xm[i, j] -= eps
        fd = (loss(X_=Xp) - loss(X_=Xm)) / (2 * eps)
        assert np.isclose(g["dX"][i, j], fd, rtol=1e-6, atol=1e-9)
    for (i, j) in [(0, 0), (5, 17)]:
        Ap, Am = Ag.copy(), Ag.copy()
        Ap[i, j] += eps
        Am[i, j] -= eps
        fd = (loss(Ag_=Ap) - loss(Ag_=Am)) / (2 * eps)
        assert np.isclose(g["dA"][0][i, j], fd, rtol=1e-6, atol=1e-9)
    for (i, j) in [(2, 1), (7, 6)]:
        Bp, Bm = Bu.copy(), Bu.copy()
        Bp[i, j] += eps
        Bm[i, j] -= eps
        fd = (loss(Bu_=Bp) - loss(Bu_=Bm)) / (2 * eps)
        assert np.isclose(g["dB"][I + i, j], fd, rtol=1e-6, atol=1e-9)
