"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes one part of what the oracle computes to something independent:
the NormalFloat construction, torch's own bf16 rounding, the independently
written block packers of the input generator, closed forms, the LoRA merge
identity, finite differences and brute-force loops.
"""
import math

import numpy as np
import pytest

import oracle
import qlora_synth as syn

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------
# NF4 levels: recomputed from the NormalFloat construction
# ---------------------------------------------------------------------------
def test_nf4_levels_match_normalfloat_construction():
    from scipy.stats import norm

    p_hi = 0.5 * ((1 - 1 / (2 * 15)) + (1 - 1 / (2 * 16)))
    positives = [norm.ppf(p) for p in np.linspace(p_hi, 0.5, 9)[:8]]
    negatives = [-norm.ppf(p) for p in np.linspace(p_hi, 0.5, 8)[:7]]
    levels = sorted(positives + negatives + [0.0])
    top = max(levels)
    want = np.array([v / top for v in levels], dtype=np.float32)
    got = oracle.NF4_LEVELS
    assert got.dtype == np.float32 and got.shape == (16,)
    # exact: every fp64 level lies at least 0.02 fp32 ulp away from a
    # rounding tie, far beyond the inverse CDF's own error
    w64 = np.array([v / top for v in levels])
    frac = np.abs(w64 - want.astype(np.float64)) / np.spacing(np.abs(want))
    assert np.all(np.abs(frac - 0.5) > 0.02)
    assert np.array_equal(got, want), (got, want)
    # structure: ascending, -1 and +1 at the ends, an exact zero at code 7
    assert np.all(np.diff(got) > 0)
    assert got[0] == -1.0 and got[15] == 1.0 and got[7] == 0.0


# ---------------------------------------------------------------------------
# bf16 rounding: against torch's conversion (a library routine)
# ---------------------------------------------------------------------------
def test_bf16_round_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 0.02,
        rng.standard_normal(20000).astype(np.float32) * 300,
        # exact ties between two bf16 values, both parities
        (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40, -1e-40], dtype=np.float32),
    ]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = oracle.bf16_round_f32(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# ---------------------------------------------------------------------------
# block decode: round trips through the independent packers of qlora_synth
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("amax", [1.0, 0.0478515625, 3.5, 2.0 ** -20])
def test_nf4_every_code_round_trips(amax):
    # one row, 4 blocks; each block holds all 16 codes (four times), so the
    # block's absmax is pinned by codes 0 and 15 (levels -1 and +1)
    K = 256
    codes = np.tile(np.arange(16, dtype=np.uint8), K // 16)
    rng = np.random.default_rng(7)
    for b in range(K // 64):
        rng.shuffle(codes[b * 64:(b + 1) * 64])
    packed = ((codes[0::2] << 4) | codes[1::2]).astype(np.uint8)
    assert np.float32(amax) == oracle.bf16_round_f32(np.float32([amax]))[0]
    w = {"fmt": "nf4", "N": 1, "K": K, "data": packed,
         "absmax": np.full(K // 64, amax, dtype=np.float32)}
    dec = oracle.dequant(w)
    re = syn.pack_nf4(dec.astype(np.float32), double_quant=False)
    assert np.array_equal(re["data"], packed)
    assert np.array_equal(re["absmax"], w["absmax"])
    # closed forms: code 7 is exactly zero, codes 0 / 15 give -/+ absmax
    flat = dec.reshape(-1)
    assert np.all(flat[codes == 7] == 0.0)
    assert np.all(flat[codes == 15] == amax) and np.all(flat[codes == 0] == -amax)


def test_nf4_double_quant_decode_closed_form():
    # absmax' = f32(q) * scale2 (fp32), value = bf16(f32(level * absmax'))
    K = 64 * 512  # 512 blocks -> two groups of 256
    codes = np.full(K, 15, dtype=np.uint8)
    codes[1::2] = 7
    packed = ((codes[0::2] << 4) | codes[1::2]).astype(np.uint8)
    q = (np.arange(512) % 128).astype(np.int8)
    scale2 = np.array([0.001, 0.25], dtype=np.float32)
    w = {"fmt": "nf4", "N": 1, "K": K, "data": packed, "absmax_q": q,
         "absmax_scale": scale2, "dq_group": 256}
    dec = oracle.dequant(w).reshape(512, 64)
    for blk in (0, 1, 100, 255, 256, 300, 511):
        a = np.float32(np.float32(q[blk]) * scale2[blk // 256])
        want = float(oracle.bf16_round_f32(np.float32([a]))[0])
        assert dec[blk, 0] == want and dec[blk, 1] == 0.0


def test_nf4_double_quant_pack_decode_error_bound():
    # decoded absmax' is within half a quantisation step of the fp32 absmax
    rng = np.random.default_rng(3)
    w = rng.standard_normal((8, 64 * 64)).astype(np.float32) * 0.02
    p = syn.pack_nf4(w, double_quant=True)
    amax = np.abs(w.reshape(-1, 64)).max(axis=1)
    s = p["absmax_scale"][np.arange(amax.size) // 256]
    dq = p["absmax_q"].astype(np.float32) * s
    assert np.all(np.abs(dq - amax) <= 0.5 * s * (1 + 1e-6))
    dec = oracle.dequant(p)
    assert np.abs(dec - w).max() < 0.25 * amax.max()


@pytest.mark.parametrize("d", [2.0 ** -7, 0.75 * 2.0 ** -6, 1.25 * 2.0 ** -9, -2.0 ** -5])
def test_q4_0_every_nibble_round_trips(d):
    nb = 4
    nib = np.tile(np.arange(16, dtype=np.uint8), 2 * nb)
    rng = np.random.default_rng(11)
    for b in range(nb):
        rng.shuffle(nib[b * 32:(b + 1) * 32])
    blocks = np.empty((nb, 18), dtype=np.uint8)
    blocks[:, 0:2] = np.full(nb, d, dtype=np.float16).view(np.uint8).reshape(nb, 2)
    nb2 = nib.reshape(nb, 32)
    blocks[:, 2:] = nb2[:, :16] | (nb2[:, 16:] << 4)
    w = {"fmt": "q4_0", "N": 1, "K": 32 * nb, "data": blocks.reshape(-1)}
    dec = oracle.dequant(w).reshape(nb, 32)
    # closed form (exact here: d has at most 3 significant bits)
    assert np.array_equal(dec, (nb2.astype(np.float64) - 8) * d)
    re = syn.pack_q4_0(dec.reshape(1, -1).astype(np.float32))
    assert np.array_equal(re["data"], blocks.reshape(-1))


@pytest.mark.parametrize("d", [2.0 ** -10, 2.0 ** -5, 1.0])
def test_q8_0_every_code_round_trips(d):
    codes = np.arange(-127, 128, dtype=np.int64)          # 255 codes
    nb = 8
    q = np.zeros(nb * 32, dtype=np.int64)
    q[:codes.size] = codes
    q = q.reshape(nb, 32)
    q[:, 0] = 127  # every block holds the extreme code, pinning d
    blocks = np.empty((nb, 34), dtype=np.uint8)
    blocks[:, 0:2] = np.full(nb, d, dtype=np.float16).view(np.uint8).reshape(nb, 2)
    blocks[:, 2:] = q.astype(np.int8).view(np.uint8)
    w = {"fmt": "q8_0", "N": 1, "K": 32 * nb, "data": blocks.reshape(-1)}
    dec = oracle.dequant(w).reshape(nb, 32)
    assert np.array_equal(dec, q.astype(np.float64) * d)
    re = syn.pack_q8_0(dec.reshape(1, -1).astype(np.float32))
    assert np.array_equal(re["data"], blocks.reshape(-1))


def test_q8_0_minus_128_and_rounding_to_bf16():
    blocks = np.zeros((1, 34), dtype=np.uint8)
    d = np.float16(0.0137)
    blocks[0, 0:2] = np.array([d]).view(np.uint8)
    q = np.zeros(32, dtype=np.int8)
    q[0], q[1], q[2] = -128, 127, 0
    blocks[0, 2:] = q.view(np.uint8)
    dec = oracle.dequant({"fmt": "q8_0", "N": 1, "K": 32, "data": blocks.reshape(-1)})
    df = float(np.float32(d))
    # q*d is exact in fp32 (8 x 11 significant bits); then one rounding to bf16
    for i, qi in ((0, -128), (1, 127), (2, 0)):
        exact = qi * df
        b = float(oracle.bf16_round_f32(np.float32([exact]))[0])
        assert dec[0, i] == b
        assert abs(b - exact) <= abs(exact) * 2.0 ** -8  # half a bf16 ulp


def test_bf16_base_is_identity():
    rng = np.random.default_rng(5)
    bits = syn.normal_bf16(rng, (16, 64), 0.02)
    w = {"fmt": "bf16", "N": 16, "K": 64, "data": bits.reshape(-1)}
    assert np.array_equal(oracle.dequant(w), syn.bf16_bits_to_f32(bits).astype(np.float64).reshape(16, 64))


# ---------------------------------------------------------------------------
# the layer
# ---------------------------------------------------------------------------
def _tiny(M=5, K=12, N=7, r=3, seed=0):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((N, K)) * 0.3
    A = rng.standard_normal((r, K)) * 0.5
    B = rng.standard_normal((N, r)) * 0.5
    dY = rng.standard_normal((M, N))
    return X, W, A, B, dY


def test_forward_base_term_matches_torch_linear_when_B_is_zero():
    torch = pytest.importorskip("torch")
    X, W, A, B, dY = _tiny()
    Y, T = oracle.linear_fwd(X, W, A, np.zeros_like(B), alpha=6.0)
    ref = torch.nn.functional.linear(torch.from_numpy(X), torch.from_numpy(W)).numpy()
    assert np.array_equal(Y, ref) or np.allclose(Y, ref, rtol=1e-14, atol=1e-14)
    g = oracle.linear_bwd(X, W, A, np.zeros_like(B), dY, alpha=6.0)
    assert np.all(g["dA"] == 0.0)


def test_forward_backward_match_merged_weight():
    # LoRA merge: X W^T + s (X A^T) B^T == X (W + s B A)^T
    X, W, A, B, dY = _tiny()
    alpha = 6.0
    s = alpha / A.shape[0]
    Y, _ = oracle.linear_fwd(X, W, A, B, alpha)
    Wm = W + s * (B @ A)
    assert np.allclose(Y, X @ Wm.T, rtol=1e-12, atol=1e-12)
    g = oracle.linear_bwd(X, W, A, B, dY, alpha)
    assert np.allclose(g["dX"], dY @ Wm, rtol=1e-12, atol=1e-12)


def test_backward_matches_central_finite_differences():
    # L = <dY, Y>; L is linear in each of X, A, B separately, so the central
    # difference quotient is exact up to fp64 rounding
    X, W, A, B, dY = _tiny(M=4, K=6, N=5, r=2, seed=3)
    alpha = 5.0

    def loss(X_, A_, B_):
        Y, _ = oracle.linear_fwd(X_, W, A_, B_, alpha)
        return float(np.sum(dY * Y))

    g = oracle.linear_bwd(X, W, A, B, dY, alpha)
    h = 1e-3
    for name, arr, grad in (("X", X, g["dX"]), ("A", A, g["dA"]), ("B", B, g["dB"])):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            args_p = {"X": (p, A, B), "A": (X, p, B), "B": (X, A, p)}[name]
            args_m = {"X": (m, A, B), "A": (X, m, B), "B": (X, A, m)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.allclose(num, grad, rtol=1e-9, atol=1e-9), name


def test_against_brute_force_loops():
    X, W, A, B, dY = _tiny(M=3, K=4, N=5, r=2, seed=9)
    alpha = 3.0
    s = alpha / 2
    M, K = X.shape
    N, r = W.shape[0], 2
    Y, T = oracle.linear_fwd(X, W, A, B, alpha)
    g = oracle.linear_bwd(X, W, A, B, dY, alpha)
    for m in range(M):
        for q in range(r):
            assert math.isclose(T[m, q], sum(X[m, k] * A[q, k] for k in range(K)), rel_tol=1e-12, abs_tol=1e-12)
        for n in range(N):
            acc = sum(X[m, k] * W[n, k] for k in range(K))
            acc += s * sum(sum(X[m, k] * A[q, k] for k in range(K)) * B[n, q] for q in range(r))
            assert math.isclose(Y[m, n], acc, rel_tol=1e-12, abs_tol=1e-12)
        for k in range(K):
            acc = sum(dY[m, n] * W[n, k] for n in range(N))
            acc += s * sum(sum(dY[m, n] * B[n, q] for n in range(N)) * A[q, k] for q in range(r))
            assert math.isclose(g["dX"][m, k], acc, rel_tol=1e-12, abs_tol=1e-12)
    for q in range(r):
        for k in range(K):
            acc = s * sum(sum(dY[m, n] * B[n, q] for n in range(N)) * X[m, k] for m in range(M))
            assert math.isclose(g["dA"][q, k], acc, rel_tol=1e-12, abs_tol=1e-12)
        for n in range(N):
            acc = s * sum(dY[m, n] * sum(X[m, k] * A[q, k] for k in range(K)) for m in range(M))
            assert math.isclose(g["dB"][n, q], acc, rel_tol=1e-12, abs_tol=1e-12)


def test_hand_worked_example():
    # X = [1 2], W = [[1 0], [0 -1]], A = [[1 1]] (r = 1), B = [[2], [0.5]],
    # alpha = 2 (s = 2), dY = [1 -1]:
    #   T = 1 + 2 = 3;  Y = [1, -2] + 2*3*[2, 0.5] = [13, 1]
    #   U = 2 - 0.5 = 1.5;  dX = [1, 1] + 2*1.5*[1, 1] = [4, 4]
    #   dB = 2*[1, -1]^T*3 = [[6], [-6]];  dA = 2*1.5*[1 2] = [[3, 6]]
    X = np.array([[1.0, 2.0]])
    W = np.array([[1.0, 0.0], [0.0, -1.0]])
    A = np.array([[1.0, 1.0]])
    B = np.array([[2.0], [0.5]])
    dY = np.array([[1.0, -1.0]])
    Y, T = oracle.linear_fwd(X, W, A, B, 2.0)
    g = oracle.linear_bwd(X, W, A, B, dY, 2.0)
    assert np.array_equal(T, [[3.0]]) and np.array_equal(Y, [[13.0, 1.0]])
    assert np.array_equal(g["U"], [[1.5]]) and np.array_equal(g["dX"], [[4.0, 4.0]])
    assert np.array_equal(g["dB"], [[6.0], [-6.0]]) and np.array_equal(g["dA"], [[3.0, 6.0]])


def test_alpha_scales_lora_terms_linearly():
    X, W, A, B, dY = _tiny(seed=4)
    y0, _ = oracle.linear_fwd(X, W, A, np.zeros_like(B), 1.0)
    y1, _ = oracle.linear_fwd(X, W, A, B, 3.0)
    y2, _ = oracle.linear_fwd(X, W, A, B, 6.0)
    assert np.allclose(y2 - y0, 2 * (y1 - y0), rtol=1e-12, atol=1e-12)
    g1 = oracle.linear_bwd(X, W, A, B, dY, 3.0)
    g2 = oracle.linear_bwd(X, W, A, B, dY, 6.0)
    assert np.allclose(g2["dA"], 2 * g1["dA"]) and np.allclose(g2["dB"], 2 * g1["dB"])


def test_row_subsets_and_adapter_grads_agree_with_full():
    X, W, A, B, dY = _tiny(M=9, seed=6)
    Y, _ = oracle.linear_fwd(X, W, A, B, 4.0)
    g = oracle.linear_bwd(X, W, A, B, dY, 4.0)
    rows = [0, 4, 8]
    ys, _ = oracle.linear_fwd_rows(X[rows], W, A, B, 4.0)
    assert np.allclose(ys, Y[rows], rtol=1e-13, atol=1e-13)
    assert np.allclose(oracle.linear_bwd_rows(dY[rows], W, A, B, 4.0), g["dX"][rows], rtol=1e-13, atol=1e-13)
    ag = oracle.linear_bwd_adapter_grads(X, A, B, dY, 4.0)
    assert np.allclose(ag["dA"], g["dA"]) and np.allclose(ag["dB"], g["dB"])


def test_grouped_reduces_to_dense():
    X, W, A, B, dY = _tiny(M=10, seed=8)
    alpha = 4.0
    # one expert == the dense layer
    Y1, _ = oracle.grouped_fwd(X, [W], A[None], B[None], [0, 10], alpha)
    Yd, _ = oracle.linear_fwd(X, W, A, B, alpha)
    assert np.allclose(Y1, Yd, rtol=1e-13, atol=1e-13)
    # three experts sharing the same weights (one of them empty): the row
    # split must not matter, and the adapter grads add up over experts
    off = [0, 4, 4, 10]
    g3 = oracle.grouped_bwd(X, [W, W, W], np.stack([A] * 3), np.stack([B] * 3), dY, off, alpha)
    gd = oracle.linear_bwd(X, W, A, B, dY, alpha)
    assert np.allclose(g3["dX"], gd["dX"], rtol=1e-12, atol=1e-12)
    assert np.allclose(g3["dA"].sum(0), gd["dA"], rtol=1e-12, atol=1e-12)
    assert np.allclose(g3["dB"].sum(0), gd["dB"], rtol=1e-12, atol=1e-12)
    assert np.all(g3["dA"][1] == 0) and np.all(g3["dB"][1] == 0)


def _expert_of_row(offsets, m):
    """Expert that owns sorted row m: the e with offsets[e] <= m < offsets[e + 1]."""
    for e in range(len(offsets) - 1):
        if offsets[e] <= m < offsets[e + 1]:
            return e
    raise AssertionError(m)


def test_grouped_distinct_experts_against_row_loops():
    # every expert has its own W, A and B; expert 1 (in the middle) and the
    # last expert own no rows.  Each row is recomputed with plain loops from
    # the tensors of the expert that owns it; every expert's dA / dB is the
    # sum over exactly its own rows (zero for the empty ones).
    rng = np.random.default_rng(21)
    M, K, N, r, E = 9, 5, 4, 2, 5
    off = [0, 3, 3, 7, 9, 9]
    X = rng.standard_normal((M, K))
    dY = rng.standard_normal((M, N))
    Ws = [rng.standard_normal((N, K)) * (e + 1) for e in range(E)]
    A = rng.standard_normal((E, r, K))
    B = rng.standard_normal((E, N, r))
    alpha = 3.0
    s = alpha / r
    Y, T = oracle.grouped_fwd(X, Ws, A, B, off, alpha)
    g = oracle.grouped_bwd(X, Ws, A, B, dY, off, alpha)
    dA_ref = np.zeros((E, r, K))
    dB_ref = np.zeros((E, N, r))
    for m in range(M):
        e = _expert_of_row(off, m)
        W, Ae, Be = Ws[e], A[e], B[e]
        t = [sum(X[m, k] * Ae[q, k] for k in range(K)) for q in range(r)]
        u = [sum(dY[m, n] * Be[n, q] for n in range(N)) for q in range(r)]
        for q in range(r):
            assert math.isclose(T[m, q], t[q], rel_tol=1e-12, abs_tol=1e-12)
        for n in range(N):
            y = sum(X[m, k] * W[n, k] for k in range(K)) + s * sum(t[q] * Be[n, q] for q in range(r))
            assert math.isclose(Y[m, n], y, rel_tol=1e-12, abs_tol=1e-12), (m, n)
        for k in range(K):
            dx = sum(dY[m, n] * W[n, k] for n in range(N)) + s * sum(u[q] * Ae[q, k] for q in range(r))
            assert math.isclose(g["dX"][m, k], dx, rel_tol=1e-12, abs_tol=1e-12), (m, k)
        for q in range(r):
            for k in range(K):
                dA_ref[e, q, k] += s * u[q] * X[m, k]
            for n in range(N):
                dB_ref[e, n, q] += s * dY[m, n] * t[q]
    assert np.allclose(g["dA"], dA_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(g["dB"], dB_ref, rtol=1e-12, atol=1e-12)
    for e in (1, 4):
        assert np.all(g["dA"][e] == 0) and np.all(g["dB"][e] == 0)


def test_grouped_hand_worked_two_experts():
    # K = N = 1, r = 1, alpha = 1 (s = 1).  Expert 0: W = 2, A = 1, B = 3 owns
    # row 0 (x = 1, dy = 1); expert 1: W = -1, A = 2, B = 0.5 owns rows 1, 2
    # (x = 1, 2; dy = 2, -1).
    #   row 0: T = 1,  Y = 2 + 1*3 = 5,        U = 3,   dX = 2 + 3*1 = 5
    #   row 1: T = 2,  Y = -1 + 2*0.5 = 0,     U = 1,   dX = -2 + 1*2 = 0
    #   row 2: T = 4,  Y = -2 + 4*0.5 = 0,     U = -0.5, dX = 1 - 0.5*2 = 0
    #   dA0 = 3*1 = 3, dB0 = 1*1 = 1;  dA1 = 1*1 - 0.5*2 = 0, dB1 = 2*2 - 1*4 = 0
    X = np.array([[1.0], [1.0], [2.0]])
    dY = np.array([[1.0], [2.0], [-1.0]])
    Ws = [np.array([[2.0]]), np.array([[-1.0]])]
    A = np.array([[[1.0]], [[2.0]]])
    B = np.array([[[3.0]], [[0.5]]])
    off = [0, 1, 3]
    Y, T = oracle.grouped_fwd(X, Ws, A, B, off, 1.0)
    g = oracle.grouped_bwd(X, Ws, A, B, dY, off, 1.0)
    assert np.array_equal(T.reshape(-1), [1.0, 2.0, 4.0])
    assert np.array_equal(Y.reshape(-1), [5.0, 0.0, 0.0])
    assert np.array_equal(g["dX"].reshape(-1), [5.0, 0.0, 0.0])
    assert np.array_equal(g["dA"].reshape(-1), [3.0, 0.0])
    assert np.array_equal(g["dB"].reshape(-1), [1.0, 0.0])


def test_multi_projection_hand_worked():
    # K = 2, two projections with N = 1 each, r = 1, alpha = 1 (s = 1):
    #   X = [1 2];  p0: W = [1 1], A = [1 0], B = [2];  p1: W = [0 -1], A = [0 1], B = [-1]
    #   T = [1 | 2];  Y = [3 + 1*2 | -2 + 2*(-1)] = [5 | -4]
    #   dY = [1 | 3]:  U = [2 | -3]
    #   dX = (dY0 W0 + U0 A0) + (dY1 W1 + U1 A1) = ([1 1] + [2 0]) + ([0 -3] + [0 -3]) = [3 -5]
    #   dA0 = U0 X = [2 4], dA1 = U1 X = [-3 -6];  dB0 = dY0 T0 = 1, dB1 = dY1 T1 = 6
    X = np.array([[1.0, 2.0]])
    Ws = [np.array([[1.0, 1.0]]), np.array([[0.0, -1.0]])]
    As = [np.array([[1.0, 0.0]]), np.array([[0.0, 1.0]])]
    Bs = [np.array([[2.0]]), np.array([[-1.0]])]
    dY = np.array([[1.0, 3.0]])
    Y, T = oracle.multi_linear_fwd(X, Ws, As, Bs, 1.0)
    g = oracle.multi_linear_bwd(X, Ws, As, Bs, dY, 1.0)
    assert np.array_equal(T, [[1.0, 2.0]]) and np.array_equal(Y, [[5.0, -4.0]])
    assert np.array_equal(g["U"], [[2.0, -3.0]]) and np.array_equal(g["dX"], [[3.0, -5.0]])
    assert np.array_equal(g["dA"], [[[2.0, 4.0]], [[-3.0, -6.0]]]) and np.array_equal(g["dB"], [[1.0], [6.0]])


def test_multi_projection_is_one_linear_with_block_diagonal_adapter():
    # P projections over X equal one linear over the stacked base rows whose
    # adapter is A' = [A_0; ...; A_{P-1}] (rank P r) and the block-diagonal B'
    # (projection p's rows of B' non-zero only in block p); the summed input
    # gradient is that linear's dX, and dA_p, dB_p are the blocks of its
    # gradients.  Checked against plain matrix algebra on random tensors.
    rng = np.random.default_rng(31)
    M, K, r, Ns = 5, 7, 2, [3, 4, 2]
    X = rng.standard_normal((M, K))
    Ws = [rng.standard_normal((n, K)) for n in Ns]
    As = [rng.standard_normal((r, K)) for _ in Ns]
    Bs = [rng.standard_normal((n, r)) for n in Ns]
    dY = rng.standard_normal((M, sum(Ns)))
    alpha = 3.0
    s = alpha / r
    Y, T = oracle.multi_linear_fwd(X, Ws, As, Bs, alpha)
    g = oracle.multi_linear_bwd(X, Ws, As, Bs, dY, alpha)
    W = np.concatenate(Ws, axis=0)
    A = np.concatenate(As, axis=0)
    Bbd = np.zeros((sum(Ns), len(Ns) * r))
    o = 0
    for p, n in enumerate(Ns):
        Bbd[o:o + n, p * r:(p + 1) * r] = Bs[p]
        o += n
    assert np.allclose(T, X @ A.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(Y, X @ W.T + s * (X @ A.T) @ Bbd.T, rtol=1e-12, atol=1e-12)
    U = dY @ Bbd
    assert np.allclose(g["U"], U, rtol=1e-12, atol=1e-12)
    assert np.allclose(g["dX"], dY @ W + s * U @ A, rtol=1e-12, atol=1e-12)
    assert np.allclose(g["dA"].reshape(-1, K), s * U.T @ X, rtol=1e-12, atol=1e-12)
    dBbd = s * dY.T @ T
    o = 0
    for p, n in enumerate(Ns):
        assert np.allclose(g["dB"][o:o + n], dBbd[o:o + n, p * r:(p + 1) * r], rtol=1e-12, atol=1e-12)
        o += n


def test_stacked_adapters_match_merged_weight_and_single_adapter():
    # two adapters of different ranks and scales: the forward equals the
    # merged weight W + s0 B0 A0 + s1 B1 A1 and dX its product with dY; each
    # adapter's gradients equal those of a single-adapter layer over the
    # same base with the other adapter merged into it (the loss is linear in
    # each adapter's A and B separately given the rest)
    rng = np.random.default_rng(41)
    M, K, N = 6, 9, 5
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((N, K))
    As = [rng.standard_normal((2, K)), rng.standard_normal((3, K))]
    Bs = [rng.standard_normal((N, 2)), rng.standard_normal((N, 3))]
    alphas = [4.0, 1.5]
    dY = rng.standard_normal((M, N))
    Y, T = oracle.stacked_linear_fwd(X, W, As, Bs, alphas)
    g = oracle.stacked_linear_bwd(X, W, As, Bs, dY, alphas)
    s = [a / A.shape[0] for a, A in zip(alphas, As)]
    Wm = W + s[0] * Bs[0] @ As[0] + s[1] * Bs[1] @ As[1]
    assert np.allclose(Y, X @ Wm.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(g["dX"], dY @ Wm, rtol=1e-12, atol=1e-12)
    assert np.allclose(T, np.concatenate([X @ As[0].T, X @ As[1].T], axis=1), rtol=1e-12, atol=1e-12)
    for i in (0, 1):
        o = 1 - i
        g1 = oracle.linear_bwd(X, W + s[o] * Bs[o] @ As[o], As[i], Bs[i], dY, alphas[i])
        assert np.allclose(g["dA"][i], g1["dA"], rtol=1e-12, atol=1e-12)
        assert np.allclose(g["dB"][i], g1["dB"], rtol=1e-12, atol=1e-12)


def test_stacked_adapters_finite_differences():
    rng = np.random.default_rng(43)
    M, K, N = 3, 4, 3
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((N, K))
    As = [rng.standard_normal((1, K)), rng.standard_normal((2, K))]
    Bs = [rng.standard_normal((N, 1)), rng.standard_normal((N, 2))]
    alphas = [2.0, 3.0]
    dY = rng.standard_normal((M, N))
    g = oracle.stacked_linear_bwd(X, W, As, Bs, dY, alphas)

    def loss(As_, Bs_):
        Y, _ = oracle.stacked_linear_fwd(X, W, As_, Bs_, alphas)
        return float(np.sum(dY * Y))

    h = 1e-3
    for i in (0, 1):
        for which, grads in (("A", g["dA"][i]), ("B", g["dB"][i])):
            base = As[i] if which == "A" else Bs[i]
            num = np.zeros_like(base)
            for idx in np.ndindex(base.shape):
                vals = []
                for sgn in (1, -1):
                    pert = base.copy()
                    pert[idx] += sgn * h
                    A2 = [pert if (which == "A" and j == i) else As[j] for j in range(2)]
                    B2 = [pert if (which == "B" and j == i) else Bs[j] for j in range(2)]
                    vals.append(loss(A2, B2))
                num[idx] = (vals[0] - vals[1]) / (2 * h)
            assert np.allclose(num, grads, rtol=1e-9, atol=1e-9), (i, which)
