"""Planted mistakes: the pins of the oracle must catch them.

Each case edits one expression of the oracle's source (a dropped term, a
flipped sign, a wrong operand, index, offset, bias, nibble or byte order),
executes the edited source as a throw-away module, points the pin modules at
it and runs the pins named for that mistake: every one of them must fail.  A
control case runs the same harness on the unedited source, where every pin
must pass, so a failure below is the planted mistake's and not the harness's.
The oracle on disk is never modified.
"""
import types

import pytest

import oracle
import oracle.qlora_oracle as oracle_src
import test_oracle_pins as pins
import test_oracle_pins_formats as pins_f

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

SOURCE = open(oracle_src.__file__, encoding="utf-8").read()

# pin name -> (module, function, arguments)
PINS = {
    "bf16_vs_torch": (pins, "test_bf16_round_matches_torch", ()),
    "nf4_levels": (pins, "test_nf4_levels_match_normalfloat_construction", ()),
    "nf4_round_trip_1": (pins, "test_nf4_every_code_round_trips", (1.0,)),
    "nf4_round_trip_3.5": (pins, "test_nf4_every_code_round_trips", (3.5,)),
    "nf4_dq_closed_form": (pins, "test_nf4_double_quant_decode_closed_form", ()),
    "nf4_dq_error_bound": (pins, "test_nf4_double_quant_pack_decode_error_bound", ()),
    "q4_0_round_trip": (pins, "test_q4_0_every_nibble_round_trips", (2.0 ** -7,)),
    "q8_0_round_trip": (pins, "test_q8_0_every_code_round_trips", (1.0,)),
    "q8_0_minus_128": (pins, "test_q8_0_minus_128_and_rounding_to_bf16", ()),
    "merged_weight": (pins, "test_forward_backward_match_merged_weight", ()),
    "finite_differences": (pins, "test_backward_matches_central_finite_differences", ()),
    "brute_force": (pins, "test_against_brute_force_loops", ()),
    "hand_worked": (pins, "test_hand_worked_example", ()),
    "row_subsets": (pins, "test_row_subsets_and_adapter_grads_agree_with_full", ()),
    "grouped_distinct": (pins, "test_grouped_distinct_experts_against_row_loops", ()),
    "grouped_hand_worked": (pins, "test_grouped_hand_worked_two_experts", ()),
    "multi_hand_worked": (pins, "test_multi_projection_hand_worked", ()),
    "multi_block_diagonal": (pins, "test_multi_projection_is_one_linear_with_block_diagonal_adapter", ()),
    "stacked_merged": (pins, "test_stacked_adapters_match_merged_weight_and_single_adapter", ()),
    "stacked_fd": (pins, "test_stacked_adapters_finite_differences", ()),
    "e4m3_vs_torch": (pins_f, "test_e4m3_matches_torch_for_every_code", ()),
    "e2m1_in_e4m3": (pins_f, "test_e2m1_embeds_in_e4m3", ()),
    "fp8_hand_worked": (pins_f, "test_fp8_hand_worked", ()),
    "fp8_round_trip": (pins_f, "test_fp8_round_trips_through_packer", ()),
    "nvfp4_hand_worked": (pins_f, "test_nvfp4_hand_worked", ()),
    "nvfp4_round_trip": (pins_f, "test_nvfp4_round_trips_through_packer", ()),
    "q4_k_scale_unpack": (pins_f, "test_q4_k_scale_unpack_hand_worked", ()),
    "q4_k_hand_worked": (pins_f, "test_q4_k_hand_worked", ()),
    "q4_k_is_q4_0": (pins_f, "test_q4_k_reduces_to_q4_0", ()),
    "q4_k_parts": (pins_f, "test_q4_k_decodes_parts_packed_independently", ()),
    "dq_map_hand_worked": (pins_f, "test_dq_map_hand_worked", ()),
    "swiglu_hand_worked": (pins_f, "test_swiglu_hand_worked", ()),
    "swiglu_fwd_hand_worked": (pins_f, "test_swiglu_forward_hand_worked", ()),
    "swiglu_fd": (pins_f, "test_swiglu_gradients_by_finite_differences", ()),
}

# (mistake, source text, planted text, pins that must fail)
MISTAKES = [
    ("forward adapter term dropped",
     "    Y = X @ Wd.T + s * (T @ B.T)\n    return Y, T\n", "    Y = X @ Wd.T\n    return Y, T\n",
     ["merged_weight", "finite_differences", "brute_force", "hand_worked"]),
    ("forward adapter sign flipped",
     "    Y = X @ Wd.T + s * (T @ B.T)\n    return Y, T\n", "    Y = X @ Wd.T - s * (T @ B.T)\n    return Y, T\n",
     ["merged_weight", "finite_differences", "brute_force", "hand_worked"]),
    ("forward scale alpha instead of alpha / r",
     "    s = float(alpha) / r\n    T = X @ A.T\n    Y =", "    s = float(alpha)\n    T = X @ A.T\n    Y =",
     ["merged_weight", "finite_differences", "brute_force"]),
    ("dX adapter term dropped",
     "    dX = dY @ Wd + s * (U @ A)\n    dB =", "    dX = dY @ Wd\n    dB =",
     ["merged_weight", "finite_differences", "brute_force", "hand_worked"]),
    ("dB from U instead of T",
     "    dB = s * (dY.T @ T)\n    dA = s * (U.T @ X)\n", "    dB = s * (dY.T @ U)\n    dA = s * (U.T @ X)\n",
     ["finite_differences", "brute_force", "hand_worked"]),
    ("dA from T instead of U",
     "    dB = s * (dY.T @ T)\n    dA = s * (U.T @ X)\n", "    dB = s * (dY.T @ T)\n    dA = s * (T.T @ X)\n",
     ["finite_differences", "brute_force", "hand_worked"]),
    ("sampled-row dX without its adapter term",
     "    return dY @ Wd + s * ((dY @ B) @ A)\n", "    return dY @ Wd\n",
     ["row_subsets"]),
    ("all-row adapter gradients: dB from U",
     '    return {"T": T, "U": U, "dA": s * (U.T @ X), "dB": s * (dY.T @ T)}',
     '    return {"T": T, "U": U, "dA": s * (U.T @ X), "dB": s * (dY.T @ U)}',
     ["row_subsets"]),
    ("bf16 rounding truncates",
     "    u = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)\n",
     "    u = (u >> np.uint64(16)) << np.uint64(16)\n",
     ["bf16_vs_torch"]),
    ("bf16 ties rounded away from zero",
     "    u = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)\n",
     "    u = ((u + np.uint64(0x8000)) >> np.uint64(16)) << np.uint64(16)\n",
     ["bf16_vs_torch"]),
    ("NF4 nibble order swapped",
     "    codes[0::2] = packed >> 4\n    codes[1::2] = packed & 0x0F\n    codes = codes.reshape(-1, 64)\n",
     "    codes[0::2] = packed & 0x0F\n    codes[1::2] = packed >> 4\n    codes = codes.reshape(-1, 64)\n",
     ["nf4_round_trip_1", "nf4_dq_closed_form"]),
    ("NF4 absmax not applied",
     "    prod = (NF4_LEVELS[codes] * amax[:, None]).astype(np.float32)",
     "    prod = (NF4_LEVELS[codes] + 0 * amax[:, None]).astype(np.float32)",
     ["nf4_round_trip_3.5", "nf4_dq_closed_form", "nf4_dq_error_bound"]),
    ("NF4 double-quantisation group index wrong",
     "        g = np.arange(nblk) // group\n", "        g = np.arange(nblk) % scale2.size\n",
     ["nf4_dq_closed_form"]),
    ("NF4 8-bit map offset dropped",
     '            amax = (amax + np.float32(w["absmax_offset"])).astype(np.float32)\n',
     "            amax = amax.astype(np.float32)\n",
     ["dq_map_hand_worked"]),
    ("Q4_0 offset 7 instead of 8",
     "    prod = ((nib - 8).astype(np.float32)", "    prod = ((nib - 7).astype(np.float32)",
     ["q4_0_round_trip", "q4_k_is_q4_0"]),
    ("Q4_0 nibble halves swapped",
     "    nib = np.concatenate([qs & 0x0F, qs >> 4], axis=1)", "    nib = np.concatenate([qs >> 4, qs & 0x0F], axis=1)",
     ["q4_0_round_trip"]),
    ("Q8_0 codes read unsigned",
     "    q = blk[:, 2:34].copy().view(np.int8).astype(np.float32)",
     "    q = blk[:, 2:34].copy().view(np.uint8).astype(np.float32)",
     ["q8_0_round_trip", "q8_0_minus_128"]),
    ("Q4_K min added instead of subtracted",
     "    val = (prod - mmn[:, :, None]).astype(np.float32)", "    val = (prod + mmn[:, :, None]).astype(np.float32)",
     ["q4_k_hand_worked", "q4_k_is_q4_0", "q4_k_parts"]),
    ("Q4_K sub-block order swapped",
     "    q = np.stack([qs & 0x0F, qs >> 4], axis=2)", "    q = np.stack([qs >> 4, qs & 0x0F], axis=2)",
     ["q4_k_parts"]),
    ("Q4_K upper scale bits from the wrong byte",
     "        sc[:, j] = (b[:, j + 4] & 0x0F) | ((b[:, j - 4] >> 6) << 4)\n",
     "        sc[:, j] = (b[:, j + 4] & 0x0F) | ((b[:, j] >> 6) << 4)\n",
     ["q4_k_scale_unpack"]),
    ("E4M3 exponent bias 8",
     "np.exp2((e - 7).astype(np.float64))", "np.exp2((e - 8).astype(np.float64))",
     ["e4m3_vs_torch", "fp8_hand_worked"]),
    ("E4M3 subnormal scale 2^-7",
     "(m / 8.0) * 2.0 ** -6", "(m / 8.0) * 2.0 ** -7",
     ["e4m3_vs_torch"]),
    ("E2M1 subnormal 1.0 instead of 0.5",
     "mag = np.where(e == 0, m * 0.5,", "mag = np.where(e == 0, m * 1.0,",
     ["e2m1_in_e4m3", "nvfp4_hand_worked"]),
    ("FP8 tensor scale not applied",
     "    prod = (e4m3_value(c).astype(np.float32) * scale).astype(np.float32)",
     "    prod = (e4m3_value(c).astype(np.float32) * np.float32(1.0)).astype(np.float32)",
     ["fp8_hand_worked"]),
    ("NVFP4 nibble order swapped",
     "    codes[0::2] = packed & 0x0F\n    codes[1::2] = packed >> 4\n    sblk",
     "    codes[0::2] = packed >> 4\n    codes[1::2] = packed & 0x0F\n    sblk",
     ["nvfp4_hand_worked", "nvfp4_round_trip"]),
    ("grouped forward uses expert 0's tensors",
     "linear_fwd(X[lo:hi], Wds[e], A[e], B[e], alpha)", "linear_fwd(X[lo:hi], Wds[0], A[0], B[0], alpha)",
     ["grouped_distinct", "grouped_hand_worked"]),
    ("grouped backward writes dA / dB to the wrong expert",
     '            dX[lo:hi], dA[e], dB[e] = g["dX"], g["dA"], g["dB"]\n',
     '            dX[lo:hi], dA[E - 1 - e], dB[E - 1 - e] = g["dX"], g["dA"], g["dB"]\n',
     ["grouped_distinct", "grouped_hand_worked"]),
    ("fused projections' dX not summed",
     '    return {"dX": sum(g["dX"] for g in gs),', '    return {"dX": gs[0]["dX"],',
     ["multi_hand_worked", "multi_block_diagonal"]),
    ("stacked adapters all scaled by the first alpha",
     "        s = float(alpha) / A.shape[0]\n        T = X @ A.T\n        Y = Y + s",
     "        s = float(alphas[0]) / A.shape[0]\n        T = X @ A.T\n        Y = Y + s",
     ["stacked_merged", "stacked_fd"]),
    ("SwiGLU derivative factor dropped",
     "    return dH * U * sg * (1.0 + G * (1.0 - sg)), dH * G * sg",
     "    return dH * U * sg, dH * G * sg",
     ["swiglu_hand_worked", "swiglu_fd"]),
    ("one NF4 level off in its last digit",
     "    0.44070974, 0.5626169, 0.72295666, 1.0,\n", "    0.44070974, 0.5626168, 0.72295666, 1.0,\n",
     ["nf4_levels"]),
    ("Q8_0 block scale not applied",
     "    prod = (q * d[:, None]).astype(np.float32)", "    prod = (q * np.float32(1.0)).astype(np.float32)",
     ["q8_0_minus_128"]),
    ("E4M3 NaN code read as a number",
     "    return np.where((e == 15) & (m == 7), np.nan, v)", "    return v",
     ["e4m3_vs_torch"]),
    ("grouped forward drops each expert's last row",
     "        lo, hi = int(offsets[e]), int(offsets[e + 1])\n        if hi > lo:\n            Y[lo:hi]",
     "        lo, hi = int(offsets[e]), int(offsets[e + 1]) - 1\n        if hi > lo:\n            Y[lo:hi]",
     ["grouped_distinct", "grouped_hand_worked"]),
    ("fused projections' T blocks in reverse order",
     "np.concatenate([t for _, t in outs], axis=1)", "np.concatenate([t for _, t in outs[::-1]], axis=1)",
     ["multi_hand_worked", "multi_block_diagonal"]),
    ("fused projections' dB blocks in reverse order",
     'np.concatenate([g["dB"] for g in gs], axis=0)', 'np.concatenate([g["dB"] for g in gs[::-1]], axis=0)',
     ["multi_hand_worked", "multi_block_diagonal"]),
    ("stacked adapters' dB from U instead of T",
     "        dB.append(s * (dY.T @ T))\n", "        dB.append(s * (dY.T @ U))\n",
     ["stacked_fd"]),
    ("SwiGLU dU from U instead of G",
     "    return dH * U * sg * (1.0 + G * (1.0 - sg)), dH * G * sg",
     "    return dH * U * sg * (1.0 + G * (1.0 - sg)), dH * U * sg",
     ["swiglu_hand_worked", "swiglu_fd"]),
    ("SwiGLU gate and up swapped",
     "    H = G * _sigmoid(G) * U\n", "    H = U * _sigmoid(U) * G\n",
     ["swiglu_fwd_hand_worked", "swiglu_fd"]),
]


def _module_from(text: str) -> types.ModuleType:
    mod = types.ModuleType("oracle_planted")
    mod.__file__ = oracle_src.__file__
    exec(compile(text, "oracle_planted", "exec"), mod.__dict__)
    return mod


def _run_pins(monkeypatch, mod, names):
    """Names of the pins that fail with `mod` as the oracle."""
    monkeypatch.setattr(pins, "oracle", mod)
    monkeypatch.setattr(pins_f, "oracle", mod)
    failed = []
    for name in names:
        module, fn, args = PINS[name]
        try:
            getattr(module, fn)(*args)
        except Exception:  # an assertion, or an exception the mistake caused
            failed.append(name)
    return failed


def test_harness_passes_every_pin_on_the_unedited_source(monkeypatch):
    assert _run_pins(monkeypatch, _module_from(SOURCE), list(PINS)) == []


@pytest.mark.parametrize("mistake,old,new,must_fail", MISTAKES, ids=[m[0] for m in MISTAKES])
def test_pins_catch_planted_mistake(monkeypatch, mistake, old, new, must_fail):
    assert SOURCE.count(old) == 1, f"source text for '{mistake}' not found exactly once"
    mod = _module_from(SOURCE.replace(old, new))
    failed = _run_pins(monkeypatch, mod, must_fail)
    assert failed == must_fail, f"{mistake}: pins that did not catch it: {sorted(set(must_fail) - set(failed))}"
    # the edit did not reach the oracle the other tests use
    assert oracle.linear_fwd is not mod.linear_fwd
