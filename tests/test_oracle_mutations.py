"""The oracle's pins catch plausible mistakes.

Each case copies oracle.c, plants one mistake in the copy (on the CPU),
compiles it with the oracle's flags, swaps it in for the real oracle and runs
the pins of test_oracle.py: at least one must fail. The real oracle passes
all of them (test_oracle.py itself)."""
import os
import tempfile

import pytest

import oracle
import test_oracle as pins

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()

MUTANTS = {
    "nibble order swapped": ("4 * (k & 1)", "4 * (1 - (k & 1))"),
    "bias -7 instead of -8": ("& 0xF) - 8;", "& 0xF) - 7;"),
    "scale amax/8": ("amax / 7.0f", "amax / 8.0f"),
    "round half away from zero": ("rintf(r)", "roundf(r)"),
    "symmetric clamp [-7, 7]": ("if (rr < -8.0f) rr = -8.0f;", "if (rr < -7.0f) rr = -7.0f;"),
    "scale indexed by byte, not k": ("s[n * G + k / g]", "s[n * G + (k / 2) / g]"),
    "abs dropped in the bound": ("aacc += fabs(p);", "aacc += p;"),
    "subnormal exponent off by one": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "Q4_K high nibbles first": ("q[i] = r < 32 ? (byte & 0x0F) : (byte >> 4);",
                                "q[i] = r < 32 ? (byte >> 4) : (byte & 0x0F);"),
    "Q4_K top bits of mn read from byte j-4": ("*mn = (b12[j + 4] >> 4) | ((b12[j] >> 6) << 4);",
                                               "*mn = (b12[j + 4] >> 4) | ((b12[j - 4] >> 6) << 4);"),
    "Q4_K scale and minimum nibbles swapped": ("*sc = (b12[j + 4] & 0x0F) |", "*sc = (b12[j + 4] >> 4) |"),
    "Q4_K minimum added, not subtracted": ("b[i] = -(dmin * (double)mn);", "b[i] = dmin * (double)mn;"),
    "Q4_K chunks 16 bytes apart": ("qs[32 * chunk + (r % 32)]", "qs[16 * chunk + (r % 32)]"),
    "Q5_1 fifth bit of the high half from bit i-16": ("q[i] = nib | (int)(((qh >> i) & 1u) << 4);",
                                                      "q[i] = nib | (int)(((qh >> (i % 16)) & 1u) << 4);"),
    "Q5_1 offset dropped": ("b[i] = m;", "b[i] = 0.0;"),
    "block bound without the offset term": ("ar[kb * bw + i] = fabs(a[i] * (double)q[i]) + fabs(b[i]);",
                                            "ar[kb * bw + i] = fabs(a[i] * (double)q[i] + b[i]);"),
    "fp32 decode drops the offset": ("out[n * K + kb * bw + i] = p + bf;", "out[n * K + kb * bw + i] = p;"),
    "dot product skips the last k": ("for (int64_t k = 0; k < K; ++k) {\n                double p",
                                     "for (int64_t k = 0; k < K - 1; ++k) {\n                double p"),
}


def _all_pins():
    yield pins.test_half_to_double_all_bit_patterns, ()
    yield pins.test_float_to_half_matches_numpy, ()
    yield pins.test_nibble_order_golden, ()
    yield pins.test_pack_unpack_round_trip_all_bytes, ()
    for case in pins._quantize_cases():
        yield pins.test_quantize_golden, (case,)
    yield pins.test_quantize_invariants, ()
    yield pins.test_linear_golden_tiny, ()
    for args in [(1, 3, 32, 32), (2, 5, 64, 32), (3, 4, 128, 64)]:
        yield pins.test_linear_exact_rational, args
    yield pins.test_linear_zero_weights_give_zero, ()
    yield pins.test_linear_one_hot_x_reads_one_weight, ()
    for c in (-8, 5):
        yield pins.test_linear_constant_q_closed_form, (c,)
    yield pins.test_linear_unit_scales_match_numpy_matmul, ()
    yield pins.test_linear_is_linear_in_x, ()
    yield pins.test_grouped_equals_loop_of_dense_calls, ()
    for fmt in ("q4_k", "q5_1"):
        yield pins.test_blocks_golden, (fmt,)
        yield pins.test_blocks_row_bytes_closed_form, (fmt,)
    yield pins.test_blocks_decode_inverts_an_encoder, ("q4_k", 3, 512)
    yield pins.test_blocks_decode_inverts_an_encoder, ("q5_1", 4, 96)
    yield pins.test_blocks_linear_exact_rational, ("q4_k", 2, 3, 256)
    yield pins.test_blocks_linear_exact_rational, ("q5_1", 3, 2, 64)
    yield pins.test_blocks_decode_f32_is_the_rounded_exact_value, ("q4_k", 512)
    yield pins.test_blocks_decode_f32_is_the_rounded_exact_value, ("q5_1", 128)
    yield pins.test_blocks_q5_1_plain_nibbles_match_numpy_matmul, ()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    old, new = MUTANTS[name]
    assert old in SRC, f"mutation anchor not found: {old!r}"
    with tempfile.TemporaryDirectory() as d:
        so = oracle.compile_variant(SRC.replace(old, new), d)
        monkeypatch.setattr(oracle, "_lib", oracle._bind(so))
        failed = []
        for fn, args in _all_pins():
            try:
                fn(*args)
            except AssertionError:
                failed.append(fn.__name__)
        assert failed, f"no pin caught: {name}"


# ---------------------------------------------------------------- routed-MoE dispatch
# The MoE functions are numpy in oracle/__init__.py: each mutant is that module's
# source with one planted mistake, executed into a fresh namespace whose MoE
# functions replace the real ones while the MoE pins run.

PY_SRC = open(oracle.__file__).read()

PY_MUTANTS = {
    "router ties go to the higher index": (
        'ids = np.argsort(-l64, axis=1, kind="stable")[:, :top_k].astype(np.int32)',
        'ids = (E - 1 - np.argsort(-l64[:, ::-1], axis=1, kind="stable"))[:, :top_k].astype(np.int32)'),
    "router ignores renormalize": ("    if renormalize:\n        w = w / w.sum", "    if False:\n        w = w / w.sum"),
    "softmax over the selected experts only": (
        "    p /= p.sum(axis=1, keepdims=True)\n",
        "    p /= np.take_along_axis(p, ids.astype(np.int64), axis=1).sum(axis=1, keepdims=True)\n"),
    "dispatch orders by (expert, slot, token)": (
        'order = np.argsort(flat, kind="stable")',
        "order = np.lexsort((np.arange(T * k) // k, np.arange(T * k) % k, flat))"),
    "dispatch offsets shifted by one expert": ("    offsets[1:] = np.cumsum(", "    offsets[:-1] = np.cumsum("),
    "combine drops the last slot": ("    for j in range(k):\n        term", "    for j in range(k - 1):\n        term"),
    "combine reads the pair index, not its row": (
        "term = w[:, j:j + 1] * ys[row_of[:, j]]", "term = w[:, j:j + 1] * ys[np.arange(T) * k + j]"),
}

MOE_FUNCS = ("moe_route", "moe_dispatch", "moe_gather", "moe_combine", "route_tolerance", "combine_tolerance")


def _moe_pins():
    yield pins.test_moe_route_hand_worked
    yield pins.test_moe_route_brute_force
    yield pins.test_moe_route_invariants
    yield pins.test_moe_dispatch_hand_worked
    yield pins.test_moe_dispatch_brute_force
    yield pins.test_moe_combine_exact
    yield pins.test_moe_chain_equals_direct_per_token


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_moe_pins_catch_planted_mistake(name, monkeypatch):
    old, new = PY_MUTANTS[name]
    assert PY_SRC.count(old) == 1, f"mutation anchor not found once: {old!r}"
    ns = {"__name__": "oracle_mutant", "__file__": oracle.__file__}
    exec(compile(PY_SRC.replace(old, new), "oracle_mutant", "exec"), ns)
    for f in MOE_FUNCS:
        monkeypatch.setattr(oracle, f, ns[f])
    failed = []
    for fn in _moe_pins():
        try:
            fn()
        except (AssertionError, ValueError, IndexError):
            failed.append(fn.__name__)
    assert failed, f"no pin caught: {name}"


# ------------------------------------------------------------ the error bound
# tolerance() is the bound every GPU parity check applies; a mutant with a
# looser or wrong bound must fail its hand-worked pin.

TOL_LINE = "    return np.ldexp(np.abs(y_ref), -9) + 1e-4 * absdot + np.ldexp(1.0, -25)\n"
TOL_MUTANTS = {
    "relative term 2^-8": "    return np.ldexp(np.abs(y_ref), -8) + 1e-4 * absdot + np.ldexp(1.0, -25)\n",
    "absolute term 1e-3": "    return np.ldexp(np.abs(y_ref), -9) + 1e-3 * absdot + np.ldexp(1.0, -25)\n",
    "signed y_ref": "    return np.ldexp(y_ref, -9) + 1e-4 * absdot + np.ldexp(1.0, -25)\n",
    "absolute term dropped": "    return np.ldexp(np.abs(y_ref), -9) + np.ldexp(1.0, -25)\n",
    "terms multiplied": "    return np.ldexp(np.abs(y_ref), -9) * (1 + 1e-4 * absdot) + np.ldexp(1.0, -25)\n",
    "rounding term 2^-24": "    return np.ldexp(np.abs(y_ref), -9) + 1e-4 * absdot + np.ldexp(1.0, -24)\n",
    "rounding term dropped": "    return np.ldexp(np.abs(y_ref), -9) + 1e-4 * absdot\n",
}


@pytest.mark.parametrize("name", sorted(TOL_MUTANTS))
def test_tolerance_pin_catches_planted_mistake(name, monkeypatch):
    assert PY_SRC.count(TOL_LINE) == 1, "mutation anchor not found once"
    ns = {"__name__": "oracle_mutant", "__file__": oracle.__file__}
    exec(compile(PY_SRC.replace(TOL_LINE, TOL_MUTANTS[name]), "oracle_mutant", "exec"), ns)
    monkeypatch.setattr(oracle, "tolerance", ns["tolerance"])
    with pytest.raises(AssertionError):
        pins.test_tolerance_hand_worked()
