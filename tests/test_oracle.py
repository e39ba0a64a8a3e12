"""Pins for the CPU oracle (no GPU needed).

Each test checks the oracle against something other than itself: numpy's own
binary16 conversion, hand-worked fixtures (tests/golden/), exact rational
arithmetic, closed forms and invariants of y = x W^T with W^ = s * q.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from conftest import GOLDEN


# ------------------------------------------------------------------ fixtures

def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def _quantize_cases():
    cases, cur = [], None
    for line in _golden_lines("quantize_groups.txt"):
        key, _, rest = line.partition(" ")
        if key == "case":
            name, g = rest.split()
            cur = dict(name=name, g=int(g))
            cases.append(cur)
        elif key == "w":
            cur["w"] = [np.float32(v) for v in rest.split()]
        elif key == "s":
            cur["s"] = [int(v, 16) for v in rest.split()]
        elif key == "q":
            cur["q"] = {int(a): int(b) for a, b in (t.split(":") for t in rest.split())}
        elif key == "bytes":
            cur["bytes"] = [int(v, 16) for v in rest.split()]
    return cases


# -------------------------------------------------------------- fp16 pins

def test_half_to_double_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0])


def test_float_to_half_matches_numpy():
    g = np.random.default_rng(1)
    parts = [
        g.normal(0, 1, 200_000),
        g.normal(0, 1e-5, 50_000),                       # subnormal fp16 range
        g.normal(0, 3e4, 50_000),                        # near overflow
        np.ldexp(g.uniform(1, 2, 50_000), g.integers(-30, 18, 50_000)),
    ]
    f = np.concatenate(parts).astype(np.float32)
    # exact ties between two fp16 neighbours, normal and subnormal
    h = g.integers(0, 0x7BFF, 20_000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    ties = ((lo + hi) / 2).astype(np.float32)
    f = np.concatenate([f, ties, -ties, np.float32([65504, 65519.99, 65520, 1e9, -1e9, 0.0, -0.0,
                                                     np.inf, -np.inf])])
    ours = oracle.float_to_half_bits(f)
    ref = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.isnan(oracle.half_to_double(oracle.float_to_half_bits(np.float32([np.nan])))[0])


# ---------------------------------------------------------- format pins

def test_nibble_order_golden():
    rows = [line.split() for line in _golden_lines("nibble_order.txt")]
    b = np.array([[int(r[0], 16) for r in rows]], np.uint8)
    q = oracle.unpack(b, 2 * b.shape[1])
    assert q[0, 0::2].tolist() == [int(r[1]) for r in rows]
    assert q[0, 1::2].tolist() == [int(r[2]) for r in rows]


def test_pack_unpack_round_trip_all_bytes():
    b = np.arange(256, dtype=np.uint8).reshape(4, 64)
    q = oracle.unpack(b, 128)
    assert q.min() == -8 and q.max() == 7
    assert np.array_equal(oracle.pack_q(q), b)
    # every (even, odd) pair of q values appears exactly once
    pairs = set(zip(q[:, 0::2].ravel().tolist(), q[:, 1::2].ravel().tolist()))
    assert len(pairs) == 256


@pytest.mark.parametrize("case", _quantize_cases(), ids=lambda c: c["name"])
def test_quantize_golden(case):
    g = case["g"]
    K = g * len(case["s"])
    w = np.zeros((1, K), np.float32)
    w[0, :len(case["w"])] = case["w"]
    qw, s = oracle.quantize(w, g)
    assert s[0].tolist() == case["s"]
    q = oracle.unpack(qw, K)[0]
    want = np.zeros(K, np.int64)
    for k, v in case["q"].items():
        want[k] = v
    assert q.tolist() == want.tolist()
    bytes_want = [0x88] * (K // 2)
    bytes_want[:len(case["bytes"])] = case["bytes"]
    assert qw[0].tolist() == bytes_want


def test_quantize_invariants():
    g = workloads.rng(3)
    for group in (32, 64, 128):
        W = workloads.weights(g, 48, 512)
        qw, s = oracle.quantize(W, group)
        q = oracle.unpack(qw, 512).astype(np.float64)
        sd = oracle.half_to_double(s)
        sk = np.repeat(sd, group, axis=1)
        Wg = W.astype(np.float64).reshape(48, -1, group)
        amax = np.abs(Wg).max(axis=2)
        # the scale is amax/7 to within fp16 rounding (relative 2^-11)
        assert np.all(np.abs(sd * 7 - amax) <= amax * 2.0 ** -11 * 7 / 6.9)
        # the element of largest magnitude lands on +-7
        arg = np.abs(Wg).argmax(axis=2)
        qg = q.reshape(48, -1, group)
        assert np.all(np.abs(np.take_along_axis(qg, arg[..., None], 2)) == 7)
        # round to nearest: |w - s q| <= s/2 (plus fp32 quotient rounding)
        err = np.abs(W - sk * q)
        assert np.all(err <= sk * (0.5 + 2.0 ** -20))
        assert q.min() >= -8 and q.max() <= 7
        # odd symmetry and power-of-two scale invariance
        qw_n, s_n = oracle.quantize(-W, group)
        assert np.array_equal(s_n, s)
        assert np.array_equal(oracle.unpack(qw_n, 512), -oracle.unpack(qw, 512))
        qw_2, s_2 = oracle.quantize(W * np.float32(4), group)
        assert np.array_equal(qw_2, qw)
        assert np.array_equal(oracle.half_to_double(s_2), 4 * sd)


# ---------------------------------------------------------- linear pins

def _raw(seed, M, N, K, g):
    r = workloads.rng(seed)
    qw, s = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    return x, qw, s


def test_linear_golden_tiny():
    cases = {c["name"]: c for c in _quantize_cases()}
    rows = []
    for name in ("A", "B"):
        w = np.zeros((1, 32), np.float32)
        w[0, :len(cases[name]["w"])] = cases[name]["w"]
        rows.append(oracle.quantize(w, 32))
    qw = np.concatenate([r[0] for r in rows])
    s = np.concatenate([r[1] for r in rows])
    x = np.zeros((2, 32), np.float16)
    x[0, :] = 1
    x[1, 0], x[1, 1] = 1, 2
    y, _ = oracle.linear(x, qw, s, 32)
    for line in _golden_lines("linear_tiny.txt"):
        _, m, n, v = line.split()
        assert y[int(m), int(n)] == float(v)


@pytest.mark.parametrize("M,N,K,g", [(1, 3, 32, 32), (2, 5, 64, 32), (3, 4, 128, 64),
                                     (2, 3, 256, 128), (1, 2, 384, 128)])
def test_linear_exact_rational(M, N, K, g):
    """fp64 oracle vs the exact sum (fp16 values are dyadic rationals)."""
    x, qw, s = _raw(7 + K, M, N, K, g)
    y, absdot = oracle.linear(x, qw, s, g)
    xb = x.view(np.uint16)
    sb = s.view(np.uint16)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            for j in range(K // g):
                sc = Fraction(float(np.uint16(sb[n, j]).view(np.float16)))
                for k in range(j * g, (j + 1) * g):
                    byte = int(qw[n, k // 2])
                    nib = (byte >> 4) if (k % 2) else (byte & 15)
                    xv = Fraction(float(np.uint16(xb[m, k]).view(np.float16)))
                    exact += xv * sc * (nib - 8)
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(K * 2.0 ** -52) * Fraction(absdot[m, n])


def test_linear_zero_weights_give_zero():
    x, _, s = _raw(11, 3, 7, 256, 64)
    qw = np.full((7, 128), 0x88, np.uint8)      # every q = 0
    y, a = oracle.linear(x, qw, s, 64)
    assert np.all(y == 0) and np.all(a == 0)


def test_linear_one_hot_x_reads_one_weight():
    K, N, g = 256, 6, 32
    _, qw, s = _raw(12, 1, N, K, g)
    q = oracle.unpack(qw, K)
    sd = oracle.half_to_double(s)
    for k in (0, 1, 31, 32, 77, 255):
        x = np.zeros((1, K), np.float16)
        x[0, k] = 1
        y, _ = oracle.linear(x, qw, s, g)
        assert np.array_equal(y[0], sd[:, k // g] * q[:, k])


@pytest.mark.parametrize("c", [-8, -3, 0, 5, 7])
def test_linear_constant_q_closed_form(c):
    K, N, g = 512, 5, 128
    _, _, s = _raw(13, 1, N, K, g)
    qw = np.full((N, K // 2), ((c + 8) | ((c + 8) << 4)), np.uint8)
    x = np.ones((1, K), np.float16)
    y, _ = oracle.linear(x, qw, s, g)
    sd = oracle.half_to_double(s)
    assert np.array_equal(y[0], c * g * sd.sum(axis=1))


def test_linear_unit_scales_match_numpy_matmul():
    M, N, K, g = 4, 33, 640, 64
    x, qw, _ = _raw(14, M, N, K, g)
    s = np.ones((N, K // g), np.float16)
    q = oracle.unpack(qw, K).astype(np.float64)
    y, a = oracle.linear(x, qw, s, g)
    ref = x.astype(np.float64) @ q.T
    assert np.all(np.abs(y - ref) <= K * 2.0 ** -52 * a)


def test_linear_is_linear_in_x():
    M, N, K, g = 2, 9, 512, 128
    _, qw, s = _raw(15, 1, N, K, g)
    r = workloads.rng(16)
    x1 = r.integers(-32, 33, (M, K)).astype(np.float16)   # small integers: sums exact
    x2 = r.integers(-32, 33, (M, K)).astype(np.float16)
    x3 = (3 * x1.astype(np.float64) - 2 * x2.astype(np.float64)).astype(np.float16)
    y1, a1 = oracle.linear(x1, qw, s, g)
    y2, a2 = oracle.linear(x2, qw, s, g)
    y3, a3 = oracle.linear(x3, qw, s, g)
    assert np.all(np.abs(y3 - (3 * y1 - 2 * y2)) <= K * 2.0 ** -50 * (a3 + 3 * a1 + 2 * a2))


def test_linear_group_permutation_invariance():
    M, N, K, g = 3, 8, 512, 64
    x, qw, s = _raw(17, M, N, K, g)
    perm = workloads.rng(18).permutation(K // g)
    kidx = np.concatenate([np.arange(p * g, (p + 1) * g) for p in perm])
    bidx = np.concatenate([np.arange(p * g // 2, (p + 1) * g // 2) for p in perm])
    y, a = oracle.linear(x, qw, s, g)
    yp, _ = oracle.linear(np.ascontiguousarray(x[:, kidx]), np.ascontiguousarray(qw[:, bidx]),
                          np.ascontiguousarray(s[:, perm]), g)
    assert np.all(np.abs(yp - y) <= K * 2.0 ** -51 * a)


def test_grouped_equals_loop_of_dense_calls():
    E, N, K, g = 6, 10, 256, 32
    r = workloads.rng(19)
    qw = r.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    s = (np.abs(r.normal(0, 0.02, (E, N, K // g))) / 7).astype(np.float16)
    counts = np.array([3, 0, 5, 1, 0, 7])                 # empty experts included
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = workloads.activations(r, int(off[-1]), K)
    y, a = oracle.grouped_linear(x, qw, s, off, g)
    for e in range(E):
        if counts[e]:
            ye, ae = oracle.linear(x[off[e]:off[e + 1]], qw[e], s[e], g)
            assert np.array_equal(y[off[e]:off[e + 1]], ye)
            assert np.array_equal(a[off[e]:off[e + 1]], ae)
    y1, _ = oracle.grouped_linear(x, qw[:1], s[:1], np.int32([0, off[-1]]), g)
    assert np.array_equal(y1, oracle.linear(x, qw[0], s[0], g)[0])


def test_tolerance_hand_worked():
    """The per-element bound of the workload specification,
    |y - y_ref| <= 2^-9 |y_ref| + 1e-4 sum_k |x_k W^_nk|, on values worked out
    by hand: each term alone, a negative y_ref (its magnitude counts), and the
    two terms together. Every GPU parity check compares against this bound."""
    h = 2.0 ** -25                          # half the binary16 subnormal spacing, in every case
    cases = [
        # y_ref, sum_k |x W^|, bound
        (1.0, 0.0, 0.001953125 + h),            # 2^-9 alone
        (0.0, 1.0, 0.0001 + h),                 # 1e-4 alone
        (-3.0, 2.0, 0.005859375 + 0.0002 + h),  # 3 * 2^-9 + 2 * 1e-4: |y_ref|, not y_ref
        (512.0, 0.0, 1.0 + h),                  # 512 * 2^-9
        (-0.25, 10000.0, 1.00048828125 + h),    # 2^-11 + 1
        (0.0, 0.0, h),
    ]
    y = np.array([c[0] for c in cases])
    a = np.array([c[1] for c in cases])
    want = np.array([c[2] for c in cases])
    got = oracle.tolerance(y, a)
    assert got.shape == want.shape
    assert np.allclose(got, want, rtol=1e-14, atol=0.0), (got, want)
    # the bound grows with both arguments, and only with |y_ref|
    assert np.array_equal(oracle.tolerance(-y, a), got)


def test_tolerance_admits_the_correctly_rounded_result():
    """Whatever the size of y, its exact value rounded to fp16 (what a perfect
    kernel returns) lies within the bound, also in the subnormal range where
    2^-9 |y| alone is far too small; and the absolute term is no larger than
    that rounding needs."""
    r = np.random.default_rng(8)
    y = np.concatenate([np.ldexp(1.0, np.arange(-34, 15)), np.exp(r.uniform(np.log(1e-10), np.log(6e4), 20000))])
    y *= r.choice([-1.0, 1.0], y.size)
    zero = np.zeros_like(y)
    err = np.abs(y.astype(np.float16).astype(np.float64) - y)
    assert np.all(err <= oracle.tolerance(y, zero))
    sub = np.abs(y) < np.ldexp(1.0, -14)
    assert np.any(err[sub] > np.ldexp(np.abs(y[sub]), -9))       # the relative term alone fails there
    assert np.max(err) <= np.ldexp(1.0, -25) + np.max(np.ldexp(np.abs(y), -11))


def test_threaded_linear_equals_single_thread():
    x, qw, s = _raw(20, 3, 101, 256, 128)
    y1, a1 = oracle.linear(x, qw, s, 128)
    y4, a4 = oracle.linear(x, qw, s, 128, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(a1, a4)


# ------------------------------------------------------------ workloads

def test_workloads_are_seeded_and_shaped():
    W, x, g = workloads.config0()
    W2, x2, _ = workloads.config0()
    assert W.shape == (256, 1024) and x.shape == (1, 1024) and g == 128
    assert np.array_equal(W, W2) and np.array_equal(x, x2)
    assert abs(W.std() - 0.02) < 0.001
    _, xp, _ = workloads.prefill(8, K=1000, N=4)
    big = np.abs(xp.astype(np.float32)).max(axis=0) > 0
    assert xp.dtype == np.float16 and big.all()
    r = workloads.routing(workloads.rng(0), 64, 16, 4)
    assert r.offsets[0] == 0 and r.offsets[-1] == 256
    assert np.all(np.diff(r.offsets) >= 0)
    assert np.all(np.diff(r.expert_of_row) >= 0)
    pairs = set(zip(r.token_of_row.tolist(), r.expert_of_row.tolist()))
    assert len(pairs) == 256                               # distinct experts per token


# ------------------------------------------------------------ gated MLP pins

def test_silu_closed_forms():
    # sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4, so silu(+-ln 3) = +-ln 3 * (3/4 | 1/4)
    l3 = np.log(3.0)
    assert oracle.silu(l3) == pytest.approx(0.75 * l3, rel=1e-15)
    assert oracle.silu(-l3) == pytest.approx(-0.25 * l3, rel=1e-15)
    assert oracle.silu(0.0) == 0.0
    # silu(v) - silu(-v) = v (sigmoid(v) + sigmoid(-v) = 1), across magnitudes
    v = np.concatenate([np.linspace(-30, 30, 601), [1e-8, -1e-8, 700.0, -700.0]])
    assert np.allclose(oracle.silu(v) - oracle.silu(-v), v, rtol=1e-14, atol=1e-300)
    # far tails: silu(v) -> v for large v, -> -0 for very negative v, never NaN
    assert oracle.silu(60.0) == pytest.approx(60.0, rel=1e-15)
    assert oracle.silu(-1000.0) == 0.0 and not np.isnan(oracle.silu(-1000.0))


def test_gated_zero_up_or_gate_gives_zero():
    x, qw, s = _raw(31, 3, 9, 256, 64)
    zero = np.full_like(qw, 0x88)                # every q = 0
    y, g, u, _, _ = oracle.gated_linear(x, qw, s, zero, s, 64)
    assert np.all(u == 0) and np.all(y == 0)
    y, g, u, _, _ = oracle.gated_linear(x, zero, s, qw, s, 64)
    assert np.all(g == 0) and np.all(y == 0)     # silu(0) = 0


def test_gated_one_hot_closed_form():
    """One-hot x picks one weight of each matrix: y = silu(sg qg) * (su qu),
    with silu evaluated independently through math.exp; swapping gate and up
    (a plausible slip) changes every value checked here."""
    import math

    K, N, g = 128, 5, 32
    _, qg, sg = _raw(32, 1, N, K, g)
    _, qu, su = _raw(33, 1, N, K, g)
    # scales of order 1 put g and u where silu is far from linear
    sg = oracle.float_to_half_bits(np.float32(16.0) * oracle.half_to_double(sg).astype(np.float32))
    su = oracle.float_to_half_bits(np.float32(16.0) * oracle.half_to_double(su).astype(np.float32))
    Wg = oracle.half_to_double(sg)[:, :, None] * oracle.unpack(qg, K).reshape(N, K // g, g)
    Wu = oracle.half_to_double(su)[:, :, None] * oracle.unpack(qu, K).reshape(N, K // g, g)
    Wg, Wu = Wg.reshape(N, K), Wu.reshape(N, K)
    for k in (0, 33, 127):
        x = np.zeros((1, K), np.float16)
        x[0, k] = 1
        y, _, _, _, _ = oracle.gated_linear(x, qg, sg, qu, su, g)
        for n in range(N):
            a, b = Wg[n, k], Wu[n, k]
            assert y[0, n] == pytest.approx(a / (1.0 + math.exp(-a)) * b, rel=1e-14, abs=1e-300)
        swapped = oracle.silu(Wu[:, k]) * Wg[:, k]
        assert np.max(np.abs(y[0] - swapped)) > 1e-3 * np.max(np.abs(y[0]))


def test_gated_tolerance_covers_linear_errors():
    """Perturbing g and u by their full linear bounds (worst signs) moves
    silu(g) * u by no more than the gated bound (fp64 check of the first-order
    propagation with the cross term)."""
    r = np.random.default_rng(5)
    g = r.normal(0, 3, 20000)
    u = r.normal(0, 3, 20000)
    ag, au = np.abs(g) * 5 + 1, np.abs(u) * 5 + 1
    eg, eu = oracle.tolerance(g, ag), oracle.tolerance(u, au)
    bound = oracle.gated_tolerance(g, u, ag, au)
    y = oracle.silu(g) * u
    for sg_ in (-1, 1):
        for su_ in (-1, 1):
            yp = oracle.silu(g + sg_ * eg) * (u + su_ * eu)
            assert np.all(np.abs(yp - y) <= bound)


def test_gated_tolerance_covers_fp16_rounding_down_to_subnormals():
    """The final rounding to fp16: for exact g and u (zero linear error terms
    apart from the 2^-9 relative part) the bound still covers |fp16(y) - y|
    for y from the largest fp16 values down through the subnormal range
    (spacing 2^-24), where the relative part alone is far too small."""
    r = np.random.default_rng(6)
    y_target = np.concatenate([np.ldexp(1.0, np.arange(-34, 15)),
                               np.exp(r.uniform(np.log(1e-10), np.log(6e4), 20000))])
    y_target *= r.choice([-1.0, 1.0], y_target.size)
    g = np.full_like(y_target, 40.0)          # silu(40) = 40 to 1e-16 relative
    u = y_target / oracle.silu(g)
    y = oracle.silu(g) * u
    zero = np.zeros_like(g)
    bound = oracle.gated_tolerance(g, u, zero, zero)
    err = np.abs(y.astype(np.float16).astype(np.float64) - y)
    assert np.all(err <= bound)
    # the subnormal values need the absolute term: 2^-9 |y| alone does not cover them
    sub = np.abs(y) < np.ldexp(1.0, -14)
    assert np.any(err[sub] > np.ldexp(np.abs(y[sub]), -9) * 3)


# ------------------------------------------------------------------ routed-MoE dispatch

def test_moe_route_hand_worked():
    """logits (0, ln 2, ln 2, ln 4): softmax = (1, 2, 2, 4)/9. Top-2 picks expert 3, then
    the tie between experts 1 and 2 goes to 1; weights 4/9 and 2/9, renormalized 2/3 and
    1/3. Equal logits over E = 4: top-2 is (0, 1) with 1/4 each, renormalized 1/2."""
    l = np.array([[0.0, np.log(2.0), np.log(2.0), np.log(4.0)], [0.5, 0.5, 0.5, 0.5]], np.float32)
    ids, w, _ = oracle.moe_route(l, 2, renormalize=False)
    assert ids.tolist() == [[3, 1], [0, 1]]
    # the fp32 logits are ln 2 and ln 4 rounded, so the weights hold to fp32 accuracy
    assert np.allclose(w, [[4 / 9, 2 / 9], [0.25, 0.25]], rtol=1e-6, atol=0)
    ids, w, _ = oracle.moe_route(l, 2)
    assert ids.tolist() == [[3, 1], [0, 1]]
    assert np.allclose(w, [[2 / 3, 1 / 3], [0.5, 0.5]], rtol=1e-6, atol=0)


def test_moe_route_brute_force():
    """Selection by repeated first-maximum scans and weights from math.exp / math.fsum,
    on small-integer logits with many ties."""
    import math

    r = np.random.default_rng(11)
    T, E, k = 40, 9, 3
    l = r.integers(-3, 4, size=(T, E)).astype(np.float32)
    for renorm in (False, True):
        ids, w, _ = oracle.moe_route(l, k, renormalize=renorm)
        for t in range(T):
            row = [float(v) for v in l[t]]
            taken, pick = set(), []
            for _ in range(k):
                best = None
                for e in range(E):
                    if e not in taken and (best is None or row[e] > row[best]):
                        best = e
                taken.add(best)
                pick.append(best)
            assert ids[t].tolist() == pick
            den = math.fsum(math.exp(v) for v in row)
            ref = [math.exp(row[e]) / den for e in pick]
            if renorm:
                sref = math.fsum(ref)
                ref = [v / sref for v in ref]
            assert np.allclose(w[t], ref, rtol=1e-13, atol=0)


def test_moe_route_invariants():
    r = np.random.default_rng(12)
    l = r.integers(-20, 20, size=(16, 32)).astype(np.float32) / 4  # exact in fp32
    ids, w, ms = oracle.moe_route(l, 32, renormalize=False)
    for t in range(16):
        assert sorted(ids[t].tolist()) == list(range(32))           # k = E: a permutation
        assert np.all(np.diff(l[t][ids[t]]) <= 0)                   # by falling logit
    assert np.allclose(w.sum(1), 1.0, rtol=1e-14)                    # the whole softmax
    ids2, w2, _ = oracle.moe_route(l + np.float32(3.0), 32, renormalize=False)  # shift invariance
    assert np.array_equal(ids, ids2) and np.allclose(w, w2, rtol=1e-13)
    ids, w, _ = oracle.moe_route(l, 5)
    assert np.allclose(w.sum(1), 1.0, rtol=1e-14) and np.all(w > 0)
    assert np.allclose(ms, (l.max(1) - l.min(1)).astype(np.float64))


def test_moe_route_tolerance_covers_fp32_softmax():
    """A plain fp32 evaluation (max, exp of the shifted logit, E-term sum, divisions)
    stays inside route_tolerance."""
    r = np.random.default_rng(13)
    T, E, k = 2000, 128, 8
    l = (r.normal(0, 3, size=(T, E))).astype(np.float32)
    for renorm in (False, True):
        ids, w_ref, ms = oracle.moe_route(l, k, renormalize=renorm)
        m = l.max(1, keepdims=True)
        e32 = np.exp((l - m).astype(np.float32)).astype(np.float32)
        den = np.zeros((T, 1), np.float32)
        for e in range(E):
            den = (den + e32[:, e:e + 1]).astype(np.float32)
        w32 = (np.take_along_axis(e32, ids.astype(np.int64), 1) / den).astype(np.float32)
        if renorm:
            s = np.zeros((T, 1), np.float32)
            for j in range(k):
                s = (s + w32[:, j:j + 1]).astype(np.float32)
            w32 = (w32 / s).astype(np.float32)
        err = np.abs(w32.astype(np.float64) - w_ref)
        assert np.all(err <= oracle.route_tolerance(w_ref, ms, E, k))


def test_moe_dispatch_hand_worked():
    """ids (1, 0), (0, 2), (1, 2): expert 0 holds pairs (0,1), (1,0); expert 1 holds
    (0,0), (2,0); expert 2 holds (1,1), (2,1)."""
    off, row_of, tok = oracle.moe_dispatch(np.array([[1, 0], [0, 2], [1, 2]]), 3)
    assert off.tolist() == [0, 2, 4, 6]
    assert row_of.tolist() == [[2, 0], [1, 4], [3, 5]]
    assert tok.tolist() == [0, 1, 0, 2, 1, 2]


def test_moe_dispatch_brute_force():
    """Rows appended expert by expert, token by token, slot by slot (repeats of an
    expert within a token and empty experts included)."""
    r = np.random.default_rng(14)
    for T, k, E in ((50, 4, 7), (1, 1, 1), (9, 3, 40), (0, 2, 3)):
        ids = r.integers(0, E, size=(T, k))
        off, row_of, tok = oracle.moe_dispatch(ids, E)
        rows, offs = [], [0]
        for e in range(E):
            for t in range(T):
                for j in range(k):
                    if ids[t, j] == e:
                        rows.append((t, j))
            offs.append(len(rows))
        assert off.tolist() == offs
        assert tok.tolist() == [t for t, _ in rows]
        for rr, (t, j) in enumerate(rows):
            assert row_of[t, j] == rr
    with pytest.raises(ValueError):
        oracle.moe_dispatch(np.array([[0, 3]]), 3)


def test_moe_combine_exact():
    """fp16 rows and dyadic weights make every product and sum exact in fp64: compare
    with Fraction arithmetic; one-hot weights pick single rows."""
    from fractions import Fraction

    r = np.random.default_rng(15)
    T, k, N, R = 6, 3, 5, 18
    ys = r.normal(0, 4, size=(R, N)).astype(np.float16)
    row_of = r.permutation(R)[: T * k].reshape(T, k)
    w = r.integers(-64, 64, size=(T, k)) / 64.0
    y, a = oracle.moe_combine(ys, row_of, w)
    for t in range(T):
        for n in range(N):
            ex = sum(Fraction(float(w[t, j])) * Fraction(float(ys[row_of[t, j], n])) for j in range(k))
            ab = sum(abs(Fraction(float(w[t, j])) * Fraction(float(ys[row_of[t, j], n]))) for j in range(k))
            assert Fraction(y[t, n]) == ex and Fraction(a[t, n]) == ab
    onehot = np.zeros((T, k))
    onehot[:, 1] = 1.0
    y1, _ = oracle.moe_combine(ys, row_of, onehot)
    assert np.array_equal(y1, ys[row_of[:, 1]].astype(np.float64))


def test_moe_combine_tolerance_covers_fp32_sum():
    r = np.random.default_rng(16)
    T, k, N = 300, 8, 256
    ys = r.normal(0, 2, size=(T * k, N)).astype(np.float16)
    row_of = r.permutation(T * k).reshape(T, k)
    w = r.random((T, k)).astype(np.float32)
    y_ref, a = oracle.moe_combine(ys, row_of, w)
    acc = np.zeros((T, N), np.float32)
    for j in range(k):
        acc = (acc + w[:, j:j + 1] * ys[row_of[:, j]].astype(np.float32)).astype(np.float32)
    y16 = acc.astype(np.float16).astype(np.float64)
    assert np.all(np.abs(y16 - y_ref) <= oracle.combine_tolerance(y_ref, a, k))


def test_moe_chain_equals_direct_per_token():
    """route -> dispatch -> gather -> grouped_linear -> combine equals, token by token,
    sum_j w_j * (x_t W_{e_j}^T) computed with the dense oracle on each expert's weights."""
    r = np.random.default_rng(17)
    T, E, k, K, N, g = 10, 5, 2, 64, 12, 32
    x = r.normal(0, 1, size=(T, K)).astype(np.float16)
    qw = r.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    s = (np.abs(r.normal(0, 0.02, size=(E, N, K // g))) / 7).astype(np.float16)
    logits = r.normal(0, 1, size=(T, E)).astype(np.float32)
    ids, w, _ = oracle.moe_route(logits, k)
    off, row_of, tok = oracle.moe_dispatch(ids, E)
    ys, _ = oracle.grouped_linear(oracle.moe_gather(x, tok), qw, s, off, g)
    y16 = oracle.float_to_half_bits(ys).view(np.float16)
    y, _ = oracle.moe_combine(y16, row_of, w)
    for t in range(T):
        direct = np.zeros(N)
        for j in range(k):
            yt, _ = oracle.linear(x[t:t + 1], qw[ids[t, j]], s[ids[t, j]], g)
            direct += w[t, j] * oracle.half_to_double(oracle.float_to_half_bits(yt))[0]
        assert np.allclose(y[t], direct, rtol=1e-12, atol=1e-15)


# ------------------------------------------------------- GGUF block formats
# Pins for the Q4_K and Q5_1 decoders: hand-worked blocks (tests/golden/), an
# encoder written here in the inverse direction from the layout (fields ->
# bytes), exact rational sums, and the special case that reduces Q5_1 to a
# plain integer matrix product.

BLOCKS = {"q4_k": (256, 144), "q5_1": (32, 24)}  # weights, bytes per block


def _block_golden(fmt):
    name = {"q4_k": "q4k_block.txt", "q5_1": "q5_1_block.txt"}[fmt]
    raw, values, x, out = bytearray(), {}, {}, {}
    for line in _golden_lines(name):
        key, _, rest = line.partition(" ")
        if key in ("header", "scales", "qs"):
            raw += bytes(int(t, 16) for t in rest.split())
        elif key == "value":
            i, v = rest.split()
            values[int(i)] = float(v)
        elif key == "x":
            x = {int(a): float(b) for a, b in (t.split(":") for t in rest.split())}
        elif key in ("y", "absterm"):
            out[key] = float(rest)
    return bytes(raw), values, x, out


def _fp16_bytes(v):
    return np.array([v], dtype=np.float16).tobytes()  # little-endian on every host we run on


def _enc_q4k(d, dmin, sc, mn, q):
    """Fields -> 144 bytes: sc/mn 6-bit (0..63), q 256 nibbles (0..15)."""
    b = bytearray(144)
    b[0:2], b[2:4] = _fp16_bytes(d), _fp16_bytes(dmin)
    for j in range(4):
        b[4 + j] = sc[j] | (sc[j + 4] >> 4) << 6
        b[8 + j] = mn[j] | (mn[j + 4] >> 4) << 6
        b[12 + j] = (sc[j + 4] & 15) | (mn[j + 4] & 15) << 4
    for i in range(256):
        c, r = divmod(i, 64)
        b[16 + 32 * c + r % 32] |= q[i] if r < 32 else q[i] << 4
    return bytes(b)


def _enc_q51(d, m, q):
    """Fields -> 24 bytes: q 32 values (0..31)."""
    b = bytearray(24)
    b[0:2], b[2:4] = _fp16_bytes(d), _fp16_bytes(m)
    qh = sum(((q[i] >> 4) & 1) << i for i in range(32))
    b[4:8] = qh.to_bytes(4, "little")
    for i in range(16):
        b[8 + i] = (q[i] & 15) | (q[i + 16] & 15) << 4
    return bytes(b)


def _random_fields(fmt, g):
    """One block's fields and its exact weights as Fractions."""
    if fmt == "q4_k":
        d, dmin = np.float16(g.uniform(0.5, 2.0) * 2.0 ** -10), np.float16(g.uniform(0.5, 2.0) * 2.0 ** -11)
        sc, mn = [int(v) for v in g.integers(0, 64, 8)], [int(v) for v in g.integers(0, 64, 8)]
        q = [int(v) for v in g.integers(0, 16, 256)]
        w = [Fraction(float(d)) * sc[i // 32] * q[i] - Fraction(float(dmin)) * mn[i // 32] for i in range(256)]
        return _enc_q4k(d, dmin, sc, mn, q), w
    d, m = np.float16(g.uniform(0.5, 2.0) * 2.0 ** -9), np.float16(-g.uniform(0.5, 2.0) * 2.0 ** -5)
    q = [int(v) for v in g.integers(0, 32, 32)]
    return _enc_q51(d, m, q), [Fraction(float(d)) * q[i] + Fraction(float(m)) for i in range(32)]


def _random_matrix(fmt, g, N, K):
    bw, bb = BLOCKS[fmt]
    rows, exact = [], []
    for _ in range(N):
        parts = [_random_fields(fmt, g) for _ in range(K // bw)]
        rows.append(b"".join(p[0] for p in parts))
        exact.append([v for p in parts for v in p[1]])
    return np.frombuffer(b"".join(rows), np.uint8).reshape(N, K // bw * bb).copy(), exact


@pytest.mark.parametrize("fmt", ["q4_k", "q5_1"])
def test_blocks_golden(fmt):
    raw, values, x, out = _block_golden(fmt)
    bw, bb = BLOCKS[fmt]
    assert len(raw) == bb
    w = np.frombuffer(raw, np.uint8).reshape(1, bb)
    dec = oracle.blocks_decode(fmt, w, bw)[0]
    for i, v in values.items():
        assert dec[i] == v, (fmt, i, dec[i], v)
    xv = np.zeros((1, bw), np.float16)
    for k, v in x.items():
        xv[0, k] = v
    y, a = oracle.blocks_linear(fmt, xv, w)
    assert y[0, 0] == out["y"] and a[0, 0] == out["absterm"]


@pytest.mark.parametrize("fmt", ["q4_k", "q5_1"])
def test_blocks_row_bytes_closed_form(fmt):
    bw, bb = BLOCKS[fmt]
    for nb in (0, 1, 3, 68):
        assert oracle.blocks_row_bytes(fmt, nb * bw) == nb * bb
    assert oracle.blocks_row_bytes(fmt, bw + bw // 2) == -1
    assert oracle.blocks_row_bytes(fmt, -bw) == -1
    assert oracle.blocks_row_bytes(7, bw) == -1


@pytest.mark.parametrize("fmt,N,K", [("q4_k", 3, 512), ("q5_1", 4, 96)])
def test_blocks_decode_inverts_an_encoder(fmt, N, K):
    """Random fields packed by the encoder above decode to exactly d*sc*q - dmin*mn
    (Q4_K) or d*q + m (Q5_1), element by element, across several blocks a row."""
    w, exact = _random_matrix(fmt, workloads.rng(11), N, K)
    dec = oracle.blocks_decode(fmt, w, K)
    for n in range(N):
        for k in range(K):
            assert Fraction(dec[n, k]) == exact[n][k], (fmt, n, k)


@pytest.mark.parametrize("fmt,M,N,K", [("q4_k", 2, 3, 256), ("q5_1", 3, 2, 64)])
def test_blocks_linear_exact_rational(fmt, M, N, K):
    g = workloads.rng(12)
    w, exact = _random_matrix(fmt, g, N, K)
    x = workloads.activations(g, M, K)
    y, a = oracle.blocks_linear(fmt, x, w)
    for m in range(M):
        for n in range(N):
            ref = sum(Fraction(float(x[m, k])) * exact[n][k] for k in range(K))
            assert abs(Fraction(y[m, n]) - ref) <= Fraction(K) * Fraction(2.0 ** -52) * Fraction(a[m, n])
            assert a[m, n] >= abs(y[m, n])


@pytest.mark.parametrize("fmt,K", [("q4_k", 512), ("q5_1", 128)])
def test_blocks_decode_f32_is_the_rounded_exact_value(fmt, K):
    """The fp32 decode is the exact weight rounded once to fp32 (its step and
    offset are exact in fp32 and so is step * q: only the sum rounds)."""
    w, exact = _random_matrix(fmt, workloads.rng(13), 5, K)
    f32 = oracle.blocks_decode_f32(fmt, w, K)
    for n in range(5):
        ref = np.array([float(v) for v in exact[n]], np.float64).astype(np.float32)
        assert np.array_equal(f32[n], ref)


def test_blocks_q5_1_plain_nibbles_match_numpy_matmul():
    """d = 1, m = 0, no fifth bits: W^ is the nibble matrix itself."""
    g = workloads.rng(14)
    N, K, M = 6, 96, 3
    q = g.integers(0, 16, size=(N, K))
    w = np.frombuffer(b"".join(_enc_q51(np.float16(1), np.float16(0), [int(v) for v in q[n, j:j + 32]])
                               for n in range(N) for j in range(0, K, 32)), np.uint8).reshape(N, -1)
    x = workloads.activations(g, M, K)
    assert np.array_equal(oracle.blocks_decode("q5_1", w, K), q.astype(np.float64))
    y, _ = oracle.blocks_linear("q5_1", x, w)
    assert np.allclose(y, x.astype(np.float64) @ q.T.astype(np.float64), rtol=0, atol=1e-9)
