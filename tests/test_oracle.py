"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here runs the CUDA library. Each test is chosen so that a plausible
mistake in the oracle (a dropped term, a wrong sign or index, a transposed
operand, a different accumulation order or precision, a wrong rounding
rule) makes at least one of them fail.
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from oracle import atomic_model, protocol
from oracle import fpformats as fp
from tp_allreduce_persistent_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ieee_sum_cases.json")


def _bits_array(hexes, dtype):
    return np.array([int(h, 16) for h in hexes], dtype=fp.BITS_DTYPE[dtype])


# ---------------------------------------------------------------- golden cases
def test_golden_ieee_cases():
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) >= 8
    for c in cases:
        dt = c["dtype"]
        x = np.stack([_bits_array(r, dt) for r in c["inputs"]])
        want = _bits_array(c["expected"], dt)
        got = orc.allreduce(x, dt)
        for row in got:
            assert [hex(v) for v in row] == [hex(v) for v in want], c["name"]
        got2 = orc.allreduce_two_shot(x, dt)
        assert np.array_equal(got2, got), c["name"]


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("dtype", fp.DTYPES)
@pytest.mark.parametrize("n", range(2, 9))
def test_rank_id_inputs_sum_to_triangle(dtype, n):
    x = inputs.bits_of(inputs.rank_ids(n, 37, dtype))
    y = fp.decode(orc.allreduce(x, dtype), dtype)
    assert np.all(y == n * (n - 1) / 2)


@pytest.mark.parametrize("dtype,lo,hi", [("fp32", -64, 64), ("fp16", -64, 64), ("bf16", -32, 32)])
def test_integer_inputs_sum_exactly(dtype, lo, hi):
    x = inputs.bits_of(inputs.integers(8, 4096, dtype, seed=11, lo=lo, hi=hi))
    ints = fp.decode(x, dtype).astype(np.int64)
    exact = ints.sum(axis=0)
    y = fp.decode(orc.allreduce(x, dtype), dtype)
    assert np.array_equal(y.astype(np.int64), np.broadcast_to(exact, y.shape))


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_rank_permutation_invariant_when_exact(dtype):
    x = inputs.bits_of(inputs.integers(6, 999, dtype, seed=3, lo=-30, hi=30))
    base = orc.allreduce(x, dtype)
    rng = np.random.default_rng(0)
    for _ in range(5):
        perm = rng.permutation(6)
        assert np.array_equal(orc.allreduce(x[perm], dtype), base)


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_all_outputs_identical_across_ranks(dtype):
    x = inputs.bits_of(inputs.normal(5, 513, dtype, seed=4))
    y = orc.allreduce(x, dtype)
    assert all(np.array_equal(y[0], y[r]) for r in range(5))


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_zero_peers_return_own_input(dtype):
    x = inputs.bits_of(inputs.normal(4, 300, dtype, seed=5))
    x[1:] = 0
    y = orc.allreduce(x, dtype)
    neg_zero = {"fp32": 0x80000000, "fp16": 0x8000, "bf16": 0x8000}[dtype]
    want = np.where(x[0] == neg_zero, 0, x[0])  # -0 + +0 = +0
    assert np.array_equal(y[2], want.astype(y.dtype))


# ----------------------------------------------------- brute force vs exact sum
def _exact_sum_check(x, dtype):
    """|oracle - exact rational sum| within the float32 recursive-summation
    bound plus one final rounding to the dtype."""
    n, count = x.shape
    vals = fp.decode(x, dtype)
    y = fp.decode(orc.allreduce(x, dtype)[0], dtype)
    u = Fraction(1, 2 ** 24)
    gamma = (n - 1) * u / (1 - (n - 1) * u)
    tiny = Fraction(n - 1, 2 ** 150)  # underflow: half the float32 subnormal step per add
    for i in range(count):
        terms = [Fraction(float(vals[r, i])) for r in range(n)]
        exact = sum(terms)
        mag = sum(abs(t) for t in terms)
        bound = gamma * mag + tiny
        if dtype != fp.FP32:
            bound += Fraction(float(fp.ulp(float(abs(exact) + bound), dtype))) / 2
        assert abs(Fraction(float(y[i])) - exact) <= bound, (i, [float(t) for t in terms], float(y[i]))


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_brute_force_against_exact_rational_sum(dtype):
    rng = np.random.default_rng(42)
    for trial in range(40):
        n = int(rng.integers(2, 9))
        count = int(rng.integers(1, 68))
        scale = float(10.0 ** rng.integers(-3, 4))
        x = inputs.bits_of(inputs.normal(n, count, dtype, seed=100 + trial, scale=scale))
        _exact_sum_check(x, dtype)


def test_exact_check_is_sharp_enough_to_catch_mistakes():
    # the bound used above must reject an oracle that drops a term, flips a
    # sign or reads a neighbouring element
    x = inputs.bits_of(inputs.normal(4, 64, "fp32", seed=9))
    vals = fp.decode(x, "fp32").astype(np.float64)
    exact = vals.sum(axis=0)
    mag = np.abs(vals).sum(axis=0)
    bound = 3 * 2.0 ** -24 * mag * 1.01
    wrong = [vals[:3].sum(0), vals[0] - vals[1] + vals[2] + vals[3],
             vals[0] + vals[1] + vals[2] + np.roll(vals[3], 1)]
    for w in wrong:
        assert np.any(np.abs(w - exact) > bound)


# ---------------------------------------------------------------- two-shot
@pytest.mark.parametrize("dtype", fp.DTYPES)
@pytest.mark.parametrize("n,count", [(2, 1), (3, 7), (8, 1), (8, 9), (8, 1000), (5, 64), (7, 130)])
def test_two_shot_equals_one_shot(dtype, n, count):
    x = inputs.bits_of(inputs.normal(n, count, dtype, seed=count + n))
    assert np.array_equal(orc.allreduce_two_shot(x, dtype), orc.allreduce(x, dtype))


@pytest.mark.parametrize("n,count", [(2, 0), (2, 1), (8, 7), (8, 64), (3, 10), (8, 1025)])
def test_shard_bounds_partition(n, count):
    seen = []
    per = -(-count // n) if count else 0
    for s in range(n):
        lo, hi = orc.shard_bounds(count, n, s)
        assert 0 <= lo <= hi <= count
        assert hi - lo <= per
        seen.extend(range(lo, hi))
    assert seen == list(range(count))


@pytest.mark.parametrize("n,count", [(3, 10), (8, 8195), (4, 2)])
def test_reduce_scatter_and_all_gather_closed_forms(n, count):
    # rank-id inputs: every element of every segment sums to n(n-1)/2
    x = inputs.bits_of(inputs.rank_ids(n, count, "fp32"))
    segs = orc.reduce_scatter(x, "fp32")
    assert [len(sg) for sg in segs] == [hi - lo for lo, hi in (orc.shard_bounds(count, n, s) for s in range(n))]
    assert all(np.all(fp.decode(sg, "fp32") == n * (n - 1) / 2) for sg in segs)
    # gathering segments filled with their own rank id puts value s at
    # exactly the elements of segment s, on every rank
    own = [fp.encode_rne(np.full(len(sg), s, np.float32), "fp32") for s, sg in enumerate(segs)]
    out = fp.decode(orc.all_gather(own, count), "fp32")
    per = -(-count // n)
    want = np.array([i // per for i in range(count)], np.float32)
    assert all(np.array_equal(out[q], want) for q in range(n))


# ---------------------------------------------------------------- chains
@pytest.mark.parametrize("dtype", fp.DTYPES)
@pytest.mark.parametrize("n", [4, 8])
def test_chain_closed_form_half(dtype, n):
    # rank-id inputs, scale 1/2: every rank holds T = n(n-1)/2 after step 0,
    # then each step sums n copies of half the previous result, so
    # y_e = T * (n/2)^e exactly, until it passes the dtype's overflow
    # threshold max + ulp/2, from which on it is +inf.
    iters = 160
    x = inputs.bits_of(inputs.rank_ids(n, 5, dtype))
    y = fp.decode(orc.allreduce_iters(x, iters, dtype, chain_scale=0.5), dtype)
    t = Fraction(n * (n - 1), 2)
    limit = Fraction(fp.max_finite(dtype)) + Fraction(float(fp.ulp(fp.max_finite(dtype), dtype))) / 2
    for e in range(iters):
        exact = t * Fraction(n, 2) ** e
        want = float(exact) if exact < limit else np.inf
        assert np.all(y[e] == want), (e, y[e][0, 0], want)


@pytest.mark.parametrize("dtype", fp.DTYPES)
@pytest.mark.parametrize("n", [4, 8])
def test_chain_scale_one_over_n_is_stationary(dtype, n):
    x = inputs.bits_of(inputs.integers(n, 33, dtype, seed=n, lo=-8, hi=8))
    y = orc.allreduce_iters(x, 20, dtype, chain_scale=1.0 / n)
    assert all(np.array_equal(y[0], y[e]) for e in range(20))


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_chain_next_halves_exactly(dtype):
    y = inputs.bits_of(inputs.normal(1, 2000, dtype, seed=8))[0]
    v = fp.decode(y, dtype).astype(np.float64)
    h = fp.decode(orc.chain_next(y, 0.5, dtype), dtype).astype(np.float64)
    normal = np.abs(v) >= 2.0 ** (fp.EMIN[dtype] + 1)
    assert np.array_equal(h[normal], v[normal] / 2)


def test_fresh_input_sequence_is_per_iteration():
    x = inputs.bits_of(inputs.uniform(2, 32, "fp32", seed=0, iters=6))
    y = orc.allreduce_iters(x, 6, "fp32")
    for e in range(6):
        assert np.array_equal(y[e], orc.allreduce(x[e], "fp32"))


# ------------------------------------------------------------ format helpers
def _structured_f32():
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], dtype=np.uint32)
    a = (hi[:, None] | lows[None, :]).ravel()
    rng = np.random.default_rng(1)
    b = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([a, b]).view(np.float32)


def test_bf16_rne_matches_torch_cast():
    f = _structured_f32()
    ours = fp.encode_rne(f, "bf16")
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(fp.is_nan_bits(ours[nan], "bf16"))


def test_fp16_rne_matches_torch_cast():
    f = _structured_f32()
    with np.errstate(over="ignore"):
        ours = fp.encode_rne(f, "fp16")
    ref = torch.from_numpy(f.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(fp.is_nan_bits(ours[nan], "fp16"))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_decode_encode_roundtrip_all_patterns(dtype):
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = fp.decode(b, dtype)
    back = fp.encode_rne(v, dtype)
    nan = np.isnan(v)
    assert np.array_equal(back[~nan], b[~nan])
    ref = torch.from_numpy(b.view(np.int16).copy()).view(inputs.TORCH_DTYPE[dtype]).float().numpy()
    assert np.array_equal(v[~nan], ref[~nan])


def test_ulp_closed_forms():
    assert fp.ulp(1.0, "fp32") == 2.0 ** -23
    assert fp.ulp(1.0, "fp16") == 2.0 ** -10
    assert fp.ulp(1.0, "bf16") == 2.0 ** -7
    assert fp.ulp(1.5, "bf16") == 2.0 ** -7
    assert fp.ulp(2.0, "bf16") == 2.0 ** -6
    assert fp.ulp(65504.0, "fp16") == 32.0
    assert fp.ulp(0.0, "fp16") == 2.0 ** -24
    assert fp.ulp(0.0, "fp32") == 2.0 ** -149
    assert fp.ulp(0.0, "bf16") == 2.0 ** -133
    assert fp.ulp(-3.0, "fp32") == 2.0 ** -22
    assert fp.max_finite("fp16") == 65504.0
    assert fp.max_finite("bf16") == float(np.float32(3.3895314e38))


# ------------------------------------------------------ atomic-path tolerance
@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_atomic_tolerance_admits_every_arrival_order(dtype):
    rng = np.random.default_rng(7)
    x = inputs.bits_of(inputs.normal(8, 2000, dtype, seed=12))
    want = orc.allreduce(x, dtype)
    worst = 0.0
    for _ in range(12):
        order = rng.permutation(8)
        got = atomic_model.atomic_sum(x, order, dtype)
        ok, _, rel = orc.compare_atomic(np.stack([got] * 8), want, x, dtype)
        assert ok
        worst = max(worst, rel)
    assert worst > 0.0 or dtype == "fp32"  # 16-bit atomics do round differently


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_atomic_tolerance_rejects_a_lost_contribution(dtype):
    x = inputs.bits_of(inputs.normal(8, 500, dtype, seed=13))
    want = orc.allreduce(x, dtype)
    lost = orc.allreduce(x[:7], dtype)[:1]
    ok, _, _ = orc.compare_atomic(np.concatenate([lost] * 8), want, x, dtype)
    assert not ok


def test_atomic_tolerance_closed_form():
    x = np.stack([fp.encode_rne(np.array([1.0], np.float32), "bf16")] * 2)
    assert orc.atomic_tolerance(x, "bf16")[0] == 2.0 ** -6  # (N-1) ulp(2) in bf16


def test_atomic_model_of_identical_values_matches_oracle():
    # n copies of one value: every order gives the same partial sums k*v
    x = np.stack([fp.encode_rne(np.array([0.3, -1.7, 5.0], np.float32), "fp32")] * 4)
    for order in ([0, 1, 2, 3], [3, 2, 1, 0]):
        assert np.array_equal(atomic_model.atomic_sum(x, order, "fp32"), orc.allreduce(x, "fp32")[0])


# ----------------------------------------------- atomic model: exact pins
ATOMIC_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "atomic_order_cases.json")
FORMAT = {"fp32": (24, -126, 127), "fp16": (11, -14, 15), "bf16": (8, -126, 127)}


def _bits_of_value(v, dtype):
    """Bits of a value that the format holds exactly (no rounding happens)."""
    if dtype == "fp16":
        return int(np.array([v], np.float16).view(np.uint16)[0])
    u = int(np.array([v], np.float32).view(np.uint32)[0])
    return u >> 16 if dtype == "bf16" else u


def _round_exact(q, neg_zero, dtype):
    """roundTiesToEven of the rational q to `dtype`, from the definition
    (IEEE 754-2008 4.3.1, 7.4); returns bits. An exact zero keeps the sign
    IEEE 6.3 gives it (neg_zero)."""
    p, emin, emax = FORMAT[dtype]
    if q == 0:
        return _bits_of_value(-0.0 if neg_zero else 0.0, dtype)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)  # subnormals share the quantum of the smallest binade
    quantum = Fraction(2) ** (e - p + 1)
    m = a / quantum
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * quantum
    if v >= Fraction(2) ** (emax + 1):
        return _bits_of_value(sign * float("inf"), dtype)
    return _bits_of_value(sign * float(v), dtype)


def _exact_atomic_sum(x_bits, order, dtype):
    """Per element: start from +0, add the ranks in `order`, each sum exact
    as a rational and then rounded once to `dtype` (finite inputs; a partial
    that overflows stays infinite)."""
    vals = fp.decode(x_bits, dtype).astype(np.float64)
    out = []
    for i in range(vals.shape[1]):
        acc, neg, inf = Fraction(0), False, 0.0
        for r in order:
            xv = float(vals[r, i])
            if inf:
                continue
            xneg = xv == 0 and np.signbit(xv)
            s = acc + Fraction(xv)
            neg = s == 0 and neg and xneg
            bits = _round_exact(s, neg, dtype)
            v = float(fp.decode(np.array([bits], fp.BITS_DTYPE[dtype]), dtype)[0])
            if np.isinf(v):
                inf = v
            else:
                acc = Fraction(v)
        out.append(_bits_of_value(inf, dtype) if inf else _round_exact(acc, neg, dtype))
    return np.array(out, dtype=fp.BITS_DTYPE[dtype])


def _hard_atomic_inputs(n, count, dtype, seed):
    """Finite values built to hit ties, subnormals, cancellation and the
    overflow threshold: a shared magnitude per element with small offsets,
    random exponents over the whole range, and halves of the spacing."""
    p, emin, emax = FORMAT[dtype]
    rng = np.random.default_rng(seed)
    base = rng.integers(emin - p + 2, emax + 1, count)
    kind = rng.integers(0, 4, (n, count))
    x = np.zeros((n, count), np.float64)
    for r in range(n):
        for i in range(count):
            mant = 1.0 + rng.integers(0, 2 ** (p - 1)) / 2.0 ** (p - 1)
            sgn = -1.0 if rng.random() < 0.4 else 1.0
            k = kind[r, i]
            if k == 0:  # same binade as the element's base
                ex = base[i]
            elif k == 1:  # half a spacing of the base binade, or a few spacings
                ex = base[i] - p + int(rng.integers(0, 3))
            elif k == 2:  # anywhere in the range, subnormals included
                ex = int(rng.integers(emin - p + 1, emax + 1))
            else:
                ex = base[i] - int(rng.integers(0, p + 3))
            x[r, i] = sgn * np.ldexp(mant, int(ex))
    bits = fp.encode_rne(x.astype(np.float32), dtype)
    vals = fp.decode(bits, dtype)
    return np.where(np.isfinite(vals), bits, np.zeros_like(bits))


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_atomic_model_equals_exact_per_add_rounding(dtype):
    # every partial sum rounded once to the element type, checked against
    # exact rational arithmetic for several arrival orders
    rng = np.random.default_rng(41)
    for n, count, seed in ((2, 300, 1), (5, 200, 2), (8, 150, 3)):
        x = _hard_atomic_inputs(n, count, dtype, seed)
        for _ in range(3):
            order = [int(v) for v in rng.permutation(n)]
            got = atomic_model.atomic_sum(x, order, dtype)
            want = _exact_atomic_sum(x, order, dtype)
            assert np.array_equal(got, want), (dtype, n, order)


def _atomic_golden_orders_hold(fn):
    for c in json.load(open(ATOMIC_GOLDEN))["orders"]:
        dt = c["dtype"]
        x = np.stack([_bits_array(r, dt) for r in c["inputs"]])
        got = fn(x, c["order"], dt)
        if [hex(v) for v in got] != [hex(v) for v in _bits_array(c["expected"], dt)]:
            return False
    return True


def _carrier_golden_holds(fn):
    for c in json.load(open(ATOMIC_GOLDEN))["carrier"]["cases"]:
        v = np.array([sum(s * 2.0 ** k for s, k in c["terms"])], np.float64)
        exact = sum(Fraction(s) * Fraction(2) ** k for s, k in c["terms"])
        assert float(exact) == v[0]  # the float64 literal holds the value exactly
        got = int(fp.encode_rne(fn(v, c["dtype"]), c["dtype"])[0])
        if got != int(c["expected"], 16):
            return False
    return True


def test_atomic_model_golden_orders():
    assert _atomic_golden_orders_hold(atomic_model.atomic_sum)
    # and the exact model agrees with the hand-worked values
    assert _atomic_golden_orders_hold(_exact_atomic_sum)


def test_atomic_golden_overflow_case_breaks_the_tolerance():
    # reading: 16-bit atomics round every partial in the element type, so a
    # partial that passes the largest finite value becomes inf even where the
    # float32 sum is finite; the tolerance only holds while sum |x| stays
    # below the overflow threshold
    x = np.stack([_bits_array(["7a00"], "fp16"), _bits_array(["7a00"], "fp16"), _bits_array(["fa00"], "fp16")])
    want = orc.allreduce(x, "fp16")
    bad = atomic_model.atomic_sum(x, [0, 1, 2], "fp16")
    good = atomic_model.atomic_sum(x, [0, 2, 1], "fp16")
    assert not orc.compare_atomic(np.stack([bad] * 3), want, x, "fp16")[0]
    assert orc.compare_atomic(np.stack([good] * 3), want, x, "fp16")[0]


def test_carrier_rounds_like_the_exact_value():
    assert _carrier_golden_holds(atomic_model._round64)


def test_float32_sum_of_two_16bit_values_rounds_innocuously():
    # why the carrier is only reachable through its own pins: float32 has
    # p32 = 24 >= 2 p + 2 bits for fp16 (p = 11) and bf16 (p = 8), so a
    # float32 sum of two such values followed by rounding to the format is
    # the correctly rounded sum (innocuous double rounding, Figueroa 1995)
    rng = np.random.default_rng(43)
    for dtype in ("fp16", "bf16"):
        x = _hard_atomic_inputs(2, 3000, dtype, 44)
        s32 = (fp.decode(x[0], dtype) + fp.decode(x[1], dtype)).astype(np.float32)
        with np.errstate(over="ignore"):
            got = fp.encode_rne(s32, dtype)
        want = _exact_atomic_sum(x, [0, 1], dtype)
        vals = fp.decode(x, dtype)
        nz = (vals[0] != 0) | (vals[1] != 0)  # signed zeros: both rules agree, skip the start value
        assert np.array_equal(got[nz], want[nz]), dtype
    del rng


def test_flushing_atomic_model_golden_cases():
    # the flush reading of float32 atomic adds: hand-worked cases, the plain
    # tolerance rejects them, the flush-aware one admits them
    for c in json.load(open(ATOMIC_GOLDEN))["flush"]["cases"]:
        dt = c["dtype"]
        x = np.stack([_bits_array(r, dt) for r in c["inputs"]])
        got = atomic_model.atomic_sum(x, c["order"], dt, flush_subnormals=True)
        assert [hex(v) for v in got] == [hex(v) for v in _bits_array(c["expected"], dt)], c["name"]
        want = orc.allreduce(x, dt)
        assert [hex(v) for v in want[0]] == [hex(v) for v in _bits_array(c["oracle"], dt)], c["name"]
        ys = np.stack([got] * x.shape[0])
        assert orc.compare_atomic(ys, want, x, dt, flush_subnormals=True)[0], c["name"]
        assert orc.compare_atomic(ys, want, x, dt)[0] == c["plain_tolerance_admits"], c["name"]


def test_flush_aware_tolerance_admits_every_order_and_still_rejects_a_lost_term():
    rng = np.random.default_rng(45)
    n, count = 8, 3000
    # subnormal-heavy float32 data: subnormals, values near the smallest
    # normal of both signs, and a few ordinary ones
    mags = np.where(rng.random((n, count)) < 0.6,
                    rng.integers(1, 2 ** 23, (n, count)),
                    rng.integers(2 ** 23, 2 ** 25, (n, count))).astype(np.uint32)
    sign = np.where(rng.random((n, count)) < 0.5, np.uint32(0x80000000), np.uint32(0))
    x = mags | sign
    x[:, :50] = fp.encode_rne(rng.standard_normal((n, 50)).astype(np.float32), "fp32")
    want = orc.allreduce(x, "fp32")
    needed = False
    for _ in range(6):
        order = [int(v) for v in rng.permutation(n)]
        got = np.stack([atomic_model.atomic_sum(x, order, "fp32", flush_subnormals=True)] * n)
        assert orc.compare_atomic(got, want, x, "fp32", flush_subnormals=True)[0]
        needed |= not orc.compare_atomic(got, want, x, "fp32")[0]
    assert needed  # the plain bound alone would not admit the flushing adds
    lost = np.stack([orc.allreduce(x[:7], "fp32")[0]] * n)
    lost_ok = orc.compare_atomic(lost[:, :50], want[:, :50], x[:, :50], "fp32", flush_subnormals=True)[0]
    assert not lost_ok


def test_atomic_model_pins_catch_planted_mistakes():
    # each plausible mistake in the model fails at least one pin above
    def no_sticky(v, dtype):
        v = np.asarray(v, dtype=np.float64)
        f = v.astype(np.float32)
        over = np.abs(f.astype(np.float64)) > np.abs(v)
        return np.where(over, np.nextafter(f, np.float32(0)), f)

    def double_rounding(v, dtype):
        return np.asarray(v, dtype=np.float64).astype(np.float32)

    def sticky_without_toward_zero(v, dtype):
        v = np.asarray(v, dtype=np.float64)
        f = v.astype(np.float32)
        inexact = f.astype(np.float64) != v
        return (f.view(np.uint32) | inexact.astype(np.uint32)).view(np.float32)

    for bad in (no_sticky, double_rounding, sticky_without_toward_zero):
        assert not _carrier_golden_holds(bad), bad.__name__

    def unrounded_partials(x_bits, order, dtype):  # one rounding at the end
        vals = fp.decode(np.asarray(x_bits), dtype).astype(np.float64)
        acc = np.zeros(vals.shape[1])
        for r in order:
            acc = acc + vals[r]
        return fp.encode_rne(atomic_model._round64(acc, dtype) if dtype != "fp32"
                             else acc.astype(np.float32), dtype)

    def ignores_order(x_bits, order, dtype):
        return atomic_model.atomic_sum(x_bits, sorted(order), dtype)

    for bad in (unrounded_partials, ignores_order):
        assert not _atomic_golden_orders_hold(bad), bad.__name__


# -------------------------------------------------------- protocol constants
def test_ll_line_halves_bandwidth_and_doubles_staging():
    assert protocol.ll_payload_fraction() == 0.5
    assert protocol.ll_staging_bytes(16384) == 32768
    assert protocol.ll_staging_bytes(12) == 32


def test_ll128_flag_overhead_matches_page_percentages():
    # "about 1.5% in FP16, about 3% in FP32"
    assert abs(protocol.ll128_overhead("fp16") * 100 - 1.5) < 0.1
    assert abs(protocol.ll128_overhead("fp32") * 100 - 3.0) < 0.15
    assert protocol.ll128_payload_elems("fp16") == 63
    assert protocol.ll128_payload_elems("bf16") == 63
    assert protocol.ll128_payload_elems("fp32") == 31
    assert protocol.LL128_LINE_BYTES == protocol.LL128_GROUP_THREADS * 16


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_ll128_staging_is_about_d_over_n(dtype):
    n = 8
    for nbytes in (1 << 20, 1 << 22):
        count = nbytes // fp.ELEM_BYTES[dtype]
        s = protocol.ll128_round_staging_bytes(count, n, dtype)
        ratio = s / (nbytes / n)
        assert 1.0 < ratio < 1.0 + 1.5 * protocol.ll128_overhead(dtype)


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_sentinel_is_a_negative_nan(dtype):
    b = np.array([protocol.sentinel_bits(dtype)], dtype=fp.BITS_DTYPE[dtype])
    v = fp.decode(b, dtype)
    assert np.isnan(v[0]) and np.signbit(v[0])
    assert protocol.sentinel_refilled(np.full(10, protocol.sentinel_bits(dtype), fp.BITS_DTYPE[dtype]), dtype)
    assert not protocol.sentinel_refilled(np.zeros(10, fp.BITS_DTYPE[dtype]), dtype)


# ---------------------------------------------------------------- point to point
def test_p2p_ring_shift_n_times_is_identity():
    from oracle import p2p
    rng = np.random.default_rng(31)
    n = 5
    x = rng.integers(0, 2 ** 16, (n, 13), dtype=np.uint16)
    ring = [(r + 1) % n for r in range(n)]
    y = x
    for _ in range(n):
        y = p2p.sendrecv(y, ring, np.zeros_like(x))
    assert np.array_equal(y, x)
    # one shift moves row r to row r + 1 (and not the other way round)
    one = p2p.sendrecv(x, ring, np.zeros_like(x))
    assert np.array_equal(one[1], x[0]) and np.array_equal(one[0], x[n - 1])


def test_p2p_permutation_then_inverse_restores_and_idle_rows_keep_fill():
    from oracle import p2p
    rng = np.random.default_rng(32)
    n = 7
    perm = [3, 0, 5, 1, 6, 2, 4]
    inv = [perm.index(q) for q in range(n)]
    x = rng.integers(0, 2 ** 32, (n, 9), dtype=np.uint32)
    assert np.array_equal(p2p.sendrecv(p2p.sendrecv(x, perm, 0 * x), inv, 0 * x), x)
    fill = np.full_like(x, 7)
    part = p2p.sendrecv(x, [2, -1, -1, -1, -1, -1, 0], fill)
    assert np.array_equal(part[2], x[0]) and np.array_equal(part[0], x[6])
    assert all(np.array_equal(part[q], fill[q]) for q in (1, 3, 4, 5, 6))


@pytest.mark.parametrize("dst", [[0, 1], [1, 1, -1], [3, 0], [1, 0, 1]])
def test_p2p_invalid_maps_rejected(dst):
    from oracle import p2p
    with pytest.raises(ValueError):
        p2p.sources(dst)
