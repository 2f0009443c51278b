"""Pins of the linear-layer oracle (oracle/linear.py) and of its float64
rounding (fpformats.encode_rne64), independent of the oracle's own code:
exact rational arithmetic, integer closed forms, identity weights, and a
model of float32 evaluation orders that the tolerance must cover (while a
planted mistake must not fit in it)."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import allreduce as orc
from oracle import fpformats as fp
from oracle import linear as olin

EMAX = {"fp32": 127, "fp16": 15, "bf16": 127}


def rne_fraction(v, dtype):
    """Exact roundTiesToEven of a rational to `dtype`, as a float (or +-inf)."""
    if v == 0:
        return 0.0
    p, emin = fp.PRECISION[dtype], fp.EMIN[dtype]
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    spacing = Fraction(2) ** (e - p + 1)
    q = a / spacing
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * spacing
    maxf = (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** EMAX[dtype]
    out = float("inf") if r > maxf else float(r)
    return -out if v < 0 else out


def _rand_values(dtype, n, rng):
    """bit patterns of finite, non-NaN values of dtype, mixed magnitudes"""
    x = rng.standard_normal(n).astype(np.float32) * np.float32(2.0) ** rng.integers(-10, 10, n).astype(np.float32)
    return fp.encode_rne(x, dtype)


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_encode_rne64_is_one_exact_rounding(dtype):
    rng = np.random.default_rng(11)
    # random float64s, values next to ties of the target format, subnormals
    x = rng.standard_normal(3000) * 2.0 ** rng.integers(-30, 30, 3000)
    base = fp.decode(_rand_values(dtype, 500, rng), dtype).astype(np.float64)
    half = fp.ulp(base, dtype) / 2
    x = np.concatenate([x, base + half, base - half, base + half * (1 + 2.0 ** -30),
                        base + half * (1 - 2.0 ** -30), [fp.max_finite(dtype) * (1 + 2.0 ** -9)],
                        [2.0 ** (fp.EMIN[dtype] - 3) * 1.37, -2.0 ** (fp.EMIN[dtype] - fp.PRECISION[dtype])]])
    got = fp.decode(fp.encode_rne64(x, dtype), dtype).astype(np.float64)
    want = np.array([rne_fraction(Fraction(v), dtype) for v in x])
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_encode_rne64_agrees_with_float32_rounding_on_float32_values(dtype):
    rng = np.random.default_rng(12)
    f32 = (rng.standard_normal(5000) * 1000).astype(np.float32)
    assert np.array_equal(fp.encode_rne64(f32.astype(np.float64), dtype), fp.encode_rne(f32, dtype))


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_partials_equal_exact_rational_dot_rounded_once(dtype):
    rng = np.random.default_rng(13)
    n, m, k, h = 3, 2, 7, 5
    x = _rand_values(dtype, n * m * k, rng).reshape(n, m, k)
    w = _rand_values(dtype, n * k * h, rng).reshape(n, k, h)
    xv = fp.decode(x, dtype).astype(np.float64)
    wv = fp.decode(w, dtype).astype(np.float64)
    got = fp.decode(olin.linear_partials(x, w, dtype), dtype).astype(np.float64)
    for r in range(n):
        for i in range(m):
            for j in range(h):
                exact = sum(Fraction(xv[r, i, t]) * Fraction(wv[r, t, j]) for t in range(k))
                assert got[r, i, j] == rne_fraction(exact, dtype), (r, i, j)


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_identity_weights_reduce_to_allreduce_of_inputs(dtype):
    rng = np.random.default_rng(14)
    n, m, k = 4, 3, 16
    x = _rand_values(dtype, n * m * k, rng).reshape(n, m, k)
    eye = np.broadcast_to(fp.encode_rne(np.eye(k, dtype=np.float32), dtype), (n, k, k))
    got = olin.linear_allreduce(x, eye, dtype)
    want = orc.allreduce(x.reshape(n, m * k), dtype).reshape(n, m, k)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_integer_inputs_give_the_exact_integer_layer(dtype):
    rng = np.random.default_rng(15)
    n, m, k, h = 8, 4, 24, 16
    xi = rng.integers(-3, 4, (n, m, k))
    wi = rng.integers(-2, 3, (n, k, h))
    x = fp.encode_rne(xi.astype(np.float32), dtype)
    w = fp.encode_rne(wi.astype(np.float32), dtype)
    want = sum(xi[r] @ wi[r] for r in range(n))  # |partial| <= 144, |sum| <= 1152
    got = fp.decode(olin.linear_allreduce(x, w, dtype), dtype)
    exact = np.array([[rne_fraction(Fraction(int(v)), dtype) for v in row] for row in want])
    for q in range(n):
        assert np.array_equal(got[q], exact)


def _fma32(a, b, c):
    """float32 fused multiply-add: the exact a*b + c (float64 holds the
    product of two float32s exactly), rounded once to float32. The float64
    addition may round first, but only when |c| is far larger than |a*b|,
    where the double rounding stays inside the bound under test."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def _gpu_like(x_bits, w_bits, dtype, order, slices, fma=False):
    """float32 dot products in a given K order and split (products rounded
    then added, or fused multiply-adds); partials rounded; rank-order float32
    sum."""
    x = fp.decode(x_bits, dtype)
    w = fp.decode(w_bits, dtype)
    n, m, k = x.shape
    h = w.shape[2]
    parts = []
    for r in range(n):
        bounds = np.linspace(0, k, slices + 1).astype(int)
        total = np.zeros((m, h), np.float32)
        for s in range(slices):
            acc = np.zeros((m, h), np.float32)
            for t in order[bounds[s]:bounds[s + 1]]:
                if fma:
                    acc = _fma32(np.broadcast_to(x[r][:, t:t + 1], acc.shape),
                                 np.broadcast_to(w[r][t:t + 1, :], acc.shape), acc)
                else:
                    prod = (x[r][:, t:t + 1] * w[r][t:t + 1, :]).astype(np.float32)
                    acc = (acc + prod).astype(np.float32)
            total = acc if s == 0 else (total + acc).astype(np.float32)
        parts.append(fp.encode_rne(total, dtype))
    p = np.stack(parts)
    return orc.allreduce(p.reshape(n, m * h), dtype).reshape(n, m, h)


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_tolerance_covers_float32_evaluation_orders(dtype):
    rng = np.random.default_rng(16)
    n, m, k, h = 4, 2, 96, 24
    x = fp.encode_rne(rng.standard_normal((n, m, k)).astype(np.float32), dtype)
    w = fp.encode_rne((rng.standard_normal((n, k, h)) * 0.05).astype(np.float32), dtype)
    for trial in range(6):
        order = np.arange(k) if trial == 0 else rng.permutation(k)
        for fma in (False, True):
            got = _gpu_like(x, w, dtype, order, slices=[1, 8, 3, 8, 5, 2][trial], fma=fma)
            ok, rel = olin.compare_linear(got, x, w, dtype)
            assert ok, (trial, fma, rel)


def _toward_zero_sum(x_bits, w_bits, dtype):
    """float32 dot products with every addition rounded toward zero (as an
    accumulator that truncates would), partials rounded to nearest, then
    the rank-order AllReduce."""
    x = fp.decode(x_bits, dtype).astype(np.float64)
    w = fp.decode(w_bits, dtype).astype(np.float64)
    n, m, k = x.shape
    parts = []
    for r in range(n):
        acc = np.zeros((m, w.shape[2]), np.float64)
        for t in range(k):
            exact = acc + x[r][:, t:t + 1] * w[r][t:t + 1, :]
            f = exact.astype(np.float32).astype(np.float64)  # nearest
            toward0 = np.where(np.abs(f) > np.abs(exact), np.nextafter(f.astype(np.float32), np.float32(0)), f)
            acc = np.asarray(toward0, np.float64)
        parts.append(fp.encode_rne(acc.astype(np.float32), dtype))
    p = np.stack(parts)
    return orc.allreduce(p.reshape(n, -1), dtype).reshape(p.shape)


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_default_tolerance_covers_truncating_accumulation(dtype):
    rng = np.random.default_rng(18)
    n, m, k, h = 4, 2, 128, 16
    x = fp.encode_rne(rng.standard_normal((n, m, k)).astype(np.float32), dtype)
    w = fp.encode_rne((rng.standard_normal((n, k, h)) * 0.05).astype(np.float32), dtype)
    got = _toward_zero_sum(x, w, dtype)
    assert olin.compare_linear(got, x, w, dtype)[0]


@pytest.mark.parametrize("dtype", fp.DTYPES)
def test_tolerance_rejects_planted_mistakes(dtype):
    rng = np.random.default_rng(17)
    n, m, k, h = 4, 2, 64, 16
    x = fp.encode_rne(rng.standard_normal((n, m, k)).astype(np.float32), dtype)
    w = fp.encode_rne((rng.standard_normal((n, k, h)) * 0.05).astype(np.float32), dtype)
    good = olin.linear_allreduce(x, w, dtype)
    assert olin.compare_linear(good, x, w, dtype)[0]
    # a dropped K term
    w_drop = w.copy()
    w_drop[:, 5, :] = 0
    assert not olin.compare_linear(olin.linear_allreduce(x, w_drop, dtype), x, w, dtype)[0]
    # a dropped rank
    x0 = x.copy()
    x0[2] = 0
    assert not olin.compare_linear(olin.linear_allreduce(x0, w, dtype), x, w, dtype)[0]
    # w read transposed within square blocks (wrong index)
    wt = w.copy()
    wt[:, :16, :16] = np.swapaxes(w[:, :16, :16], 1, 2)
    assert not olin.compare_linear(olin.linear_allreduce(x, wt, dtype), x, w, dtype)[0]
    # sign error on one rank's partial
    xs = x.copy()
    xs[1] = fp.encode_rne(-fp.decode(x[1], dtype), dtype)
    assert not olin.compare_linear(olin.linear_allreduce(xs, w, dtype), x, w, dtype)[0]
