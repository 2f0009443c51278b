"""IEEE special values through every protocol, against the CPU oracle.

Columns of signed zeros, subnormals, infinities, quiet NaNs and sums at the
element type's overflow threshold, mixed with ordinary values, at ragged
sizes (one size large enough for the TMA two-shot). The fixed-order
protocols must match the oracle bit for bit, a NaN matching a NaN whatever
its payload (the oracle keeps numpy's NaN bits, the GPU's float32 adds and
conversions return a canonical NaN). The atomic LL128 path must stay
within the atomic tolerance, an infinity matching the same infinity and a
NaN a NaN; it starts each element from +0, so an all-(-0) column gives +0
where the rank-order oracle gives -0 (equal values). Its float32 atomic
additions (red.add.f32) read subnormal operands as zero and return zero for
subnormal results, so for float32 the tolerance adds 2 N 2^-126; a test
pins that behaviour (fp16 and bf16 use .noftz and keep subnormals).

The sentinel protocol reserves the all-ones pattern of the element type;
the NaNs here are the quiet NaNs 0x7FC0.. / 0xFFC0.., never all ones.

Also the domain of the 16-bit LL128 tolerance: its atomics round every
partial sum in the element type, so a partial can overflow where the
float32 sum would not. Below sum |x| <= max - N ulp(max) / 2 no partial can
overflow and the tolerance holds; above it, with cancelling inputs, each
result must be one that some arrival order gives.
"""

import itertools

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from oracle import atomic_model
from oracle import fpformats as fp
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import allreduce, context

PROTOCOLS = ["ll", "sentinel", "fixed_oneshot", "fixed_twoshot", "ll128", "ll128_direct"]
DTYPES = ["fp32", "fp16", "bf16"]
KINDS = ["negzero", "zeromix", "subnormal", "subnormal_cancel", "posinf", "neginf", "infcancel",
         "qnan", "overflow_up", "overflow_below", "normal"]


def _const(v, dtype):
    return int(fp.encode_rne(np.array([v], np.float32), dtype)[0])


def _specials(dtype):
    """Bit patterns used by the columns (all exact in the type)."""
    p, emin = fp.PRECISION[dtype], fp.EMIN[dtype]
    mx = fp.max_finite(dtype)
    half_ulp_max = 2.0 ** (int(np.floor(np.log2(mx))) - p)  # half the spacing at max
    return {
        "pinf": 0x7F800000 if dtype == "fp32" else (0x7C00 if dtype == "fp16" else 0x7F80),
        "ninf": 0xFF800000 if dtype == "fp32" else (0xFC00 if dtype == "fp16" else 0xFF80),
        "pnan": 0x7FC00000 if dtype == "fp32" else (0x7E00 if dtype == "fp16" else 0x7FC0),
        "nnan": 0xFFC00000 if dtype == "fp32" else (0xFE00 if dtype == "fp16" else 0xFFC0),
        "pzero": 0, "nzero": 0x80000000 if dtype == "fp32" else 0x8000,
        "max": _const(mx, dtype),
        # max + half an ulp rounds to +inf; max + a little less stays max
        "half_ulp": _const(half_ulp_max, dtype),
        "below_half_ulp": _const(half_ulp_max * (1 - 2.0 ** -(p - 1)), dtype),
        "min_sub": 1, "sub_bits": (2 ** (p - 1)) - 1,  # largest subnormal's bit pattern
        "emin": emin,
    }


def special_inputs(n, count, dtype, seed):
    """[n, count] raw bits: columns cycling through KINDS in a shuffled order."""
    rng = np.random.default_rng(seed)
    sp = _specials(dtype)
    bdt = fp.BITS_DTYPE[dtype]
    sign = np.uint32(0x80000000 if dtype == "fp32" else 0x8000)
    x = inputs.bits_of(inputs.normal(n, count, dtype, seed=seed)).astype(np.uint32)
    kinds = rng.permutation(np.arange(count) % len(KINDS))
    for i in range(count):
        k = KINDS[kinds[i]]
        col = x[:, i]
        if k == "negzero":
            col[:] = sp["nzero"]
        elif k == "zeromix":
            col[:] = np.where(rng.random(n) < 0.5, sp["nzero"], sp["pzero"])
        elif k in ("subnormal", "subnormal_cancel"):
            mag = rng.integers(1, sp["sub_bits"] + 1, n).astype(np.uint32)
            neg = rng.random(n) < 0.5
            if k == "subnormal_cancel":
                mag[1::2] = mag[0:n - n % 2:2] if n > 1 else mag[1::2]
                neg = np.arange(n) % 2 == 1
            col[:] = mag | np.where(neg, sign, np.uint32(0))
        elif k == "posinf":
            col[rng.integers(0, n)] = sp["pinf"]
        elif k == "neginf":
            col[rng.integers(0, n)] = sp["ninf"]
        elif k == "infcancel":
            a, b = rng.choice(n, 2, replace=False)
            col[a], col[b] = sp["pinf"], sp["ninf"]
        elif k == "qnan":
            col[rng.integers(0, n)] = sp["pnan"] if rng.random() < 0.5 else sp["nnan"]
        elif k in ("overflow_up", "overflow_below"):
            col[:] = sp["pzero"]
            a, b = rng.choice(n, 2, replace=False)
            col[a] = sp["max"]
            col[b] = sp["half_ulp"] if k == "overflow_up" else sp["below_half_ulp"]
            if rng.random() < 0.5:  # the negative mirror image
                col[a] |= sign
                col[b] |= sign
        x[:, i] = col
    return x.astype(bdt)


def assert_same_up_to_nan_payload(got, want, dtype, what):
    g = fp.decode(got, dtype)
    w = fp.decode(np.broadcast_to(want, got.shape), dtype)
    gn, wn = np.isnan(g), np.isnan(w)
    assert np.array_equal(gn, wn), (what, "NaN positions differ")
    same = got == np.broadcast_to(want, got.shape)
    bad = ~same & ~wn
    assert not bad.any(), (what, np.argwhere(bad)[:5].tolist())


def _torch_of(bits, dtype):
    t = torch.from_numpy(bits.view(np.int32 if dtype == "fp32" else np.int16).copy())
    return t.view(inputs.TORCH_DTYPE[dtype])


def test_special_inputs_hit_every_case_in_the_oracle():
    # the generator is not vacuous: the oracle sees every special outcome
    for dtype in DTYPES:
        x = special_inputs(8, 4099, dtype, seed=1)
        y = fp.decode(orc.allreduce(x, dtype)[0], dtype)
        assert np.isnan(y).any() and np.isposinf(y).any() and np.isneginf(y).any()
        assert (np.signbit(y) & (y == 0)).any() and ((~np.signbit(y)) & (y == 0)).any()
        tiny = (y != 0) & (np.abs(y) < 2.0 ** fp.EMIN[dtype])
        assert tiny.any()
        assert (np.abs(y) == fp.max_finite(dtype)).any()
        assert not (x == inputs.SENTINEL_BITS[dtype]).any()


@pytest.mark.gpu
@pytest.mark.parametrize("proto", PROTOCOLS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [2, 5, 8])
def test_special_values_against_oracle(proto, dtype, n):
    with context(n, dtype, 1 << 20):
        for count, seed in ((4099, 10 * n + 1), (40001, 10 * n + 2)):
            xb = special_inputs(n, count, dtype, seed)
            got = allreduce(_torch_of(xb, dtype), dtype, proto)
            want = orc.allreduce(xb, dtype)
            assert all(np.array_equal(got[0], got[r]) for r in range(1, n))
            if proto.startswith("ll128"):
                # float32 atomic adds flush subnormal operands and results
                ok, err, rel = orc.compare_atomic(got, want, xb, dtype, flush_subnormals=dtype == "fp32")
                assert ok, (dtype, n, count, err, rel)
            else:
                assert_same_up_to_nan_payload(got, want[0], dtype, (proto, dtype, n, count))


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_ll128_16bit_tolerance_holds_below_the_overflow_domain_bound(dtype):
    # every column's sum of |x| sits just under max - N ulp(max) / 2, signs random
    n, count = 8, 16384
    mx = fp.max_finite(dtype)
    bound = mx - n * fp.ulp(mx, dtype) / 2
    g = torch.Generator().manual_seed(21)
    v = torch.randn(n, count, generator=g, dtype=torch.float64)
    v = v / v.abs().sum(0, keepdim=True) * bound * (1 - 2.0 ** -7)
    x = v.to(torch.float32).to(inputs.TORCH_DTYPE[dtype])
    xb = inputs.bits_of(x)
    assert np.all(np.sum(np.abs(fp.decode(xb, dtype).astype(np.float64)), axis=0) <= bound)
    with context(n, dtype, 1 << 20):
        got = allreduce(x, dtype, "ll128")
    ok, err, rel = orc.compare_atomic(got, orc.allreduce(xb, dtype), xb, dtype)
    assert ok, (err, rel)
    assert np.isfinite(fp.decode(got, dtype)).all()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_ll128_16bit_partial_overflow_gives_an_arrival_order_result(dtype):
    # two large positives and two large negatives per column, placed on
    # random ranks: the float32 sum is 0, but an order that adds both values
    # of one sign first overflows to an infinity in the element type
    # (for bf16 the pair sums to the overflow threshold (2 - 2^-8) 2^127,
    # finite in float32, which shares bf16's exponent range)
    n, count = 4, 8192
    a, b = {"fp16": (49152.0, 49152.0), "bf16": (2.0 ** 127, (1 - 2.0 ** -8) * 2.0 ** 127)}[dtype]
    rng = np.random.default_rng(22)
    vals = np.array([a, b, -a, -b], np.float32)
    cols = np.stack([rng.permutation(vals) for _ in range(count)], axis=1)
    xb = fp.encode_rne(cols, dtype)
    admitted = {int(v) for order in itertools.permutations(range(4))
                for v in atomic_model.atomic_sum(xb[:, :1], list(order), dtype)}
    assert admitted == {_const(0.0, dtype), _const(np.inf, dtype), _const(-np.inf, dtype)}
    with context(n, dtype, 1 << 20):
        got = allreduce(_torch_of(xb, dtype), dtype, "ll128")
    assert all(np.array_equal(got[0], got[r]) for r in range(1, n))
    outside = [int(v) for v in np.unique(got[0]) if int(v) not in admitted]
    assert not outside, [hex(v) for v in outside]
    # the rank-order oracle gives 0 for every column; the atomic path may not
    assert np.all(orc.allreduce(xb, dtype) == _const(0.0, dtype))


@pytest.mark.gpu
@pytest.mark.parametrize("n", [2, 8])
def test_ll128_fp32_flushes_subnormals_and_16bit_keeps_them(n):
    # every input subnormal: the float32 atomic adds read each as zero, so
    # every output is +0; fp16 / bf16 (.noftz) give the subnormal sums
    count = 4099
    rng = np.random.default_rng(23)
    for dtype in DTYPES:
        p = fp.PRECISION[dtype]
        mag = rng.integers(1, 2 ** (p - 1), (n, count)).astype(np.uint32)
        sign = np.where(rng.random((n, count)) < 0.5, 0x80000000 if dtype == "fp32" else 0x8000, 0)
        xb = (mag | sign.astype(np.uint32)).astype(fp.BITS_DTYPE[dtype])
        with context(n, dtype, 1 << 20):
            got = allreduce(_torch_of(xb, dtype), dtype, "ll128")
        if dtype == "fp32":
            assert np.all(got == 0)
        else:
            ok, err, rel = orc.compare_atomic(got, orc.allreduce(xb, dtype), xb, dtype)
            assert ok, (dtype, err, rel)
            assert np.any(got != 0)


@pytest.mark.gpu
@pytest.mark.parametrize("proto", ["ll", "fixed_oneshot", "sentinel", "ll128"])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [3, 8])
def test_special_values_reduce_scatter(proto, dtype, n):
    # the first half of the two-shot on the same special columns
    count = 4099
    xb = special_inputs(n, count, dtype, seed=40 + n)
    seg = -(-count // n)
    with context(n, dtype, 1 << 20):
        ins = [_torch_of(xb[r], dtype).cuda() for r in range(n)]
        outs = [torch.empty(seg, dtype=inputs.TORCH_DTYPE[dtype], device="cuda") for _ in range(n)]
        llar.llar_reduce_scatter(ins, outs, count, proto)
        torch.cuda.synchronize()
        assert llar.llar_get_status()[0] == llar.OK
    want = orc.reduce_scatter(xb, dtype)
    for s in range(n):
        got = inputs.bits_of(outs[s])[: len(want[s])]
        if proto == "ll128":
            lo, hi = orc.shard_bounds(count, n, s)
            ok, err, rel = orc.compare_atomic(got[None], want[s][None], xb[:, lo:hi], dtype,
                                              flush_subnormals=dtype == "fp32")
            assert ok, (s, err, rel)
        else:
            assert_same_up_to_nan_payload(got[None], want[s], dtype, (proto, dtype, n, s))


@pytest.mark.gpu
@pytest.mark.parametrize("proto", ["ll", "sentinel", "ll128"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_special_values_llbuffer_allreduce(proto, dtype):
    # the AllReduces written on the public device primitives
    n, count = 8, 4099
    xb = special_inputs(n, count, dtype, seed=50)
    with llar.LLBuffer(n, count * inputs.ELEM_BYTES[dtype]) as buf:
        ins = [_torch_of(xb[r], dtype).cuda() for r in range(n)]
        outs = [torch.empty_like(t) for t in ins]
        buf.allreduce(ins, outs, count, dtype, proto)
        torch.cuda.synchronize()
        assert buf.status()[0] == llar.OK
    got = np.stack([inputs.bits_of(o) for o in outs])
    want = orc.allreduce(xb, dtype)
    assert all(np.array_equal(got[0], got[r]) for r in range(1, n))
    if proto == "ll128":
        ok, err, rel = orc.compare_atomic(got, want, xb, dtype, flush_subnormals=dtype == "fp32")
        assert ok, (err, rel)
    else:
        assert_same_up_to_nan_payload(got, want[0], dtype, (proto, dtype))
