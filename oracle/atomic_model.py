"""Model of an order-free atomic sum, used only to pin the tolerance.

TEST INFRASTRUCTURE (same import rule as the rest of `oracle/`).

The two-shot LL128 AllReduce accumulates the N contributions into a staging
line with floating-point atomic adds in the output dtype; arrival order is
not fixed, so results are not deterministic ("Every Microsecond Matters",
summary page, technique 4). This model performs that accumulation for one
given arrival order: start from zero, and after every add round the partial
sum to the dtype (an atomic add in the dtype returns a dtype value).
It is not used to judge the GPU; tests use it to show that
`allreduce.atomic_tolerance` admits every arrival order and is not vacuous,
and to show where that tolerance stops holding (a 16-bit partial sum that
overflows).

Pins (tests/test_oracle.py): hand-worked arrival orders in
tests/golden/atomic_order_cases.json (ties decided by the order, a partial
that overflows, the +0 start); equality with an exact rational model that
rounds every partial once, over tie-, subnormal- and overflow-heavy inputs;
the float32 carrier against exact roundings of values that sit just off a
midpoint (where rounding to float32 first would double-round); planted
mistakes (no sticky bit, plain float32 rounding, no step toward zero,
unrounded partials, ignored order) each fail one of them.
"""

import numpy as np

from . import fpformats as fp


def _flush(v, dtype):
    """Subnormal values of the format -> zero of the same sign."""
    tiny = np.abs(v) < np.float32(2.0 ** fp.EMIN[dtype])
    return np.where(tiny, np.copysign(np.float32(0), v), v).astype(np.float32)


def atomic_sum(x_bits, order, dtype, flush_subnormals=False):
    """Sum rows of x_bits ([N, count] raw bits) in `order`, rounding each add.

    flush_subnormals: each addition reads a subnormal operand as zero and
    returns zero for a subnormal result (sign kept), as float32 atomic adds
    on the GPU do."""
    vals = fp.decode(np.asarray(x_bits), dtype)
    acc = np.zeros(vals.shape[1], dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        for r in order:
            xr = _flush(vals[r], dtype) if flush_subnormals else vals[r]
            s = (acc + xr).astype(np.float32)
            # the add of two dtype values, rounded once to the dtype. For
            # fp16/bf16 the model takes the float64 sum and a float32
            # carrier that rounds to the dtype like the float64 value does,
            # so that there is visibly one rounding. (A float32 sum would also
            # round innocuously here: 24 >= 2p + 2 for p = 11 and 8.)
            if dtype != fp.FP32:
                s64 = acc.astype(np.float64) + xr.astype(np.float64)
                s = _round64(s64, dtype)
            acc = fp.decode(fp.encode_rne(s, dtype), dtype)
            if flush_subnormals:
                acc = _flush(acc, dtype)
    return fp.encode_rne(acc, dtype)


def _round64(v, dtype):
    """float64 -> float32 value that rounds to the same dtype value as v.

    Used for fp16/bf16 only: a float64 sum of two such values is exact; we
    need a float32 carrier that preserves which side of every dtype rounding
    boundary v lies on. Sticky rounding (round toward zero, then set the
    last float32 bit if inexact) keeps the tie information intact because
    float32 has at least 3 more significand bits than fp16/bf16.
    """
    v = np.asarray(v, dtype=np.float64)
    f = v.astype(np.float32)  # RNE to float32
    back = f.astype(np.float64)
    # move toward zero if float32 rounding went away from zero
    over = np.abs(back) > np.abs(v)
    f_tz = np.where(over, np.nextafter(f, np.float32(0)), f)
    inexact = f_tz.astype(np.float64) != v
    u = f_tz.view(np.uint32) | (inexact.astype(np.uint32))
    return np.where(np.isfinite(v), u.view(np.float32), f)
