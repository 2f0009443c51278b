"""CPU oracle for the N-rank sum AllReduce, one-shot and two-shot.

TEST INFRASTRUCTURE. Only `tests/`, `__graft_entry__.smoke()` and the CPU
baseline leg of `bench.py` may import this module. It shares no code with
the CUDA library under `tp_allreduce_persistent_b300/`, and the library
never calls it.

What is computed, and where the pages define it:

* AllReduce: after the collective every rank holds the complete aggregated
  result ("zcube network architecture for LLM inference", section
  "All-Reduce, All-Gather and Reduce-Scatter", collectives table, row
  All-Reduce). In tensor parallelism the aggregation is the sum of the
  per-rank partial outputs (same page, "Why does Tensor Parallel affect
  every token"; "TP All-Reduce and TTFT" page, section 2.1).
* Only addition, only FP32/FP16/BF16 ("Every Microsecond Matters",
  summary page, technique 4).
* Two-shot = ReduceScatter followed by AllGather (same page, technique 4);
  ReduceScatter leaves each rank one reduced segment and AllGather gives
  every rank every segment (zcube page, collectives table, rows
  Reduce-Scatter and All-Gather).

Readings where the pages are silent:

* Accumulation: float32, ranks added in order 0, 1, ..., N-1 with IEEE
  addition (roundTiesToEven, no fused operations), one final
  roundTiesToEven to the buffer's dtype.
* Segments of the two-shot split: rank s owns elements
  [s*ceil(count/N), min(count, (s+1)*ceil(count/N))); the last segments
  may be short or empty.
* Chain mode (dependent AllReduces of a decode step): the next input of
  every rank is roundTiesToEven(scale * float32(output)), the product taken
  in float32.

Arrays are raw bit patterns (see `fpformats`): shape [N, count] for one
AllReduce, [iters, N, count] for a sequence.
"""

import numpy as np

from . import fpformats as fp


def _sum_rank_order(x_bits, dtype):
    """float32 sum over axis 0 (the ranks), added strictly in rank order."""
    vals = fp.decode(x_bits, dtype)
    acc = vals[0].astype(np.float32).copy()
    with np.errstate(over="ignore", invalid="ignore"):
        for r in range(1, vals.shape[0]):
            acc = (acc + vals[r]).astype(np.float32)
    return acc


def allreduce(x_bits, dtype):
    """One-shot AllReduce: every rank's output is the rounded rank-order sum.

    x_bits: [N, count] raw bits. Returns [N, count] raw bits, all rows equal.
    """
    x_bits = np.asarray(x_bits)
    n = x_bits.shape[0]
    y = fp.encode_rne(_sum_rank_order(x_bits, dtype), dtype)
    return np.stack([y] * n, axis=0)


def shard_bounds(count, nranks, s):
    """Element range [lo, hi) of the segment owned by rank s."""
    per = -(-count // nranks) if count else 0
    lo = min(count, s * per)
    hi = min(count, (s + 1) * per)
    return lo, hi


def reduce_scatter(x_bits, dtype):
    """ReduceScatter: rank s keeps the reduced segment s (list of N arrays)."""
    x_bits = np.asarray(x_bits)
    n, count = x_bits.shape
    out = []
    for s in range(n):
        lo, hi = shard_bounds(count, n, s)
        out.append(fp.encode_rne(_sum_rank_order(x_bits[:, lo:hi], dtype), dtype))
    return out


def all_gather(segments, count):
    """AllGather: every rank receives every rank's segment, in rank order."""
    n = len(segments)
    full = np.concatenate(segments) if n else np.zeros(0)
    assert full.shape[0] == count
    return np.stack([full] * n, axis=0)


def allreduce_two_shot(x_bits, dtype):
    """Two-shot AllReduce = AllGather(ReduceScatter(x))."""
    x_bits = np.asarray(x_bits)
    return all_gather(reduce_scatter(x_bits, dtype), x_bits.shape[1])


def chain_next(y_bits, scale, dtype):
    """Next input of a dependent AllReduce: roundTiesToEven(scale * y)."""
    with np.errstate(over="ignore", invalid="ignore"):
        prod = (np.float32(scale) * fp.decode(y_bits, dtype)).astype(np.float32)
    return fp.encode_rne(prod, dtype)


def allreduce_iters(x_bits, iters, dtype, chain_scale=0.0):
    """A sequence of `iters` AllReduces.

    Without a chain (chain_scale == 0), x_bits is [iters, N, count] and
    iteration e reduces x_bits[e]. With a chain, x_bits is [N, count], the
    first input, and iteration e+1 reduces chain_next(output of e).
    Returns [iters, N, count].
    """
    x_bits = np.asarray(x_bits)
    outs = []
    if chain_scale == 0.0:
        assert x_bits.ndim == 3 and x_bits.shape[0] == iters
        for e in range(iters):
            outs.append(allreduce(x_bits[e], dtype))
    else:
        assert x_bits.ndim == 2
        cur = x_bits
        for _ in range(iters):
            y = allreduce(cur, dtype)
            outs.append(y)
            cur = chain_next(y, chain_scale, dtype)
    return np.stack(outs, axis=0)


def atomic_tolerance(x_bits, dtype, flush_subnormals=False):
    """Per-element bound for paths that sum with atomics in any order.

    The LL128 path adds the N contributions with floating-point atomics in
    an unspecified order, so its result is not deterministic ("Every
    Microsecond Matters", summary page, technique 4). The bound allowed
    against the oracle is (N-1) units in the last place of the output dtype,
    taken at sum_r |x_r| (reading: a sum with cancellation has a tiny
    result whose own ulp says nothing about the rounding of the partial
    sums; sum |x_r| bounds every partial sum).

    flush_subnormals: the atomic additions treat a subnormal operand as zero
    and return zero for a subnormal result (the page leaves the atomics'
    arithmetic open; float32 atomic adds on the GPU work that way). Each of
    the N additions then moves by less than the smallest normal 2^emin
    twice (its operand, its result), so 2 N 2^emin is added to the bound.
    """
    x_bits = np.asarray(x_bits)
    n = x_bits.shape[0]
    mag = np.sum(np.abs(fp.decode(x_bits, dtype).astype(np.float64)), axis=0)
    tol = (n - 1) * fp.ulp(mag, dtype)
    if flush_subnormals:
        tol = tol + 2 * n * 2.0 ** fp.EMIN[dtype]
    return tol


def compare_atomic(got_bits, want_bits, x_bits, dtype, flush_subnormals=False):
    """Check an order-free result against the oracle within `atomic_tolerance`.

    Returns (ok, max_abs_err, max_err_in_tolerances). Infinities and NaNs
    must match as classes (same infinity, NaN for NaN).
    """
    got = fp.decode(got_bits, dtype).astype(np.float64)
    want = fp.decode(want_bits, dtype).astype(np.float64)
    tol = np.broadcast_to(atomic_tolerance(x_bits, dtype, flush_subnormals), want.shape)
    nan_ok = np.isnan(got) == np.isnan(want)
    inf_ok = np.where(np.isinf(want) | np.isinf(got), got == want, True)
    finite = np.isfinite(got) & np.isfinite(want)
    with np.errstate(invalid="ignore", over="ignore"):
        err = np.where(finite, np.abs(got - want), 0.0)
    ok = bool(np.all(nan_ok) and np.all(inf_ok) and np.all(err <= tol))
    rel = float(np.max(err / tol)) if err.size else 0.0
    return ok, float(err.max()) if err.size else 0.0, rel
