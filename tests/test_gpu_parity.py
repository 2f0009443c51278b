"""Parity of every protocol with the CPU oracle, through the C ABI.

Fixed-order protocols (LL, SENTINEL, FIXED_ONESHOT, FIXED_TWOSHOT) must
match bit for bit; LL128_ATOMIC, whose atomic accumulation order is free,
must stay within (N-1) ulp of the output dtype at sum_r |x_r| and be exact
on integer-valued inputs. Every rank's output must equal every other's.
Sizes span several CTAs, several words per thread and ragged tails.
"""

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import allreduce, allreduce_iters, context

pytestmark = pytest.mark.gpu

FIXED_ORDER = ["ll", "sentinel", "fixed_oneshot", "fixed_twoshot"]
DTYPES = ["fp32", "fp16", "bf16"]
COUNTS = [1, 3, 8, 31, 64, 129, 1000, 4099, 16389]


def _ranks_identical(y):
    assert all(np.array_equal(y[0], y[r]) for r in range(1, y.shape[0]))


@pytest.mark.parametrize("proto", FIXED_ORDER)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_fixed_order_bit_exact(proto, dtype, n):
    with context(n, dtype, 1 << 20):
        for i, count in enumerate(COUNTS):
            x = inputs.normal(n, count, dtype, seed=1000 + 17 * n + i)
            got = allreduce(x, dtype, proto)
            want = orc.allreduce(inputs.bits_of(x), dtype)
            assert np.array_equal(got, want), (proto, dtype, n, count)
            _ranks_identical(got)


@pytest.mark.parametrize("proto", ["ll128", "ll128_direct"])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_ll128_within_tolerance(proto, dtype, n):
    with context(n, dtype, 1 << 20):
        for i, count in enumerate(COUNTS):
            x = inputs.normal(n, count, dtype, seed=2000 + 17 * n + i)
            got = allreduce(x, dtype, proto)
            xb = inputs.bits_of(x)
            ok, err, rel = orc.compare_atomic(got, orc.allreduce(xb, dtype), xb, dtype)
            assert ok, (dtype, n, count, err, rel)
            _ranks_identical(got)


@pytest.mark.parametrize("proto", ["ll128", "ll128_direct"])
@pytest.mark.parametrize("dtype,lo,hi", [("fp32", -64, 64), ("fp16", -64, 64), ("bf16", -32, 32)])
def test_ll128_exact_on_integers(proto, dtype, lo, hi):
    with context(8, dtype, 1 << 20):
        for count in (63, 1000, 32768):
            x = inputs.integers(8, count, dtype, seed=count, lo=lo, hi=hi)
            got = allreduce(x, dtype, proto)
            assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), dtype))


@pytest.mark.parametrize("proto", FIXED_ORDER + ["ll128", "ll128_direct"])
def test_rank_id_inputs(proto):
    for n in (2, 8):
        with context(n, "bf16", 1 << 16):
            x = inputs.rank_ids(n, 777, "bf16")
            got = allreduce(x, "bf16", proto)
            assert np.all(got == inputs.bits_of(torch.full((1,), n * (n - 1) / 2).to(torch.bfloat16))[0])


@pytest.mark.parametrize("proto,shapes", [
    ("ll", [(1, 32), (3, 64), (7, 96), (18, 512)]),
    ("sentinel", [(1, 32), (2, 64), (5, 128), (16, 256)]),
    ("ll128", [(1, 32), (3, 64), (9, 256), (18, 512)]),
    ("ll128_direct", [(1, 32), (3, 64), (9, 256), (18, 512)]),
    ("fixed_oneshot", [(1, 32), (4, 64), (37, 256)]),
    ("fixed_twoshot", [(1, 32), (4, 96), (74, 256)]),
])
def test_launch_shapes(proto, shapes):
    # several words per thread, idle CTAs, uneven splits
    dtype, n = "fp16", 4
    with context(n, dtype, 1 << 20):
        for g, t in shapes:
            llar.llar_set_launch(g, t)
            for count in (5, 2053, 70001):
                x = inputs.normal(n, count, dtype, seed=g * 1000 + t + count)
                got = allreduce(x, dtype, proto)
                xb = inputs.bits_of(x)
                want = orc.allreduce(xb, dtype)
                if proto.startswith("ll128"):
                    assert orc.compare_atomic(got, want, xb, dtype)[0]
                else:
                    assert np.array_equal(got, want), (g, t, count)


@pytest.mark.parametrize("chunk", [16, 256, 4096, 65536])
def test_sentinel_chunk_sizes(chunk):
    dtype, n = "bf16", 8
    with context(n, dtype, 1 << 20):
        llar.llar_set_sentinel_chunk(chunk)
        for count in (9, 3000, 65536 + 3):
            x = inputs.normal(n, count, dtype, seed=chunk + count)
            got = allreduce(x, dtype, "sentinel")
            assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), dtype))


@pytest.mark.parametrize("proto", FIXED_ORDER + ["ll128", "ll128_direct"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_iters_fresh_inputs(proto, dtype):
    n, iters = 4, 9
    with context(n, dtype, 1 << 20):
        for count in (13, 4096, 9001):
            x = inputs.uniform(n, count, dtype, seed=count, iters=iters)
            got = allreduce_iters(x, dtype, proto, iters)
            xb = inputs.bits_of(x)
            want = orc.allreduce_iters(xb, iters, dtype)
            if proto.startswith("ll128"):
                for e in range(iters):
                    assert orc.compare_atomic(got[e], want[e], xb[e], dtype)[0], e
            else:
                assert np.array_equal(got, want)


@pytest.mark.parametrize("proto", FIXED_ORDER)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("scale", [0.5, 0.25])
def test_chain_bit_exact(proto, dtype, scale):
    n, iters = 4, 24
    with context(n, dtype, 1 << 20):
        for count in (7, 8192, 20001):
            x = inputs.normal(n, count, dtype, seed=count, scale=0.02)
            got = allreduce_iters(x, dtype, proto, iters, chain_scale=scale)
            want = orc.allreduce_iters(inputs.bits_of(x), iters, dtype, chain_scale=scale)
            assert np.array_equal(got, want), (proto, dtype, count)


@pytest.mark.parametrize("proto", ["ll128", "ll128_direct"])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [2, 4, 8])
def test_chain_ll128_exact_fixed_point(n, dtype, proto):
    # integers in [-2, 2] with scale 1/N (a power of two): every partial sum
    # of every step is exact in every element type, so the atomic chain must
    # equal the oracle's chain bit for bit (it settles on a fixed point after
    # the first step: N copies of y/N sum to y)
    iters = 12
    with context(n, dtype, 1 << 20):
        for count in (7, 8192, 20001):
            x = inputs.integers(n, count, dtype, seed=count + n, lo=-2, hi=2)
            got = allreduce_iters(x, dtype, proto, iters, chain_scale=1.0 / n)
            assert np.array_equal(got, orc.allreduce_iters(inputs.bits_of(x), iters, dtype, chain_scale=1.0 / n))


@pytest.mark.parametrize("proto", ["ll128", "ll128_direct"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_chain_ll128_general_data(dtype, proto):
    # atomic sums may differ from the oracle in the last place, and a chain
    # carries that on: the first step is held to the atomic tolerance, every
    # step to what must hold whatever the order (every rank the same result,
    # finite where the oracle's chain is finite)
    n, iters, scale = 8, 12, 0.125
    with context(n, dtype, 1 << 20):
        count = 65536
        x = inputs.normal(n, count, dtype, seed=5, scale=0.02)
        got = allreduce_iters(x, dtype, proto, iters, chain_scale=scale)
        xb = inputs.bits_of(x)
        ok, err, rel = orc.compare_atomic(got[0], orc.allreduce(xb, dtype), xb, dtype)
        assert ok, (err, rel)
        want = orc.allreduce_iters(xb, iters, dtype, chain_scale=scale)
        from oracle import fpformats as fp
        for e in range(iters):
            assert all(np.array_equal(got[e][0], got[e][q]) for q in range(n)), e
            assert np.array_equal(np.isfinite(fp.decode(got[e], dtype)), np.isfinite(fp.decode(want[e], dtype))), e


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("n", [5, 6, 7, 8])
def test_two_shot_tma_path_at_small_sizes(n, dtype):
    # 6-8 ranks stream the two-shot through shared memory with TMA bulk copies
    # from 32 KiB per rank, 5 ranks from 512 KiB: ragged and tile-crossing sizes
    e = inputs.ELEM_BYTES[dtype]
    with context(n, dtype, 2 << 20):
        for nbytes in (32 << 10, (48 << 10) + 6, 64 << 10, (200 << 10) + 2, 512 << 10, (1 << 20) + 14):
            count = nbytes // e
            x = inputs.normal(n, count, dtype, seed=count + n)
            got = allreduce(x, dtype, "fixed_twoshot")
            assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), dtype)), count
            got_auto = allreduce(x, dtype, "auto")
            assert np.array_equal(got_auto, orc.allreduce(inputs.bits_of(x), dtype)), count


@pytest.mark.parametrize("n,kib,chain", [(8, 64, True), (8, 1024, True), (4, 1024, True),
                                         (8, 64, False), (8, 256, False), (2, 16, True)])
def test_persistent_auto_follows_its_rule(n, kib, chain):
    # llar_allreduce_iters with AUTO takes llar_select_protocol_iters' choice
    # (LL for chains up to the LL capacity, the two-shot for 7-8 ranks above
    # 512 KiB; LL up to 64 KiB back to back with 6-8 ranks); bits as the oracle
    dtype, iters = "bf16", 6
    count = kib * 512
    with context(n, dtype, 1 << 20):
        if chain:
            x = inputs.normal(n, count, dtype, seed=kib + n, scale=0.02)
            got = allreduce_iters(x, dtype, "auto", iters, chain_scale=1.0 / n)
            want = orc.allreduce_iters(inputs.bits_of(x), iters, dtype, chain_scale=1.0 / n)
        else:
            x = inputs.uniform(n, count, dtype, seed=kib + n, iters=iters)
            got = allreduce_iters(x, dtype, "auto", iters)
            want = orc.allreduce_iters(inputs.bits_of(x), iters, dtype)
        assert llar.llar_last_launch()[0] == llar.llar_select_protocol_iters(n, dtype, count, iters, chain)
        assert np.array_equal(got, want)


def test_nondeterministic_auto_takes_ll128_direct_in_long_chains():
    # after llar_set_auto_nondeterministic(1), AUTO runs an 8-rank chain of
    # 256 KiB per rank with the LL128 direct form; integers in [-2, 2] with
    # scale 1/N keep every partial sum exact, so the chain is the oracle's
    n, dtype, iters = 8, "bf16", 6
    count = 256 * 512
    x = inputs.integers(n, count, dtype, seed=9, lo=-2, hi=2)
    want = orc.allreduce_iters(inputs.bits_of(x), iters, dtype, chain_scale=1.0 / n)
    with context(n, dtype, 1 << 20):
        got = allreduce_iters(x, dtype, "auto", iters, chain_scale=1.0 / n)
        assert llar.llar_last_launch()[0] == "ll"  # deterministic by default
        assert np.array_equal(got, want)
        llar.llar_set_auto_nondeterministic(True)
        got = allreduce_iters(x, dtype, "auto", iters, chain_scale=1.0 / n)
        assert llar.llar_last_launch()[0] == "ll128_direct"
        assert np.array_equal(got, want)
    with context(n, dtype, 1 << 20):  # a new context starts deterministic again
        allreduce_iters(x, dtype, "auto", iters, chain_scale=1.0 / n)
        assert llar.llar_last_launch()[0] == "ll"
