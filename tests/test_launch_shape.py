"""The runtime's launch-shape rule, on the CPU (llar_debug_launch_shape).

The rule picks CTAs per rank and threads per CTA from the rank count, the
message size, the element type, the protocol and the SM count; a launch
then clamps the CTAs to what the GPU can hold resident. These tests pin
the shapes the measurements were taken with (the bench's launches and the
per-configuration rows) and the properties every shape must have: all of
a CTA's work items covered by its threads in one pass where one CTA per
SM of 512 threads can hold them, thread counts that are whole warps, and
no more CTAs per rank than the chain flags address.
"""

import math
import random

import pytest

from tp_allreduce_persistent_b300 import llar

SMS = 148  # B300


def shape(n, dtype, count, proto, chained=False, chunk=64 << 10):
    return llar.llar_debug_launch_shape(n, dtype, count, proto, chained, SMS, chunk)


def ll128_lines(n, dtype, count):
    payload = 128 // (4 if dtype == "fp32" else 2) - 1
    return math.ceil(math.ceil(count / n) / payload)


def test_shapes_the_measurements_ran_with():
    assert shape(8, "bf16", 8192, "ll") == (16, 128)  # headline LL, 8 x 16 KiB
    assert shape(8, "fp16", 32768, "sentinel", chunk=8192) == (16, 32)  # C4
    assert shape(4, "bf16", 8192, "sentinel", chunk=16384) == (16, 64)  # C2
    assert shape(8, "bf16", 16 * 512, "ll128") == (9, 128)  # C3 16 KiB
    assert shape(8, "bf16", 64 * 512, "ll128") == (18, 256)  # C3 64 KiB
    assert shape(8, "bf16", 65536, "ll128", chained=True) == (18, 512)  # 8-rank LL128 chain
    assert shape(4, "bf16", 65536, "ll128", chained=True) == (37, 256)


def test_ll128_threads_cover_whole_lines_in_one_pass():
    # a CTA takes ceil(L / G) lines of each of the N segments, 8 lanes each
    rng = random.Random(5)
    cases = [(8, "bf16", 65536), (3, "bf16", 40000), (4, "fp32", 12345), (7, "fp16", 999)]
    cases += [(rng.randint(2, 8), rng.choice(["fp32", "fp16", "bf16"]), rng.randint(1, 1 << 20)) for _ in range(300)]
    for n, dtype, count in cases:
        for chained in (False, True):
            g, t = shape(n, dtype, count, "ll128", chained)
            lines = ll128_lines(n, dtype, count)
            items = math.ceil(lines / g) * n * 8
            wide = lines * n * 8 > max(1, SMS // n) * 512
            assert t % 32 == 0 and 1 <= g <= 1024, (n, dtype, count, g, t)
            if wide:
                assert t == 256, (n, dtype, count, g, t)
            else:
                assert t >= min(items, 512), (n, dtype, count, g, t, items)


def test_ll_and_sentinel_shapes_cover_the_message():
    rng = random.Random(6)
    for _ in range(300):
        n = rng.randint(2, 8)
        dtype = rng.choice(["fp32", "fp16", "bf16"])
        e = 4 if dtype == "fp32" else 2
        count = rng.randint(1, 1 << 18)
        one_per_sm = max(1, SMS // n)
        g, t = shape(n, dtype, count, "ll")
        words = math.ceil(count * e / 8)
        assert t % 32 == 0 and g * t >= min(words, one_per_sm * 512), (n, dtype, count, g, t)
        chunk = rng.choice([16, 1024, 8192, 16384, 65536])
        g, t = shape(n, dtype, count, "sentinel", chunk=chunk)
        vecs = min(chunk, math.ceil(count * e / 16) * 16) // 16
        assert t % 32 == 0 and g >= min(16, max(1, 2 * SMS // n)), (n, dtype, count, chunk, g, t)
        assert g * t >= min(vecs, g * 512), (n, dtype, count, chunk, g, t)


def test_forced_shape_is_reported_and_arguments_are_checked():
    llar.llar_set_launch(5, 96)
    try:
        assert shape(8, "bf16", 8192, "ll") == (5, 96)
    finally:
        llar.llar_set_launch(0, 0)
    assert shape(8, "bf16", 8192, "ll") == (16, 128)
    for bad in [(1, "bf16", 8, "ll"), (9, "bf16", 8, "ll"), (8, "bf16", 0, "ll"), (8, "bf16", 8, "auto")]:
        with pytest.raises(llar.LlarError) as ei:
            shape(*bad)
        assert ei.value.code == llar.ERR_INVALID
    with pytest.raises(llar.LlarError):
        llar.llar_debug_launch_shape(8, "bf16", 8, "sentinel", False, SMS, 24)  # chunk not a multiple of 16


def test_ll128_direct_takes_the_ll128_shapes():
    # the direct-AllGather variant runs the same (segment, line, lane) items
    rng = random.Random(5)
    for _ in range(200):
        n = rng.randint(2, 8)
        dtype = rng.choice(["fp32", "fp16", "bf16"])
        count = rng.choice([1, 63, 500, rng.randint(1, 1 << 20)])
        chained = rng.random() < 0.3
        assert shape(n, dtype, count, "ll128_direct", chained) == shape(n, dtype, count, "ll128", chained)


def test_single_calls_of_the_fixed_paths_take_one_vector_a_thread():
    # one AllReduce per launch: CTAs of 128 threads, one 16-byte vector a
    # thread, while the one-shot's N reads (or a two-shot segment) stay small
    for n, count, proto in ((4, 32768, "fixed_oneshot"), (8, 8192, "fixed_oneshot"),
                            (4, 131072, "fixed_twoshot"), (2, 8192, "fixed_twoshot")):
        vecs = count * 2 // 16
        per_rank = vecs if proto == "fixed_oneshot" else -(-vecs // n)
        g, t = shape(n, "bf16", count, proto, 2)
        assert t == 128 and g == min(-(-per_rank // 128), SMS * 8 // n), (n, count, proto, g, t)
        assert shape(n, "bf16", count, proto, 0)[1] == 256  # a persistent loop keeps 256-thread CTAs
    # large one-shot messages keep the loop's shape
    assert shape(8, "bf16", 131072, "fixed_oneshot", 2) == shape(8, "bf16", 131072, "fixed_oneshot", 0)
    # the other protocols do not depend on it
    for proto in ("ll", "sentinel", "ll128", "ll128_direct"):
        assert shape(8, "bf16", 8192, proto, 2) == shape(8, "bf16", 8192, proto, 0)
