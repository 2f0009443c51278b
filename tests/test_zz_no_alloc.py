"""The allocation-free entry point, llar_allreduce_noalloc.

It serves callers that cannot allocate device memory when they need the
AllReduce (all device memory owned by a caching allocator or a fixed
budget, or a path that must not take cudaMalloc's implicit device
synchronisation): its LL staging is a fixed array inside the library.
Its output must equal the CPU oracle's and the regular entry point's on
the same inputs, on two calls in a row (the second call reuses the array
the first one left behind). A wait that runs out must be reported exactly
once. This file sorts last so a run that stops at the first failure has
run every other test already.
"""

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import context, device_inputs, filled_outputs


def test_noalloc_rejects_oversized_messages_before_any_device_work():
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_allreduce_noalloc([0] * 8, [0] * 8, (32 << 10) // 2 + 1, 8, "bf16", stream=0)
    assert ei.value.code == llar.ERR_TOO_LARGE


def _noalloc(x, n, dtype):
    count = x.shape[1]
    ins = device_inputs(x)
    outs = filled_outputs(n, count, dtype)
    llar.llar_allreduce_noalloc(ins, outs, count, n, dtype)
    torch.cuda.synchronize()
    return np.stack([inputs.bits_of(o) for o in outs])


@pytest.mark.gpu
@pytest.mark.parametrize("n,dtype,count", [(8, "bf16", 8192), (4, "fp32", 8192 - 3), (2, "fp16", 16384),
                                           (8, "bf16", 16384), (3, "fp16", 1)])
def test_noalloc_matches_oracle_and_regular_entry_point_twice(n, dtype, count):
    xs = [inputs.normal(n, count, dtype, seed=100 + k, scale=0.02) for k in range(2)]
    # outputs of the regular entry point (same LL protocol)
    refs = []
    with context(n, dtype, 1 << 20):
        for x in xs:
            ins = device_inputs(x)
            outs = filled_outputs(n, count, dtype)
            llar.llar_allreduce(ins, outs, count, "ll")
            torch.cuda.synchronize()
            refs.append(np.stack([inputs.bits_of(o) for o in outs]))
    # two calls in a row through the allocation-free entry point; LL is
    # fixed-order, so the tolerance is bit-exact
    for x, ref in zip(xs, refs):
        got = _noalloc(x, n, dtype)
        assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), dtype))
        assert np.array_equal(got, ref)
        assert all(np.array_equal(got[0], got[r]) for r in range(1, n))


@pytest.mark.gpu
def test_noalloc_reports_a_timeout_exactly_once():
    # rank 1 never sends: the other ranks' waits run out (20 ms bound, no GPU
    # fault). The call queued behind it while the stream is busy gives up at
    # once; the first call on the idle stream reports the timeout; the next
    # one works again.
    n, dtype, count = 4, "bf16", 4096
    x = inputs.normal(n, count, dtype, seed=7, scale=0.02)
    want = orc.allreduce(inputs.bits_of(x), dtype)
    ins = device_inputs(x)
    outs = filled_outputs(n, count, dtype)
    torch.cuda.synchronize()
    try:
        llar.llar_set_timeout_ns(20_000_000)
        llar.llar_debug_inject(1, "skip")
        llar.llar_allreduce_noalloc(ins, outs, count, n, dtype)  # launches; its waits run out
        llar.llar_debug_inject(-1, "none")
        llar.llar_allreduce_noalloc(ins, outs, count, n, dtype)  # stream busy: no check, invalid output
        torch.cuda.synchronize()
        with pytest.raises(llar.LlarError) as ei:
            llar.llar_allreduce_noalloc(ins, outs, count, n, dtype)
        assert ei.value.code == llar.ERR_TIMEOUT
        torch.cuda.synchronize()
        outs2 = filled_outputs(n, count, dtype)
        llar.llar_allreduce_noalloc(ins, outs2, count, n, dtype)  # reported once: works again
        torch.cuda.synchronize()
        got = np.stack([inputs.bits_of(o) for o in outs2])
        assert np.array_equal(got, want)
    finally:
        llar.llar_debug_inject(-1, "none")
        llar.llar_set_timeout_ns(1_000_000_000)
