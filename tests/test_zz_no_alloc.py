"""The allocation-free entry point, llar_allreduce_noalloc.

It serves callers that cannot allocate device memory when they need the
AllReduce (all device memory owned by a caching allocator or a fixed
budget, or a path that must not take cudaMalloc's implicit device
synchronisation): its LL staging is a fixed array inside the library.
Its output must equal the regular entry point's on the same inputs, on two
calls in a row (the second call reuses the array the first one left
behind). This file sorts last so a run that stops at the first failure has
run every other test already.
"""

import numpy as np
import pytest
import torch

from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import context, device_inputs, filled_outputs


def test_noalloc_rejects_oversized_messages_before_any_device_work():
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_allreduce_noalloc([0] * 8, [0] * 8, (32 << 10) // 2 + 1, 8, "bf16", stream=0)
    assert ei.value.code == llar.ERR_TOO_LARGE


@pytest.mark.gpu
@pytest.mark.parametrize("n,dtype,count", [(8, "bf16", 8192), (4, "fp32", 8192 - 3), (2, "fp16", 16384)])
def test_noalloc_matches_regular_entry_point_twice(n, dtype, count):
    xs = [inputs.normal(n, count, dtype, seed=100 + k, scale=0.02) for k in range(2)]
    # reference outputs from the regular entry point (same LL protocol)
    refs = []
    with context(n, dtype, 1 << 20):
        for x in xs:
            ins = device_inputs(x)
            outs = filled_outputs(n, count, dtype)
            llar.llar_allreduce(ins, outs, count, "ll")
            torch.cuda.synchronize()
            refs.append(np.stack([inputs.bits_of(o) for o in outs]))
    # two calls in a row through the allocation-free entry point
    for x, ref in zip(xs, refs):
        ins = device_inputs(x)
        outs = filled_outputs(n, count, dtype)
        llar.llar_allreduce_noalloc(ins, outs, count, n, dtype)
        torch.cuda.synchronize()
        got = np.stack([inputs.bits_of(o) for o in outs])
        assert np.array_equal(got, ref)  # LL is fixed-order: bit-exact, the tests' tolerance
