"""LLAR_COOP=0: the kernels whose CTAs wait on each other launch without
the cooperative attribute (the grid still sized to fit the GPU at once).
Same results as the cooperative launches: every protocol, single calls,
back-to-back and chained persistent launches, ReduceScatter / AllGather
and point to point, against the oracle; the context's status stays OK.
Nothing else runs on the GPU meanwhile, which is the knob's condition."""

import os

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from oracle import p2p
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import FILL, allreduce, allreduce_iters, context, device_inputs, filled_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture
def no_coop():
    saved = os.environ.get("LLAR_COOP")
    os.environ["LLAR_COOP"] = "0"
    try:
        yield
    finally:
        if saved is None:
            os.environ.pop("LLAR_COOP", None)
        else:
            os.environ["LLAR_COOP"] = saved


def _ok(got, x, dtype, proto):
    want = orc.allreduce(inputs.bits_of(x), dtype)
    if proto.startswith("ll128"):
        return orc.compare_atomic(got, want, inputs.bits_of(x), dtype)[0]
    return np.array_equal(got, want)


@pytest.mark.parametrize("proto", ["ll", "sentinel", "ll128", "ll128_direct", "fixed_oneshot", "fixed_twoshot"])
@pytest.mark.parametrize("n,dtype", [(8, "bf16"), (4, "fp32"), (3, "fp16")])
def test_allreduce_without_cooperative_launch(no_coop, proto, n, dtype):
    with context(n, dtype, 1 << 20):
        for count in (5, 8192, 65539):
            x = inputs.normal(n, count, dtype, seed=count + n, scale=0.02, exclude_sentinel=True)
            assert _ok(allreduce(x, dtype, proto), x, dtype, proto), (proto, count)
        assert llar.llar_get_status()[0] == llar.OK


@pytest.mark.parametrize("proto", ["ll", "sentinel", "ll128", "fixed_twoshot"])
def test_persistent_launches_without_cooperative_launch(no_coop, proto):
    n, dtype, count, iters = 8, "bf16", 8192, 50
    with context(n, dtype, 1 << 20):
        x = inputs.normal(n, count, dtype, seed=7, scale=0.02, iters=iters, exclude_sentinel=True)
        got = allreduce_iters(x, dtype, proto, iters)
        for it in range(iters):
            assert _ok(got[it], x[it], dtype, proto), it
        xc = inputs.normal(n, count, dtype, seed=8, scale=0.02, exclude_sentinel=True)
        got = allreduce_iters(xc, dtype, proto, iters, chain_scale=0.125)
        if proto.startswith("ll128"):
            assert _ok(got[0], xc, dtype, proto)
        else:
            assert np.array_equal(got, orc.allreduce_iters(inputs.bits_of(xc), iters, dtype, chain_scale=0.125))
        assert llar.llar_get_status()[0] == llar.OK


def test_segments_and_p2p_without_cooperative_launch(no_coop):
    n, dtype = 8, "bf16"
    with context(n, dtype, 1 << 20):
        for count in (1000, 65536):
            x = inputs.normal(n, count, dtype, seed=count, scale=0.02, exclude_sentinel=True)
            seg = -(-count // n)
            for proto in ("ll", "sentinel", "ll128", "fixed_oneshot"):
                mid = filled_outputs(n, seg, dtype)
                llar.llar_reduce_scatter(device_inputs(x), mid, count, proto)
                outs = filled_outputs(n, count, dtype)
                llar.llar_all_gather(mid, outs, count, "ll" if proto == "ll128" else proto)
                torch.cuda.synchronize()
                got = np.stack([inputs.bits_of(o) for o in outs])
                assert _ok(got, x, dtype, proto), (proto, count)
            dst = [(r + 1) % n for r in range(n)]
            for proto in ("ll", "sentinel", "fixed_oneshot"):
                recvs = filled_outputs(n, count, dtype)
                llar.llar_sendrecv(device_inputs(x), recvs, dst, count, proto)
                torch.cuda.synchronize()
                fill = np.full((n, count), FILL[dtype], dtype=inputs.bits_of(x).dtype)
                want = p2p.sendrecv(inputs.bits_of(x), dst, fill)
                assert np.array_equal(np.stack([inputs.bits_of(o) for o in recvs]), want), (proto, count)
        assert llar.llar_get_status()[0] == llar.OK
