"""ReduceScatter and AllGather through the C ABI against the oracle.

Both are fixed-order (rank-order float32 sums, one rounding; copies are
copies), so results must match bit for bit, including ragged and empty
segments. AllGather(ReduceScatter(x)) must equal AllReduce(x).
"""

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import context, device_inputs, filled_outputs

pytestmark = pytest.mark.gpu

COUNTS = [1, 5, 8, 31, 100, 1000, 4097, 65539]


def _seg_len(count, n):
    return -(-count // n) if count else 0


@pytest.mark.parametrize("proto", ["ll", "fixed_oneshot"])
@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_reduce_scatter(proto, dtype, n):
    with context(n, dtype, 1 << 20):
        for count in COUNTS:
            x = inputs.normal(n, count, dtype, seed=count + n)
            ins = device_inputs(x)
            seg = _seg_len(count, n)
            outs = filled_outputs(n, max(seg, 1), dtype)
            llar.llar_reduce_scatter(ins, outs, count, proto)
            torch.cuda.synchronize()
            assert llar.llar_get_status()[0] == llar.OK
            want = orc.reduce_scatter(inputs.bits_of(x), dtype)
            for s in range(n):
                got = inputs.bits_of(outs[s])[: len(want[s])]
                assert np.array_equal(got, want[s]), (count, s)


@pytest.mark.parametrize("proto", ["ll", "fixed_oneshot"])
@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_all_gather(proto, dtype, n):
    with context(n, dtype, 1 << 20):
        for count in COUNTS:
            full = inputs.normal(1, count, dtype, seed=count * 3 + n)[0]
            segs = [full[lo:hi] for lo, hi in (orc.shard_bounds(count, n, s) for s in range(n))]
            ins = []
            for sg in segs:
                t = torch.empty(max(len(sg), 1), dtype=sg.dtype, device="cuda")
                t[: len(sg)] = sg.cuda()
                ins.append(t)
            outs = filled_outputs(n, count, dtype)
            llar.llar_all_gather(ins, outs, count, proto)
            torch.cuda.synchronize()
            assert llar.llar_get_status()[0] == llar.OK
            want = orc.all_gather([inputs.bits_of(sg) for sg in segs], count)
            got = np.stack([inputs.bits_of(o) for o in outs])
            assert np.array_equal(got, want), count


@pytest.mark.parametrize("proto", ["ll", "fixed_oneshot"])
def test_all_gather_of_reduce_scatter_is_allreduce(proto):
    n, dtype = 8, "bf16"
    with context(n, dtype, 1 << 20):
        for count in (8192, 8195):
            x = inputs.normal(n, count, dtype, seed=count, scale=0.02)
            ins = device_inputs(x)
            seg = _seg_len(count, n)
            mid = filled_outputs(n, seg, dtype)
            outs = filled_outputs(n, count, dtype)
            llar.llar_reduce_scatter(ins, mid, count, proto)
            llar.llar_all_gather(mid, outs, count, proto)
            torch.cuda.synchronize()
            got = np.stack([inputs.bits_of(o) for o in outs])
            assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), dtype))


def test_segment_collectives_reject_other_protocols():
    with context(4, "fp32", 1 << 12):
        ins = device_inputs(inputs.normal(4, 64, "fp32", seed=1))
        outs = filled_outputs(4, 64, "fp32")
        for proto in ("sentinel", "ll128", "fixed_twoshot"):
            with pytest.raises(llar.LlarError) as ei:
                llar.llar_reduce_scatter(ins, outs, 64, proto)
            assert ei.value.code == llar.ERR_UNSUPPORTED
