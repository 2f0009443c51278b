"""AllReduce launches captured in a CUDA graph and replayed.

Epochs are kept on the device, so every replay of a captured launch uses
fresh epochs: replays with new inputs must give exact new results (a
replay that reused the captured epochs would accept the previous replay's
LL lines). Decode loops are commonly captured this way.
"""

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import context, filled_outputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("proto", ["ll", "sentinel", "ll128", "ll128_direct", "fixed_oneshot", "fixed_twoshot"])
def test_graph_replays_with_fresh_inputs(proto):
    n, dtype, count, calls = 8, "bf16", 8192, 6
    with context(n, dtype, 1 << 20):
        ins = [torch.zeros(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        outs = [filled_outputs(n, count, dtype) for _ in range(calls)]
        # warm up outside the capture (first calls resolve launch shapes)
        llar.llar_allreduce(ins, outs[0], count, proto)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for k in range(calls):
                llar.llar_allreduce(ins, outs[k], count, proto)
        for rep in range(3):
            x = inputs.normal(n, count, dtype, seed=50 + rep, scale=0.02)
            for r in range(n):
                ins[r].copy_(x[r])
            g.replay()
            torch.cuda.synchronize()
            assert llar.llar_get_status()[0] == llar.OK
            xb = inputs.bits_of(x)
            want = orc.allreduce(xb, dtype)
            for k in range(calls):
                got = np.stack([inputs.bits_of(o) for o in outs[k]])
                if proto.startswith("ll128"):
                    assert orc.compare_atomic(got, want, xb, dtype)[0], (rep, k)
                else:
                    assert np.array_equal(got, want), (rep, k)


def test_epoch_advances_on_every_replay():
    n, count = 4, 1024
    with context(n, "fp32", 1 << 16):
        ins = [torch.ones(count, device="cuda") for _ in range(n)]
        outs = [torch.empty(count, device="cuda") for _ in range(n)]
        llar.llar_allreduce(ins, outs, count, "ll")
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            llar.llar_allreduce_iters(ins, outs, count, "ll", 7, 0, 0, 0.0)
        e0 = llar.llar_epoch()
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        assert llar.llar_epoch() == e0 + 14
        assert all(torch.all(o == n) for o in outs)
