"""Shared helpers of the GPU tests: a context guard and a call wrapper.

Inputs come from `tp_allreduce_persistent_b300.inputs`; expected values
from `oracle/`; the AllReduce itself only from the C-ABI library.
"""

import contextlib

import numpy as np
import torch

from tp_allreduce_persistent_b300 import inputs, llar

FILL = {"fp32": 0x5A5A5A5A, "fp16": 0x5A5A, "bf16": 0x5A5A}  # marks unwritten outputs


@contextlib.contextmanager
def context(nranks, dtype, max_bytes, timeout_ns=2_000_000_000):
    llar.llar_init(nranks, dtype, max_bytes)
    llar.llar_set_timeout_ns(timeout_ns)
    llar.llar_set_launch(0, 0)
    try:
        yield
    finally:
        llar.llar_debug_inject(-1, "none")
        llar.llar_set_launch(0, 0)
        llar.llar_destroy()


def device_inputs(x_cpu):
    """One separate device allocation per rank (as separate ranks would have)."""
    return [x_cpu[r].contiguous().cuda() for r in range(x_cpu.shape[0])]


def filled_outputs(n, numel, dtype):
    outs = []
    for _ in range(n):
        t = torch.empty(numel, dtype=inputs.TORCH_DTYPE[dtype], device="cuda")
        if dtype == "fp32":
            t.view(torch.int32).fill_(FILL[dtype])
        else:
            t.view(torch.int16).fill_(FILL[dtype])
        outs.append(t)
    return outs


def check_status():
    code, rank, cta, epoch = llar.llar_get_status()
    assert code == llar.OK, f"device status {code} at rank {rank} cta {cta} epoch {epoch}"


def allreduce(x_cpu, dtype, protocol):
    """Run one AllReduce of [N, count] CPU input; return [N, count] output bits."""
    n, count = x_cpu.shape
    ins = device_inputs(x_cpu)
    outs = filled_outputs(n, count, dtype)
    llar.llar_allreduce(ins, outs, count, protocol)
    torch.cuda.synchronize()
    check_status()
    return np.stack([inputs.bits_of(o) for o in outs])


def allreduce_iters(x_cpu, dtype, protocol, iters, chain_scale=0.0):
    """Run `iters` AllReduces in one launch.

    Without a chain x_cpu is [iters, N, count] (fresh input per iteration);
    with a chain it is [N, count]. Returns [iters, N, count] output bits.
    """
    if chain_scale:
        n, count = x_cpu.shape
    else:
        _, n, count = x_cpu.shape
    e = inputs.ELEM_BYTES[dtype]
    stride = -(-count * e // 16) * 16 // e  # iteration stride, whole 16-byte units
    if chain_scale:
        ins = device_inputs(x_cpu)
        in_stride = 0
    else:
        ins = []
        for r in range(n):
            buf = torch.zeros(iters * stride, dtype=inputs.TORCH_DTYPE[dtype], device="cuda")
            buf.view(iters, stride)[:, :count] = x_cpu[:, r, :].cuda()
            ins.append(buf)
        in_stride = stride
    outs = filled_outputs(n, iters * stride, dtype)
    llar.llar_allreduce_iters(ins, outs, count, protocol, iters, in_stride, stride, chain_scale)
    torch.cuda.synchronize()
    check_status()
    res = np.stack([inputs.bits_of(o).reshape(iters, stride)[:, :count] for o in outs], axis=1)
    return res
