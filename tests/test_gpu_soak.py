"""Long-lived contexts: one context serves a seeded random sequence of calls
(AllReduce single and persistent, pipelined and chained, ReduceScatter,
AllGather, point to point) with random protocols, sizes and sentinel
chunks, so that each call starts from whatever staging state, epoch, slot
parity, ring position and LL128 line slot the previous calls left. Every
result is checked against the oracle (bit-exact on the fixed-order paths,
within the atomic tolerance for LL128)."""

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from oracle import p2p
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import FILL, context, device_inputs, filled_outputs

pytestmark = pytest.mark.gpu

AR_PROTOS = ["auto", "ll", "sentinel", "ll128", "ll128_direct", "fixed_oneshot", "fixed_twoshot"]
SEG_PROTOS = {"rs": ["auto", "ll", "sentinel", "ll128", "fixed_oneshot"],
              "ag": ["auto", "ll", "sentinel", "fixed_oneshot"]}
MAX_BYTES = 512 << 10


def _count(rng, e):
    kind = int(rng.integers(0, 5))
    if kind == 0:
        return int(rng.integers(0, 4))
    if kind == 1:
        return int(rng.integers(4, 600))
    if kind == 2:
        return int(rng.integers(600, 20000))
    return int(rng.integers(20000, MAX_BYTES // e + 1))


def _check_ar(got, xb, dtype, proto):
    want = orc.allreduce(xb, dtype)
    if proto.startswith("ll128"):
        assert orc.compare_atomic(got, want, xb, dtype)[0]
    else:
        assert np.array_equal(got, want)


def _allreduce(rng, n, dtype, e, count, proto):
    x = inputs.normal(n, max(count, 1), dtype, seed=int(rng.integers(1 << 30)), exclude_sentinel=True)[:, :count]
    ins = device_inputs(x.contiguous()) if count else [torch.zeros(8, device="cuda") for _ in range(n)]
    outs = filled_outputs(n, max(count, 1), dtype)
    llar.llar_allreduce(ins, outs, count, proto)
    torch.cuda.synchronize()
    if count:
        _check_ar(np.stack([inputs.bits_of(o)[:count] for o in outs]), inputs.bits_of(x), dtype, proto)


def _iters(rng, n, dtype, e, count, proto, chain):
    if count == 0:
        return
    iters = int(rng.integers(2, 7))
    stride = -(-count * e // 16) * 16 // e
    xi = inputs.normal(n, count, dtype, seed=int(rng.integers(1 << 30)), iters=iters, exclude_sentinel=True,
                       scale=0.02)
    if chain:
        ins, in_stride = device_inputs(xi[0].contiguous()), 0
    else:
        ins = []
        for r in range(n):
            buf = torch.zeros(iters * stride, dtype=inputs.TORCH_DTYPE[dtype], device="cuda")
            buf.view(iters, stride)[:, :count] = xi[:, r, :].cuda()
            ins.append(buf)
        in_stride = stride
    outs = filled_outputs(n, iters * stride, dtype)
    scale = 0.5 if chain else 0.0
    llar.llar_allreduce_iters(ins, outs, count, proto, iters, in_stride, stride, scale)
    torch.cuda.synchronize()
    got = np.stack([inputs.bits_of(o).reshape(iters, stride)[:, :count] for o in outs], axis=1)
    xb = inputs.bits_of(xi)
    used = llar.llar_last_launch()[0]
    if chain:
        if used.startswith("ll128"):
            _check_ar(got[0], xb[0], dtype, used)
            for it in range(iters):
                assert all(np.array_equal(got[it][0], got[it][q]) for q in range(n))
        else:
            assert np.array_equal(got, orc.allreduce_iters(xb[0], iters, dtype, chain_scale=scale))
    else:
        for it in range(iters):
            _check_ar(got[it], xb[it], dtype, used)


def _segments(rng, n, dtype, e, count, proto, rs):
    if count == 0:
        return
    x = inputs.normal(n, count, dtype, seed=int(rng.integers(1 << 30)), exclude_sentinel=True)
    seg = -(-count // n)
    bounds = [orc.shard_bounds(count, n, s) for s in range(n)]
    if rs:
        ins = device_inputs(x.contiguous())
        outs = filled_outputs(n, seg, dtype)
        llar.llar_reduce_scatter(ins, outs, count, proto)
        torch.cuda.synchronize()
        want = orc.reduce_scatter(inputs.bits_of(x), dtype)
        for s, (lo, hi) in enumerate(bounds):
            got = inputs.bits_of(outs[s])[: hi - lo]
            if llar.llar_last_launch()[0] == "ll128":
                full = inputs.bits_of(x)[:, lo:hi]
                assert orc.compare_atomic(got[None], want[s][None], full, dtype)[0]
            else:
                assert np.array_equal(got, want[s]), s
    else:
        full = x[0]
        ins = []
        for lo, hi in bounds:
            t = torch.empty(max(hi - lo, 1), dtype=full.dtype, device="cuda")
            t[: hi - lo] = full[lo:hi].cuda()
            ins.append(t)
        outs = filled_outputs(n, count, dtype)
        llar.llar_all_gather(ins, outs, count, proto)
        torch.cuda.synchronize()
        want = orc.all_gather([inputs.bits_of(full[lo:hi]) for lo, hi in bounds], count)
        assert np.array_equal(np.stack([inputs.bits_of(o) for o in outs]), want)


def _p2p(rng, n, dtype, e, count, proto):
    if count == 0:
        return
    dst = [int(v) for v in rng.permutation(n)]
    dst = [d if d != r else -1 for r, d in enumerate(dst)]
    x = inputs.normal(n, count, dtype, seed=int(rng.integers(1 << 30)), exclude_sentinel=True)
    sends = device_inputs(x.contiguous())
    recvs = filled_outputs(n, count, dtype)
    llar.llar_sendrecv(sends, recvs, dst, count, proto)
    torch.cuda.synchronize()
    fill = np.full((n, count), FILL[dtype], dtype=inputs.bits_of(x).dtype)
    assert np.array_equal(np.stack([inputs.bits_of(o) for o in recvs]), p2p.sendrecv(inputs.bits_of(x), dst, fill))


@pytest.mark.parametrize("n,dtype,seed", [(8, "bf16", 1), (5, "fp16", 2), (3, "fp32", 3), (8, "fp32", 4)])
def test_one_context_serves_a_random_sequence(n, dtype, seed):
    e = inputs.ELEM_BYTES[dtype]
    rng = np.random.default_rng(seed)
    with context(n, dtype, MAX_BYTES):
        for step in range(90):
            if rng.random() < 0.1:
                llar.llar_set_sentinel_chunk(16 * int(rng.integers(1, 4097)))
            count = _count(rng, e)
            op = int(rng.integers(0, 6))
            if op in (3, 4):
                rs = op == 3
                proto = SEG_PROTOS["rs" if rs else "ag"][int(rng.integers(0, len(SEG_PROTOS["rs" if rs else "ag"])))]
            elif op == 5:
                proto = ["auto", "ll", "sentinel", "fixed_oneshot"][int(rng.integers(0, 4))]
            else:
                proto = AR_PROTOS[int(rng.integers(0, len(AR_PROTOS)))]
            try:
                if op == 0:
                    _allreduce(rng, n, dtype, e, count, proto)
                elif op in (1, 2):
                    _iters(rng, n, dtype, e, count, proto, chain=op == 2)
                elif op in (3, 4):
                    _segments(rng, n, dtype, e, count, proto, rs=op == 3)
                else:
                    _p2p(rng, n, dtype, e, count, proto)
            except llar.LlarError as ex:
                # sentinel segments and transfers must fit the chunk set above
                assert ex.code == llar.ERR_TOO_LARGE and proto == "sentinel", (step, op, proto, count, ex.code)
            assert llar.llar_get_status()[0] == llar.OK, (step, op, proto, count)
