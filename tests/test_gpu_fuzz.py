"""Seeded random parity sweep across the entry points: random rank count,
element type, size (empty, one element, ragged, chunk- and tile-crossing),
protocol, iteration count, strides and chains, each checked against the
oracle (bit-exact for fixed-order paths, within the atomic tolerance for
LL128). The cases are drawn once from a fixed seed, so a failure names a
reproducible case."""

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from oracle import p2p
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import FILL, context, device_inputs, filled_outputs

pytestmark = pytest.mark.gpu

PROTOS = ["auto", "ll", "sentinel", "ll128", "ll128_direct", "fixed_oneshot", "fixed_twoshot"]


def draw_cases(seed, k):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(k):
        n = int(rng.integers(2, 9))
        dtype = ["fp32", "fp16", "bf16"][int(rng.integers(0, 3))]
        kind = int(rng.integers(0, 4))
        count = [0, 1, int(rng.integers(2, 64)), int(rng.integers(64, 5000)),
                 int(rng.integers(5000, 140000))][int(rng.integers(0, 5))]
        cases.append((n, dtype, count, PROTOS[int(rng.integers(0, len(PROTOS)))], kind, int(rng.integers(0, 1 << 30))))
    return cases


def check(got, xb, dtype, proto):
    want = orc.allreduce(xb, dtype)
    if proto.startswith("ll128"):
        ok, err, rel = orc.compare_atomic(got, want, xb, dtype)
        assert ok, (err, rel)
    else:
        assert np.array_equal(got, want)


@pytest.mark.parametrize("case", draw_cases(2026, 60) + draw_cases(99, 60))
def test_random_allreduce(case):
    n, dtype, count, proto, kind, seed = case
    e = inputs.ELEM_BYTES[dtype]
    rng = np.random.default_rng(seed)
    with context(n, dtype, max(count * e, 16) * 2 + 4096):
        # a random sentinel chunk, and now and then a forced launch shape
        llar.llar_set_sentinel_chunk(16 * int(rng.integers(1, 4097)))
        if rng.random() < 0.3:
            llar.llar_set_launch(int(rng.integers(1, 33)), 32 * int(rng.integers(1, 17)))
        x = inputs.normal(n, max(count, 1), dtype, seed=seed, exclude_sentinel=True)[:, :count]
        if kind == 0:  # one call
            ins = device_inputs(x.contiguous()) if count else [torch.zeros(8, device="cuda") for _ in range(n)]
            outs = filled_outputs(n, max(count, 1), dtype)
            try:
                llar.llar_allreduce(ins, outs, count, proto)
            except llar.LlarError as ex:  # a forced shape that cannot be co-resident
                assert ex.code == llar.ERR_OCCUPANCY
                return
            torch.cuda.synchronize()
            assert llar.llar_get_status()[0] == llar.OK
            if count:
                got = np.stack([inputs.bits_of(o)[:count] for o in outs])
                check(got, inputs.bits_of(x), dtype, proto)
            else:
                assert all(np.all(inputs.bits_of(o) == FILL[dtype]) for o in outs)  # nothing written
        else:  # back to back with strides, fresh inputs per iteration (kind 3: a chain)
            if count == 0:
                return
            iters = [0, 3, 17, 5][kind]
            stride = -(-count * e // 16) * 16 // e
            xi = inputs.normal(n, count, dtype, seed=seed + 1, iters=iters, exclude_sentinel=True)
            chain = 0.5 if kind == 3 else 0.0
            if chain:
                ins = device_inputs(xi[0].contiguous())
                in_stride = 0
            else:
                ins = []
                for r in range(n):
                    buf = torch.zeros(iters * stride, dtype=inputs.TORCH_DTYPE[dtype], device="cuda")
                    buf.view(iters, stride)[:, :count] = xi[:, r, :].cuda()
                    ins.append(buf)
                in_stride = stride
            outs = filled_outputs(n, iters * stride, dtype)
            try:
                llar.llar_allreduce_iters(ins, outs, count, proto, iters, in_stride, stride, chain)
            except llar.LlarError as ex:
                assert ex.code == llar.ERR_OCCUPANCY
                return
            torch.cuda.synchronize()
            assert llar.llar_get_status()[0] == llar.OK
            got = np.stack([inputs.bits_of(o).reshape(iters, stride)[:, :count] for o in outs], axis=1)
            xb = inputs.bits_of(xi)
            if chain:
                if proto.startswith("ll128"):  # atomic order: first step, then ranks agree
                    check(got[0], xb[0], dtype, proto)
                    for it in range(iters):
                        assert all(np.array_equal(got[it][0], got[it][q]) for q in range(n))
                else:
                    assert np.array_equal(got, orc.allreduce_iters(xb[0], iters, dtype, chain_scale=chain))
            else:
                for it in range(iters):
                    check(got[it], xb[it], dtype, proto)


@pytest.mark.parametrize("case", draw_cases(7, 30))
def test_random_segments_and_p2p(case):
    n, dtype, count, proto, kind, seed = case
    e = inputs.ELEM_BYTES[dtype]
    count = max(count, 1)
    with context(n, dtype, count * e * 2 + 4096):
        x = inputs.normal(n, count, dtype, seed=seed, exclude_sentinel=True)
        xb = inputs.bits_of(x)
        seg = -(-count // n)
        if kind in (0, 1):  # ReduceScatter
            p = {"auto": "auto", "ll": "ll", "sentinel": "sentinel", "ll128": "ll128"}.get(proto, "fixed_oneshot")
            if p == "sentinel" and -(-seg * e // 16) * 16 > 65536:
                return
            outs = filled_outputs(n, seg, dtype)
            llar.llar_reduce_scatter(device_inputs(x), outs, count, p)
            torch.cuda.synchronize()
            want = orc.reduce_scatter(xb, dtype)
            for s in range(n):
                got = inputs.bits_of(outs[s])[: len(want[s])]
                if p == "ll128":
                    lo, hi = orc.shard_bounds(count, n, s)
                    assert orc.compare_atomic(got[None], want[s][None], xb[:, lo:hi], dtype)[0]
                else:
                    assert np.array_equal(got, want[s])
        elif kind == 2:  # AllGather
            p = {"ll": "ll", "sentinel": "sentinel"}.get(proto, "fixed_oneshot")
            if p == "sentinel" and -(-seg * e // 16) * 16 > 65536:
                return
            segs = [x[0, lo:hi] for lo, hi in (orc.shard_bounds(count, n, s) for s in range(n))]
            ins = []
            for sg in segs:
                t = torch.zeros(max(len(sg), 8), dtype=sg.dtype, device="cuda")
                t[: len(sg)] = sg.cuda()
                ins.append(t)
            outs = filled_outputs(n, count, dtype)
            llar.llar_all_gather(ins, outs, count, p)
            torch.cuda.synchronize()
            want = orc.all_gather([inputs.bits_of(sg) for sg in segs], count)
            assert np.array_equal(np.stack([inputs.bits_of(o) for o in outs]), want)
        else:  # point to point along a random map
            rng = np.random.default_rng(seed)
            perm = list(rng.permutation(n))
            dst = [int(perm[(perm.index(r) + 1) % n]) for r in range(n)]  # a ring in random order
            if rng.integers(0, 2):
                dst[int(rng.integers(0, n))] = -1
            p = {"sentinel": "sentinel", "ll": "ll", "auto": "auto"}.get(proto, "fixed_oneshot")
            if p == "ll" and count * e > (1 << 20):
                return
            recvs = filled_outputs(n, count, dtype)
            llar.llar_sendrecv(device_inputs(x), recvs, dst, count, p)
            torch.cuda.synchronize()
            fill = np.full(xb.shape, FILL[dtype], dtype=xb.dtype)
            assert np.array_equal(np.stack([inputs.bits_of(o) for o in recvs]), p2p.sendrecv(xb, dst, fill))
        assert llar.llar_get_status()[0] == llar.OK


@pytest.mark.parametrize("case", draw_cases(314, 40))
def test_random_llbuffer_allreduce(case):
    n, dtype, count, proto, kind, seed = case
    proto = {"auto": "ll", "fixed_oneshot": "ll", "fixed_twoshot": "sentinel",
             "ll128_direct": "ll128"}.get(proto, proto)  # the LL buffer API's protocols
    e = inputs.ELEM_BYTES[dtype]
    count = max(count, 1)
    iters = [1, 2, 9, 40][kind]
    with llar.LLBuffer(n, count * e) as buf:
        x = inputs.normal(n, count, dtype, seed=seed, exclude_sentinel=True)
        ins = device_inputs(x)
        outs = filled_outputs(n, count, dtype)
        buf.allreduce(ins, outs, count, dtype, proto, iters)
        torch.cuda.synchronize()
        assert buf.status()[0] == llar.OK
        check(np.stack([inputs.bits_of(o) for o in outs]), inputs.bits_of(x), dtype, proto)


def draw_linear(seed, k):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(k):
        out.append((int(rng.integers(2, 9)), int(rng.integers(1, 17)), int(rng.integers(1, 300)),
                    8 * int(rng.integers(1, 66)), ["fp32", "fp16", "bf16"][int(rng.integers(0, 3))],
                    int(rng.integers(0, 1 << 30))))
    return out


@pytest.mark.parametrize("case", draw_linear(2718, 30))
def test_random_fused_linear(case):
    from oracle import linear as olin
    n, m, k, h, dtype, seed = case
    x, w = inputs.linear_layer(n, m, k, h, dtype, seed=seed)
    xs = [x[r].contiguous().cuda() for r in range(n)]
    ws = [w[r].contiguous().cuda() for r in range(n)]
    with llar.LLBuffer(n, m * h * inputs.ELEM_BYTES[dtype]) as buf:
        outs = filled_outputs(n, m * h, dtype)
        buf.fused_linear_allreduce(xs, ws, outs, m, k, h, dtype)
        parts = filled_outputs(n, m * h, dtype)
        llar.llar_linear_partials(xs, ws, parts, m, k, h, dtype)
        outs2 = filled_outputs(n, m * h, dtype)
        buf.allreduce(parts, outs2, m * h, dtype, "ll")
        torch.cuda.synchronize()
        assert buf.status()[0] == llar.OK
    got = np.stack([inputs.bits_of(o).reshape(m, h) for o in outs])
    ok, rel = olin.compare_linear(got, inputs.bits_of(x), inputs.bits_of(w), dtype)
    assert ok, rel
    assert np.array_equal(got, np.stack([inputs.bits_of(o).reshape(m, h) for o in outs2]))


@pytest.mark.parametrize("case", draw_cases(4242, 30))
def test_random_p2p_back_to_back(case):
    n, dtype, count, proto, kind, seed = case
    rng = np.random.default_rng(seed)
    count = max(count, 1)
    e = inputs.ELEM_BYTES[dtype]
    p = "sentinel" if proto in ("sentinel", "ll128", "fixed_twoshot") else "ll"
    if p == "ll" and count * e > (1 << 20):
        p = "sentinel"
    iters = int(rng.integers(2, 12))
    perm = list(rng.permutation(n))
    dst = [int(perm[(perm.index(r) + 1) % n]) for r in range(n)]
    if rng.integers(0, 2):
        dst[int(rng.integers(0, n))] = -1
    stride = -(-count * e // 16) * 16 // e
    with context(n, dtype, count * e + 4096):
        llar.llar_set_sentinel_chunk(16 * int(rng.integers(1, 4097)))
        x = inputs.normal(n, count, dtype, seed=seed, iters=iters, exclude_sentinel=True)
        sends = []
        for r in range(n):
            buf = torch.zeros(iters * stride, dtype=inputs.TORCH_DTYPE[dtype], device="cuda")
            buf.view(iters, stride)[:, :count] = x[:, r, :].cuda()
            sends.append(buf)
        recvs = filled_outputs(n, iters * stride, dtype)
        llar.llar_sendrecv(sends, recvs, dst, count, p, iters, stride, stride)
        torch.cuda.synchronize()
        assert llar.llar_get_status()[0] == llar.OK
        got = np.stack([inputs.bits_of(o).reshape(iters, stride)[:, :count] for o in recvs], axis=1)
        xb = inputs.bits_of(x)
        fill = np.full(xb.shape[1:], FILL[dtype], dtype=xb.dtype)
        for it in range(iters):
            assert np.array_equal(got[it], p2p.sendrecv(xb[it], dst, fill)), it
