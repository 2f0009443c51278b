"""Protocol state, errors, fault handling and the probes, through the C ABI.

* Sentinel staging holds the all-ones (-NaN) pattern again after every call
  ("Every Microsecond Matters", summary page, technique 2: the buffer must be
  reset after each use).
* LL128 line staging is all zero after every call (the owner clears each
  line after reading it, so the next count starts from zero).
* Epochs only grow.
* Invalid arguments are refused before any launch.
* A virtual rank that never sends makes its peers' waits run out: the
  status word says TIMEOUT, nothing hangs, and after llar_reset the same
  context computes exact results again. No GPU fault is raised.
"""

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from oracle import protocol as oproto
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import allreduce, allreduce_iters, context, device_inputs, filled_outputs

pytestmark = pytest.mark.gpu


class _Raw:
    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (ptr, False), "version": 3}


def staging_bytes(protocol, n):
    ptr, stride, used = llar.llar_staging(protocol)
    torch.cuda.synchronize()
    return [torch.as_tensor(_Raw(ptr + r * stride, used), device="cuda").cpu().numpy()
            for r in range(n)]


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_sentinel_staging_refilled_after_each_call(dtype):
    n = 8
    with context(n, dtype, 1 << 20):
        llar.llar_set_sentinel_chunk(8192)
        for count in (4096, 32768, 32771):
            x = inputs.normal(n, count, dtype, seed=count, exclude_sentinel=True)
            got = allreduce(x, dtype, "sentinel")
            assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), dtype))
            for buf in staging_bytes("sentinel", n):
                assert np.all(buf == 0xFF)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_ll128_lines_clear_after_each_call(dtype):
    n = 8
    with context(n, dtype, 1 << 20):
        for count in (100, 65536, 70001):
            x = inputs.normal(n, count, dtype, seed=count)
            allreduce(x, dtype, "ll128")
            for buf in staging_bytes("ll128", n):
                assert oproto.ll128_lines_clear(buf)


def test_ll128_direct_keeps_only_the_last_slot_after_each_call():
    # three line slots in turn (sequence s uses slot s % 3, counted per
    # context over direct AllReduces only); each AllReduce zeroes the slot
    # before its own, so after a call only the last one holds data, whatever
    # other protocols ran in between
    n, dtype = 8, "bf16"
    with context(n, dtype, 1 << 20):
        seq = 0
        for count, iters, other in ((100, 1, None), (65536, 1, "ll"), (70001, 4, "ll128"), (3000, 2, "sentinel")):
            if other:
                allreduce(inputs.normal(n, 1000, dtype, seed=count + 1, exclude_sentinel=True), dtype, other)
            x = inputs.normal(n, count, dtype, seed=count, iters=iters)
            got = allreduce_iters(x, dtype, "ll128_direct", iters)
            xb = inputs.bits_of(x)
            for e in range(iters):
                assert orc.compare_atomic(got[e], orc.allreduce(xb[e], dtype), xb[e], dtype)[0], (count, e)
            seq += iters
            _, _, used = llar.llar_staging("ll128_direct")
            per_slot = used // 3
            for buf in staging_bytes("ll128_direct", n):
                for slot in range(3):
                    part = buf[slot * per_slot:(slot + 1) * per_slot]
                    if slot != seq % 3:
                        assert oproto.ll128_lines_clear(part), (count, slot)
                    else:
                        assert part.any()  # the last AllReduce's reduced lines


def test_epochs_strictly_increase():
    with context(4, "bf16", 1 << 16):
        x = inputs.normal(4, 100, "bf16", seed=1)
        e0 = llar.llar_epoch()
        allreduce(x, "bf16", "ll")
        e1 = llar.llar_epoch()
        allreduce_iters(inputs.normal(4, 100, "bf16", seed=2, iters=5), "bf16", "ll", 5)
        e2 = llar.llar_epoch()
        assert e0 >= 1 and e1 == e0 + 1 and e2 == e1 + 5


def test_layout_matches_page_constants():
    # 8 bytes of flag per 8 bytes of data; 128-byte lines with one flag element
    for dtype in ("fp32", "fp16", "bf16"):
        lb, pl, st = llar.llar_layout("ll", dtype, 8, 8192)
        e = inputs.ELEM_BYTES[dtype]
        assert lb == 16 and pl * e == 8
        assert st == 2 * oproto.ll_staging_bytes(8192 * e)
        lb, pl, st = llar.llar_layout("ll128", dtype, 8, 1 << 18)
        assert lb == oproto.LL128_LINE_BYTES and pl == oproto.ll128_payload_elems(dtype)
        assert st == 2 * oproto.ll128_round_staging_bytes(1 << 18, 8, dtype)


def test_invalid_arguments_rejected():
    with context(4, "fp16", 1 << 16):
        x = inputs.normal(4, 256, "fp16", seed=3)
        ins = device_inputs(x)
        outs = filled_outputs(4, 256, "fp16")
        cases = [
            (lambda: llar.llar_allreduce(ins, outs, 256, 9), llar.ERR_INVALID),
            (lambda: llar.llar_allreduce(ins, [o.data_ptr() + 2 for o in outs], 200, "ll"), llar.ERR_INVALID),
            (lambda: llar.llar_allreduce(ins, [ins[0]] + outs[1:], 256, "ll"), llar.ERR_INVALID),
            (lambda: llar.llar_allreduce(ins, [outs[0]] * 4, 256, "ll"), llar.ERR_INVALID),
            (lambda: llar.llar_allreduce(ins, outs, (1 << 16) // 2 + 8, "ll"), llar.ERR_TOO_LARGE),
            (lambda: llar.llar_init(4, "fp16", 1 << 16), llar.ERR_INVALID),
        ]
        for fn, code in cases:
            with pytest.raises(llar.LlarError) as ei:
                fn()
            assert ei.value.code == code
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_allreduce(ins, outs, 256, "ll")
    assert ei.value.code == llar.ERR_NOT_INIT


@pytest.mark.parametrize("proto", ["ll", "sentinel", "ll128", "ll128_direct"])
def test_dead_rank_times_out_then_recovers(proto):
    n, dtype, count = 4, "bf16", 4096
    with context(n, dtype, 1 << 20, timeout_ns=20_000_000):
        x = inputs.normal(n, count, dtype, seed=4)
        llar.llar_debug_inject(2, "skip")
        ins = device_inputs(x)
        outs = filled_outputs(n, count, dtype)
        llar.llar_allreduce(ins, outs, count, proto)
        torch.cuda.synchronize()
        code, rank, cta, epoch = llar.llar_get_status()
        assert code == llar.ERR_TIMEOUT and 0 <= rank < n and epoch >= 1
        if not proto.startswith("ll128"):  # in LL128 the silent rank also waits, as owner of its segment
            assert rank != 2
        with pytest.raises(llar.LlarError) as ei:  # sticky until reset
            llar.llar_allreduce(ins, outs, count, proto)
        assert ei.value.code == llar.ERR_TIMEOUT
        llar.llar_debug_inject(-1, "none")
        llar.llar_reset()
        got = allreduce(x, dtype, proto)
        want = orc.allreduce(inputs.bits_of(x), dtype)
        if proto.startswith("ll128"):
            assert orc.compare_atomic(got, want, inputs.bits_of(x), dtype)[0]
        else:
            assert np.array_equal(got, want)


@pytest.mark.parametrize("proto", ["ll", "sentinel", "ll128", "ll128_direct"])
def test_poisoned_rank_times_out(proto):
    n, dtype, count = 8, "fp16", 2048
    with context(n, dtype, 1 << 20, timeout_ns=20_000_000):
        llar.llar_debug_inject(5, "poison")
        x = inputs.normal(n, count, dtype, seed=6)
        ins = device_inputs(x)
        outs = filled_outputs(n, count, dtype)
        llar.llar_allreduce(ins, outs, count, proto)
        torch.cuda.synchronize()
        assert llar.llar_get_status()[0] == llar.ERR_TIMEOUT
        llar.llar_debug_inject(-1, "none")
        llar.llar_reset()
        assert llar.llar_get_status()[0] == llar.OK


@pytest.mark.parametrize("proto", ["fixed_oneshot", "fixed_twoshot"])
def test_fixed_chain_dead_rank_times_out(proto):
    n, dtype, count = 4, "fp32", 4096
    with context(n, dtype, 1 << 20, timeout_ns=20_000_000):
        llar.llar_debug_inject(1, "skip")
        x = inputs.normal(n, count, dtype, seed=7)
        ins = device_inputs(x)
        outs = filled_outputs(n, count, dtype)
        llar.llar_allreduce_iters(ins, outs, count, proto, 4, 0, 0, 0.5)
        torch.cuda.synchronize()
        assert llar.llar_get_status()[0] == llar.ERR_TIMEOUT
        llar.llar_debug_inject(-1, "none")
        llar.llar_reset()


@pytest.mark.parametrize("proto", ["ll", "sentinel", "ll128", "ll128_direct", "fixed_oneshot", "fixed_twoshot"])
def test_delayed_rank_still_exact(proto):
    n, dtype, count, iters = 4, "bf16", 8192, 6
    with context(n, dtype, 1 << 20):
        llar.llar_debug_inject(3, "delay")
        x = inputs.normal(n, count, dtype, seed=8, scale=0.02)
        got = allreduce_iters(x, dtype, proto, iters, chain_scale=0.5)
        want = orc.allreduce_iters(inputs.bits_of(x), iters, dtype, chain_scale=0.5)
        if proto.startswith("ll128"):
            assert orc.compare_atomic(got[0], want[0], inputs.bits_of(x), dtype)[0]
        else:
            assert np.array_equal(got, want)


def test_host_buffer_entry_point():
    n, dtype, count = 8, "bf16", 8192
    with context(n, dtype, 1 << 20):
        x = inputs.normal(n, count, dtype, seed=9).pin_memory()
        out = torch.empty_like(x).pin_memory()
        for proto in ("ll", "sentinel", "fixed_twoshot"):
            llar.llar_allreduce_host(x, out, count, proto)
            torch.cuda.synchronize()
            assert np.array_equal(inputs.bits_of(out), orc.allreduce(inputs.bits_of(x), dtype))


def test_host_buffer_registration():
    # registered pinned buffers skip the per-call pointer queries; results
    # are the same, sub-ranges of a registered buffer resolve too, and the
    # table refuses overlaps, pageable memory and unknown addresses
    n, dtype, count = 8, "bf16", 8192
    with context(n, dtype, 1 << 20):
        x = inputs.normal(n, 2 * count, dtype, seed=11).pin_memory()
        out = torch.empty_like(x).pin_memory()
        llar.llar_host_register(x)
        llar.llar_host_register(out)
        try:
            for proto in ("ll", "fixed_twoshot"):
                for _ in range(2):
                    llar.llar_allreduce_host(x, out, 2 * count, proto)
                    torch.cuda.synchronize()
                    assert np.array_equal(inputs.bits_of(out), orc.allreduce(inputs.bits_of(x), dtype))
            # a [n][count] view that starts inside the registered buffers
            xs = x.view(-1)[count:count + n * count].view(n, count)
            os_ = out.view(-1)[count:count + n * count].view(n, count)
            llar.llar_allreduce_host(xs, os_, count, "ll")
            torch.cuda.synchronize()
            assert np.array_equal(inputs.bits_of(os_), orc.allreduce(inputs.bits_of(xs.clone()), dtype))
            with pytest.raises(llar.LlarError):
                llar.llar_host_register(x.view(-1)[8:], 64)  # overlaps x
            with pytest.raises(llar.LlarError):
                llar.llar_host_register(torch.empty(64, dtype=torch.uint8))  # pageable
        finally:
            llar.llar_host_unregister(x)
            llar.llar_host_unregister(out)
        with pytest.raises(llar.LlarError):
            llar.llar_host_unregister(x)  # no longer registered
        # unregistered pinned buffers still work (queried per call)
        llar.llar_allreduce_host(x, out, 2 * count, "ll")
        torch.cuda.synchronize()
        assert np.array_equal(inputs.bits_of(out), orc.allreduce(inputs.bits_of(x), dtype))


@pytest.mark.parametrize("n,dtype", [(8, "bf16"), (3, "fp32"), (6, "fp16")])
def test_host_buffer_auto_follows_the_host_rule(n, dtype):
    # AUTO on host memory takes the host rule (LL for a few KiB, the direct
    # two-shot above, which from 32 KiB with 6-8 ranks streams the host
    # inputs through shared memory with TMA bulk copies); bits as the oracle
    e = inputs.ELEM_BYTES[dtype]
    with context(n, dtype, 1 << 20):
        for nbytes in (64, 4096, 16384 + 16, 65536, 262144 + 32):
            count = nbytes // e
            x = inputs.normal(n, count, dtype, seed=nbytes + n).pin_memory()
            out = torch.empty_like(x).pin_memory()
            llar.llar_host_register(x)
            llar.llar_host_register(out)
            try:
                llar.llar_allreduce_host(x, out, count, "auto")
                torch.cuda.synchronize()
                assert llar.llar_last_launch()[0] == llar.llar_select_protocol_host(n, dtype, count)
                assert np.array_equal(inputs.bits_of(out), orc.allreduce(inputs.bits_of(x), dtype)), nbytes
            finally:
                llar.llar_host_unregister(x)
                llar.llar_host_unregister(out)


def test_host_buffer_entry_point_pageable_and_ragged():
    # pageable host memory (and a row size that is not a multiple of 16
    # bytes) takes the staged-copy path
    n, dtype = 4, "fp16"
    with context(n, dtype, 1 << 20):
        for count in (8192, 8191):
            x = inputs.normal(n, count, dtype, seed=10 + count)
            out = torch.empty_like(x)
            for proto in ("ll", "fixed_oneshot"):
                llar.llar_allreduce_host(x, out, count, proto)
                torch.cuda.synchronize()
                assert np.array_equal(inputs.bits_of(out), orc.allreduce(inputs.bits_of(x), dtype))


def test_sol_probe_is_consistent():
    with context(2, "fp32", 1 << 12):
        l2, wr, sol = llar.llar_sol_probe()
        assert 0.05 < l2 < 5.0 and 0.05 < wr < 10.0
        assert abs(sol - (2 * l2 + wr)) < 1e-9
        d = llar.llar_sol_probe_detail()
        assert len(d["chase_ns"]) >= 100 and all(v > 0 for v in d["rt_ns"])
        assert all(a != b for a, b in zip(d["smid_a"], d["smid_b"]))


@pytest.mark.parametrize("n,dtype,count,chunk,iters", [(5, "fp16", 118700, 65536, 17),
                                                      (8, "bf16", 3 * 4096 + 100, 8192, 50),
                                                      (3, "fp32", 2 * 2048 + 1, 8192, 9)])
def test_sentinel_partial_last_chunk_across_iterations(n, dtype, count, chunk, iters):
    # vectors beyond a partial last chunk miss that chunk's exchange, so the
    # next iteration's first push must wait for the peer's reset itself
    with context(n, dtype, 1 << 20):
        llar.llar_set_sentinel_chunk(chunk)
        x = inputs.normal(n, count, dtype, seed=count, iters=iters, exclude_sentinel=True)
        got = allreduce_iters(x, dtype, "sentinel", iters)
        xb = inputs.bits_of(x)
        for e in range(iters):
            assert np.array_equal(got[e], orc.allreduce(xb[e], dtype)), e
        for buf in staging_bytes("sentinel", n):
            assert np.all(buf == 0xFF)
