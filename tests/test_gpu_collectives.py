"""ReduceScatter and AllGather through the C ABI against the oracle.

LL, sentinel and direct-read variants are fixed-order (rank-order float32
sums, one rounding; copies are copies), so results must match bit for bit,
including ragged and empty segments. The LL128 ReduceScatter adds with
atomics in the element type: within (N-1) ulp of sum |x|, exact on
integers. AllGather(ReduceScatter(x)) must equal AllReduce(x). Sentinel
variants move a segment in one chunk (larger segments are refused) and
leave their slots all-ones; LL128 leaves its lines zero.
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


def _fits(proto, count, n, dtype):
    # sentinel segments travel in one 64 KiB chunk
    return proto != "sentinel" or -(-_seg_len(count, n) * inputs.ELEM_BYTES[dtype] // 16) * 16 <= 65536


@pytest.mark.parametrize("proto", ["ll", "fixed_oneshot", "sentinel", "ll128"])
@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_reduce_scatter(proto, dtype, n):
    with context(n, dtype, 1 << 20):
        for count in COUNTS:
            x = inputs.normal(n, count, dtype, seed=count + n, exclude_sentinel=True)
            ins = device_inputs(x)
            seg = _seg_len(count, n)
            outs = filled_outputs(n, max(seg, 1), dtype)
            if not _fits(proto, count, n, dtype):
                with pytest.raises(llar.LlarError) as ei:
                    llar.llar_reduce_scatter(ins, outs, count, proto)
                assert ei.value.code == llar.ERR_TOO_LARGE
                continue
            llar.llar_reduce_scatter(ins, outs, count, proto)
            torch.cuda.synchronize()
            assert llar.llar_get_status()[0] == llar.OK
            xb = inputs.bits_of(x)
            want = orc.reduce_scatter(xb, dtype)
            for s in range(n):
                got = inputs.bits_of(outs[s])[: len(want[s])]
                if proto == "ll128":
                    lo, hi = orc.shard_bounds(count, n, s)
                    ok, err, rel = orc.compare_atomic(got[None], want[s][None], xb[:, lo:hi], dtype)
                    assert ok, (count, s, err, rel)
                else:
                    assert np.array_equal(got, want[s]), (count, s)


@pytest.mark.parametrize("n", [2, 4, 8])
def test_reduce_scatter_ll128_integers_exact(n):
    for dtype, lo, hi in (("fp32", -64, 64), ("fp16", -64, 64), ("bf16", -32, 32)):
        with context(n, dtype, 1 << 20):
            for count in (100, 4097, 65539):
                x = inputs.integers(n, count, dtype, seed=count, lo=lo, hi=hi)
                ins = device_inputs(x)
                outs = filled_outputs(n, _seg_len(count, n), dtype)
                llar.llar_reduce_scatter(ins, outs, count, "ll128")
                torch.cuda.synchronize()
                want = orc.reduce_scatter(inputs.bits_of(x), dtype)
                for s in range(n):
                    assert np.array_equal(inputs.bits_of(outs[s])[: len(want[s])], want[s]), (dtype, count, s)


@pytest.mark.parametrize("proto", ["ll", "fixed_oneshot", "sentinel"])
@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_all_gather(proto, dtype, n):
    with context(n, dtype, 1 << 20):
        for count in COUNTS:
            if not _fits(proto, count, n, dtype):
                continue
            full = inputs.normal(1, count, dtype, seed=count * 3 + n, exclude_sentinel=True)[0]
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


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_direct_read_segments_of_whole_vectors(dtype, n):
    # segments a whole number of 16-byte vectors long take the vector paths
    # (ReduceScatter above 64 KiB per rank: 128-thread CTAs while the grid
    # holds one vector per thread, 512-thread CTAs beyond, one element per
    # thread in 256-thread CTAs up to 64 KiB; AllGather owner push: 128- or
    # 256-thread CTAs); the last segment is ragged when count < n * per
    e = inputs.ELEM_BYTES[dtype]
    with context(n, dtype, 4 << 20):
        seen = set()
        for per in (16 // e, 1024, 40960):
            for k in (0, 1, n - 1):
                count = n * per - k
                if count * e > 4 << 20:
                    continue
                x = inputs.normal(n, count, dtype, seed=count + 7 * n, scale=0.02, exclude_sentinel=True)
                ins = device_inputs(x)
                mid = filled_outputs(n, per, dtype)
                outs = filled_outputs(n, count, dtype)
                llar.llar_reduce_scatter(ins, mid, count, "fixed_oneshot")
                seen.add(("rs", llar.llar_last_launch()[2]))
                llar.llar_all_gather(mid, outs, count, "fixed_oneshot")
                seen.add(("ag", llar.llar_last_launch()[2]))
                torch.cuda.synchronize()
                assert llar.llar_get_status()[0] == llar.OK
                xb = inputs.bits_of(x)
                want = orc.reduce_scatter(xb, dtype)
                for s in range(n):
                    assert np.array_equal(inputs.bits_of(mid[s])[: len(want[s])], want[s]), (count, s)
                got = np.stack([inputs.bits_of(o) for o in outs])
                assert np.array_equal(got, orc.allreduce(xb, dtype)), count
        assert ("rs", 256) in seen and ("ag", 128) in seen, seen
        assert ("rs", 128) in seen or ("rs", 512) in seen, seen
        if n == 8 and dtype == "fp32":
            assert ("rs", 512) in seen, seen
        if n == 2 and dtype == "fp32":
            assert ("ag", 256) in seen, seen


@pytest.mark.parametrize("n,dtype,per,k", [(8, "bf16", 560000, 3), (5, "fp32", 2000000, 2), (2, "fp16", 4194304, 0),
                                           (3, "bf16", 1400008, 1)])
def test_large_all_gather_every_element(n, dtype, per, k):
    # the owner push of whole-vector segments above 8 MiB per rank (the
    # larger thread shape), the last segment k elements short of a whole
    # vector
    e = inputs.ELEM_BYTES[dtype]
    count = n * per - k
    assert per * e % 16 == 0 and count * e > 8 << 20
    with context(n, dtype, count * e):
        full = inputs.normal(1, count, dtype, seed=per + n, exclude_sentinel=True)[0]
        bounds = [orc.shard_bounds(count, n, s) for s in range(n)]
        ins = []
        for lo, hi in bounds:
            t = torch.empty(max(hi - lo, 1), dtype=full.dtype, device="cuda")
            t[: hi - lo] = full[lo:hi].cuda()
            ins.append(t)
        outs = filled_outputs(n, count, dtype)
        llar.llar_all_gather(ins, outs, count, "auto")
        launch = llar.llar_last_launch()
        torch.cuda.synchronize()
        assert llar.llar_get_status()[0] == llar.OK
        assert launch[0] == "fixed_oneshot", launch
        want = inputs.bits_of(full)
        for r, o in enumerate(outs):
            bad = np.flatnonzero(inputs.bits_of(o) != want)
            assert bad.size == 0, (r, bad[:8].tolist())


@pytest.mark.parametrize("n", [2, 7, 8])
def test_auto_follows_the_segment_rule(n):
    # AUTO takes llar_select_protocol_segment's choice (the direct copies)
    # and the oracle's bits, for segments of whole vectors and ragged ones
    dtype = "bf16"
    with context(n, dtype, 1 << 20):
        for count in (512, 509, 32768, 32768 + 8 * 7 + 3):
            x = inputs.normal(n, count, dtype, seed=count + n, scale=0.02)
            ins = device_inputs(x)
            mid = filled_outputs(n, _seg_len(count, n), dtype)
            outs = filled_outputs(n, count, dtype)
            llar.llar_reduce_scatter(ins, mid, count, "auto")
            assert llar.llar_last_launch()[0] == llar.llar_select_protocol_segment(True, n, dtype, count)
            llar.llar_all_gather(mid, outs, count, "auto")
            assert llar.llar_last_launch()[0] == llar.llar_select_protocol_segment(False, n, dtype, count)
            torch.cuda.synchronize()
            assert llar.llar_get_status()[0] == llar.OK
            got = np.stack([inputs.bits_of(o) for o in outs])
            assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), dtype)), count


@pytest.mark.parametrize("rs,ag", [("ll", "ll"), ("fixed_oneshot", "fixed_oneshot"), ("sentinel", "sentinel"),
                                   ("ll128", "ll"), ("sentinel", "ll"), ("ll", "sentinel")])
def test_all_gather_of_reduce_scatter_is_allreduce(rs, ag):
    n, dtype = 8, "bf16"
    with context(n, dtype, 1 << 20):
        for count in (8192, 8195):
            x = inputs.normal(n, count, dtype, seed=count, scale=0.02, exclude_sentinel=True)
            ins = device_inputs(x)
            seg = _seg_len(count, n)
            mid = filled_outputs(n, seg, dtype)
            outs = filled_outputs(n, count, dtype)
            llar.llar_reduce_scatter(ins, mid, count, rs)
            llar.llar_all_gather(mid, outs, count, ag)
            torch.cuda.synchronize()
            got = np.stack([inputs.bits_of(o) for o in outs])
            xb = inputs.bits_of(x)
            if rs == "ll128":
                assert orc.compare_atomic(got, orc.allreduce(xb, dtype), xb, dtype)[0]
            else:
                assert np.array_equal(got, orc.allreduce(xb, dtype))


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_segment_staging_state_after_use(dtype):
    from test_gpu_protocol import staging_bytes
    n = 8
    with context(n, dtype, 1 << 20):
        for count in (1000, 8195, 32768):
            x = inputs.normal(n, count, dtype, seed=count, exclude_sentinel=True)
            ins = device_inputs(x)
            seg = _seg_len(count, n)
            llar.llar_reduce_scatter(ins, filled_outputs(n, seg, dtype), count, "sentinel")
            segs = [t[:seg].contiguous() for t in ins]
            llar.llar_all_gather(segs, filled_outputs(n, count, dtype), count, "sentinel")
            torch.cuda.synchronize()
            for buf in staging_bytes("sentinel", n):
                assert np.all(buf == 0xFF)
            llar.llar_reduce_scatter(ins, filled_outputs(n, seg, dtype), count, "ll128")
            torch.cuda.synchronize()
            for buf in staging_bytes("ll128", n):
                assert np.all(buf == 0)


def test_segment_collectives_reject_other_protocols():
    with context(4, "fp32", 1 << 12):
        ins = device_inputs(inputs.normal(4, 64, "fp32", seed=1))
        outs = filled_outputs(4, 64, "fp32")
        for fn, proto in ((llar.llar_reduce_scatter, "fixed_twoshot"), (llar.llar_all_gather, "fixed_twoshot"),
                          (llar.llar_all_gather, "ll128")):
            with pytest.raises(llar.LlarError) as ei:
                fn(ins, outs, 64, proto)
            assert ei.value.code == llar.ERR_UNSUPPORTED
