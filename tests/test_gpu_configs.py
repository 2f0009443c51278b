"""Parity at the full sizes of the five workload configurations.

C1  N=2, fp32, 32 elements (128 B), 1000 iterations of fresh U[-1,1)
    inputs, LL and fixed-order one-shot: every output compared.
C2  N=4, bf16, 8192 elements (16 KiB), N(0,1)*0.02, 10000 back-to-back
    AllReduces in one launch, LL and sentinel: fresh inputs per iteration,
    every iteration compared in full.
C3  N=8, LL128 two-shot, fp32/fp16/bf16, 4 KiB .. 1 MiB per rank in powers
    of two: N(0,1) within the atomic tolerance, integers exactly.
C4  N=8, fp16, 64 KiB, sentinel with 8 KiB double-buffered chunks: 100
    calls, staging back to all-ones after each.
C5  decode chain: N=4 and 8, bf16, 65536 elements, 160 dependent
    AllReduces with scale 0.5 (and 1/N) for every protocol; bandwidth sweep
    1 .. 256 MiB per rank at N=8 with the fixed-order two-shot path, every
    element up to 64 MiB, sampled elements above.
Also the exact launches bench.py times: 8 ranks x 16 KiB bf16, 10000
back-to-back AllReduces of the same buffers, 8 ranks x 64 MiB bf16 (every
element), and the ReduceScatter and AllGather of 8 ranks x 64 MiB bf16
(every element).
"""

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from oracle import fpformats as fp
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import allreduce, allreduce_iters, context, device_inputs, filled_outputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("proto", ["ll", "fixed_oneshot"])
def test_c1_two_ranks_128_bytes_1000_fresh_iterations(proto):
    n, count, iters = 2, 32, 1000
    x = inputs.uniform(n, count, "fp32", seed=0, iters=iters)
    with context(n, "fp32", 1 << 12):
        got = allreduce_iters(x, "fp32", proto, iters)
    assert np.array_equal(got, orc.allreduce_iters(inputs.bits_of(x), iters, "fp32"))


@pytest.mark.parametrize("proto", ["ll", "sentinel"])
def test_c2_four_ranks_16k_bf16_10000_calls(proto):
    n, count, iters = 4, 8192, 10000
    x = inputs.normal(n, count, "bf16", seed=1, scale=0.02, iters=iters)
    with context(n, "bf16", 1 << 16):
        llar.llar_set_sentinel_chunk(16384)
        got = allreduce_iters(x, "bf16", proto, iters)
    # every iteration: the oracle is elementwise, so the [iters, N, count]
    # inputs are reduced as one [N, iters * count] problem
    xb = inputs.bits_of(x)
    want = orc.allreduce(np.ascontiguousarray(xb.transpose(1, 0, 2)).reshape(n, iters * count), "bf16")
    got_flat = np.ascontiguousarray(got.transpose(1, 0, 2)).reshape(n, iters * count)
    bad = np.flatnonzero((got_flat != want).any(axis=0))
    assert bad.size == 0, (bad[:8] // count).tolist()


@pytest.mark.parametrize("proto", ["ll128", "ll128_direct"])
@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_c3_ll128_eight_ranks_4k_to_1m(dtype, proto):
    n = 8
    e = fp.ELEM_BYTES[dtype]
    lo, hi = (-32, 32) if dtype == "bf16" else (-64, 64)
    with context(n, dtype, 1 << 20):
        for k in range(9):
            count = (4096 << k) // e
            x = inputs.normal(n, count, dtype, seed=2)
            xb = inputs.bits_of(x)
            got = allreduce(x, dtype, proto)
            ok, err, rel = orc.compare_atomic(got, orc.allreduce(xb, dtype), xb, dtype)
            assert ok, (count, err, rel)
            xi = inputs.integers(n, count, dtype, seed=2, lo=lo, hi=hi)
            assert np.array_equal(allreduce(xi, dtype, proto), orc.allreduce(inputs.bits_of(xi), dtype))


def test_c4_sentinel_eight_ranks_64k_fp16_8k_chunks_100_calls():
    from test_gpu_protocol import staging_bytes
    n, count = 8, 32768
    with context(n, "fp16", 1 << 16):
        llar.llar_set_sentinel_chunk(8192)
        for call in range(100):
            x = inputs.normal(n, count, "fp16", seed=3 + call, exclude_sentinel=True)
            got = allreduce(x, "fp16", "sentinel")
            assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), "fp16")), call
            if call % 10 == 0:
                for buf in staging_bytes("sentinel", n):
                    assert np.all(buf == 0xFF)


@pytest.mark.parametrize("n", [4, 8])
@pytest.mark.parametrize("proto", ["ll", "sentinel", "fixed_oneshot", "fixed_twoshot", "ll128", "ll128_direct"])
def test_c5_decode_chain_160_layers(n, proto):
    count, iters = 65536, 160
    x = inputs.normal(n, count, "bf16", seed=4, scale=0.02)
    xb = inputs.bits_of(x)
    with context(n, "bf16", 1 << 20):
        for scale in (0.5, 1.0 / n):
            got = allreduce_iters(x, "bf16", proto, iters, chain_scale=scale)
            if proto.startswith("ll128"):
                # atomic order: the first step within the tolerance, every
                # step the same on every rank (the exact chain is pinned in
                # test_gpu_parity with inputs whose sums are all exact)
                ok, err, rel = orc.compare_atomic(got[0], orc.allreduce(xb, "bf16"), xb, "bf16")
                assert ok, (scale, err, rel)
                for e in range(iters):
                    assert all(np.array_equal(got[e][0], got[e][q]) for q in range(n)), (scale, e)
            else:
                want = orc.allreduce_iters(xb, iters, "bf16", chain_scale=scale)
                assert np.array_equal(got, want), scale


def _sampled_check(ins, outs, count, idx):
    """Compare outputs at element indices idx with the oracle on those columns."""
    n = len(ins)
    cols = torch.as_tensor(idx, device=ins[0].device)
    xb = np.stack([inputs.bits_of(t[cols]) for t in ins])
    want = orc.allreduce(xb, "bf16")
    got = np.stack([inputs.bits_of(t[cols]) for t in outs])
    assert np.array_equal(got, want)


def _full_check(ins, outs):
    """Compare every element of every rank's output with the oracle."""
    xb = np.stack([inputs.bits_of(t) for t in ins])
    want = orc.allreduce(xb, "bf16")[0]
    del xb
    for r, t in enumerate(outs):
        got = inputs.bits_of(t)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, (r, bad[:8].tolist())


def _bw_inputs(n, count):
    gen = torch.Generator(device="cuda")
    ins = []
    for r in range(n):
        gen.manual_seed(5 + r)
        ins.append(torch.randn(count, device="cuda", generator=gen).to(torch.bfloat16))
    return ins


def test_c5_bandwidth_sweep_1m_to_256m():
    # every element up to 64 MiB per rank (tile boundaries of the TMA ring
    # included), sampled elements at 128 and 256 MiB
    n = 8
    with context(n, "bf16", 256 << 20):
        rng = np.random.default_rng(5)
        for mib in (1, 2, 4, 8, 16, 32, 64, 128, 256):
            count = (mib << 20) // 2
            ins = _bw_inputs(n, count)
            outs = [torch.empty_like(t) for t in ins]
            llar.llar_allreduce(ins, outs, count, "fixed_twoshot")
            torch.cuda.synchronize()
            if mib <= 64:
                _full_check(ins, outs)
            else:
                idx = np.concatenate([rng.integers(0, count, 4000), np.arange(64), np.arange(count - 64, count)])
                _sampled_check(ins, outs, count, idx)
            del ins, outs
            torch.cuda.empty_cache()


def test_bench_latency_launch_exactly():
    # 8 ranks x 16 KiB bf16, 10000 back-to-back AllReduces on the same buffers
    n, count, iters = 8, 8192, 10000
    x = inputs.normal(n, count, "bf16", seed=1, scale=0.02)
    with context(n, "bf16", 64 << 20):
        ins = device_inputs(x)
        outs = filled_outputs(n, count, "bf16")
        llar.llar_allreduce_iters(ins, outs, count, "auto", iters, 0, 0, 0.0)
        torch.cuda.synchronize()
        assert llar.llar_get_status()[0] == llar.OK
        assert llar.llar_last_launch()[0] == "ll"
        got = np.stack([inputs.bits_of(o) for o in outs])
    assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), "bf16"))


def test_bench_bandwidth_launch_exactly_every_element():
    # the launch bench.py times: 8 ranks x 64 MiB bf16, AUTO -> TMA two-shot
    n, count = 8, 32 << 20
    with context(n, "bf16", 64 << 20):
        ins = _bw_inputs(n, count)
        outs = [torch.empty_like(t) for t in ins]
        llar.llar_allreduce(ins, outs, count, "fixed_twoshot")
        torch.cuda.synchronize()
        assert llar.llar_get_status()[0] == llar.OK
        _full_check(ins, outs)


def test_bench_segment_launches_exactly_every_element():
    # the launches of bench.py's segment row: 8 ranks x 64 MiB bf16,
    # ReduceScatter then AllGather by AUTO (direct copies, vector paths)
    n, count = 8, 32 << 20
    seg = count // n
    with context(n, "bf16", 64 << 20):
        ins = _bw_inputs(n, count)
        mid = [torch.empty(seg, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        llar.llar_reduce_scatter(ins, mid, count, "auto")
        rs_launch = llar.llar_last_launch()
        outs = [torch.empty_like(t) for t in ins]
        llar.llar_all_gather(mid, outs, count, "auto")
        ag_launch = llar.llar_last_launch()
        torch.cuda.synchronize()
        assert llar.llar_get_status()[0] == llar.OK
        assert rs_launch[0] == ag_launch[0] == "fixed_oneshot"
        assert rs_launch[2] == 512 and ag_launch[2] == 256, (rs_launch, ag_launch)
        xb = np.stack([inputs.bits_of(t) for t in ins])
        want = orc.allreduce(xb, "bf16")[0]
        del xb
        for s in range(n):
            bad = np.flatnonzero(inputs.bits_of(mid[s]) != want[s * seg:(s + 1) * seg])
            assert bad.size == 0, ("reduce_scatter", s, bad[:8].tolist())
        for r, t in enumerate(outs):
            bad = np.flatnonzero(inputs.bits_of(t) != want)
            assert bad.size == 0, ("all_gather", r, bad[:8].tolist())


@pytest.mark.parametrize("n,count,chain", [(8, 65536, 0.5), (4, 65536, 0.5), (8, 32768, 0.0), (8, 8192, 0.0),
                                           (8, 2048, 0.0), (3, 40000, 0.0)])
def test_ll128_threads_cover_a_ctas_lines_in_one_pass(n, count, chain):
    # an LL128 CTA takes ceil(L / G) whole lines of every segment (8 lanes
    # each); below the wide shape (more items than one 512-thread CTA per
    # SM holds) its threads cover them in one pass
    x = inputs.normal(n, count, "bf16", seed=9, scale=0.02)
    with context(n, "bf16", count * 2):
        ins = device_inputs(x)
        outs = filled_outputs(n, count, "bf16")
        llar.llar_allreduce_iters(ins, outs, count, "ll128", 2, 0, 0, chain)
        torch.cuda.synchronize()
        assert llar.llar_get_status()[0] == llar.OK
        proto, G, T, _ = llar.llar_last_launch()
        got = np.stack([inputs.bits_of(o) for o in outs])
    assert proto == "ll128"
    lines = -(-(-(-count // n)) // 63)
    items = n * (-(-lines // G)) * 8
    assert T >= min(items, 512), (G, T, items)
    assert all(np.array_equal(got[0], got[q]) for q in range(n))
