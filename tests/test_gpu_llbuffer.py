"""The LL buffer API (include/llar_llbuffer.h, include/llar_llbuffer.cuh):
the library's kernels written only against the public device primitives,
checked against the oracle.

* LL and sentinel AllReduces built from the primitives are bit-identical to
  the rank-order float32 sum; the LL128 one is within the atomic tolerance
  and exact on integers ("Every Microsecond Matters", summary page,
  techniques 1, 2, 4, packaged as a buffer API for custom kernels).
* Back-to-back iterations in one launch, graph replay and epochs.
* Staging state after use: sentinel vectors all ones, LL128 lines zero.
* A wait for an epoch nobody publishes times out (no fault), and reset
  makes the descriptor usable again.
* The row-parallel linear layer with the AllReduce fused into the GEMV
  epilogue matches the oracle (within the float32 dot-product bound, and
  exactly on integers), and equals the unfused pipeline bit for bit.
"""

import numpy as np
import pytest
import torch

from oracle import allreduce as orc
from oracle import linear as olin
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import FILL, device_inputs, filled_outputs

pytestmark = pytest.mark.gpu


class _Raw:
    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (ptr, False), "version": 3}


def raw(ptr, nbytes):
    torch.cuda.synchronize()
    return torch.as_tensor(_Raw(ptr, nbytes), device="cuda").cpu().numpy()


def run(buf, x, dtype, proto, iters=1):
    n, count = x.shape
    ins = device_inputs(x)
    outs = filled_outputs(n, count, dtype)
    buf.allreduce(ins, outs, count, dtype, proto, iters)
    torch.cuda.synchronize()
    assert buf.status()[0] == llar.OK, buf.status()
    return np.stack([inputs.bits_of(o) for o in outs])


def check(got, x, dtype, proto):
    xb = inputs.bits_of(x)
    want = orc.allreduce(xb, dtype)
    if proto == "ll128":
        ok, err, rel = orc.compare_atomic(got, want, xb, dtype)
        assert ok, (err, rel)
    else:
        assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("proto", ["ll", "sentinel", "ll128"])
def test_primitives_allreduce_matches_oracle(proto, dtype):
    for n in (2, 3, 5, 8):
        with llar.LLBuffer(n, 1 << 17) as buf:
            e = inputs.ELEM_BYTES[dtype]
            for count in (1, 3, 8, 33, 1000, 4097, (1 << 17) // e):
                x = inputs.normal(n, count, dtype, seed=count + n, exclude_sentinel=True)
                check(run(buf, x, dtype, proto), x, dtype, proto)


@pytest.mark.parametrize("proto", ["ll", "sentinel", "ll128"])
def test_primitives_allreduce_integers_exact(proto):
    for dtype, lo, hi in (("fp32", -64, 64), ("fp16", -64, 64), ("bf16", -32, 32)):
        with llar.LLBuffer(8, 1 << 16) as buf:
            x = inputs.integers(8, 12345, dtype, seed=3, lo=lo, hi=hi)
            got = run(buf, x, dtype, proto)
            assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), dtype))


@pytest.mark.parametrize("proto", ["ll", "sentinel", "ll128"])
def test_back_to_back_iterations_and_epochs(proto):
    n, count, dtype = 4, 8192, "bf16"
    with llar.LLBuffer(n, 1 << 15) as buf:
        x = inputs.normal(n, count, dtype, seed=7, exclude_sentinel=True)
        e0 = buf.epoch()
        check(run(buf, x, dtype, proto, iters=500), x, dtype, proto)
        assert buf.epoch() == e0 + 500
        check(run(buf, x, dtype, proto, iters=1), x, dtype, proto)
        assert buf.epoch() == e0 + 501


def test_two_ranks_128_bytes_one_shot_10000_iterations():
    # the pages' two-rank 128-byte one-shot case, through the buffer API
    with llar.LLBuffer(2, 128) as buf:
        x = inputs.uniform(2, 32, "fp32", seed=0)
        assert np.array_equal(run(buf, x, "fp32", "ll", iters=10000), orc.allreduce(inputs.bits_of(x), "fp32"))


def test_graph_replay_gets_fresh_epochs():
    n, count, dtype = 8, 8192, "bf16"
    with llar.LLBuffer(n, 1 << 14) as buf:
        x = inputs.normal(n, count, dtype, seed=9)
        ins = device_inputs(x)
        outs = filled_outputs(n, count, dtype)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            buf.allreduce(ins, outs, count, dtype, "ll", 1, stream=s)  # warm the caches outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            buf.allreduce(ins, outs, count, dtype, "ll", 1, stream=s)
        e0 = buf.epoch()
        for _ in range(5):
            for o in outs:
                o.view(torch.int16).fill_(FILL[dtype])
            g.replay()
            torch.cuda.synchronize()
            got = np.stack([inputs.bits_of(o) for o in outs])
            assert np.array_equal(got, orc.allreduce(inputs.bits_of(x), dtype))
        assert buf.epoch() == e0 + 5


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_staging_state_after_use(dtype):
    n = 8
    with llar.LLBuffer(n, 1 << 16) as buf:
        d = buf.desc
        for count in (100, 8191, (1 << 16) // inputs.ELEM_BYTES[dtype]):
            x = inputs.normal(n, count, dtype, seed=count, exclude_sentinel=True)
            check(run(buf, x, dtype, "sentinel", iters=3), x, dtype, "sentinel")
            assert np.all(raw(d.sen, n * d.sen_rank_stride) == 0xFF)
            check(run(buf, x, dtype, "ll128", iters=3), x, dtype, "ll128")
            assert np.all(raw(d.ll128, n * d.ll128_rank_stride) == 0)


def test_wait_that_nobody_satisfies_times_out_and_reset_recovers():
    n, count, dtype = 4, 4096, "fp16"
    with llar.LLBuffer(n, 1 << 14) as buf:
        buf.set_timeout_ns(2_000_000)  # 2 ms
        e = buf.epoch()
        buf.probe_wait(rank=1, src=3, epoch=e + 1000, word=5)
        torch.cuda.synchronize()
        code, rank, epoch = buf.status()
        assert (code, rank, epoch) == (llar.ERR_TIMEOUT, 1, e + 1000)
        with pytest.raises(llar.LlarError) as ei:
            buf.allreduce(device_inputs(inputs.normal(n, count, dtype, seed=1)),
                          filled_outputs(n, count, dtype), count, dtype, "ll")
        assert ei.value.code == llar.ERR_TIMEOUT
        buf.reset()
        assert buf.status()[0] == llar.OK
        buf.set_timeout_ns(2_000_000_000)
        for proto in ("ll", "sentinel", "ll128"):
            x = inputs.normal(n, count, dtype, seed=2, exclude_sentinel=True)
            check(run(buf, x, dtype, proto), x, dtype, proto)


def test_argument_errors():
    with llar.LLBuffer(4, 1024) as buf:
        x = device_inputs(inputs.normal(4, 512, "fp16", seed=1))
        o = filled_outputs(4, 512, "fp16")
        with pytest.raises(llar.LlarError) as ei:
            buf.allreduce(x, o, 513, "fp16", "ll")
        assert ei.value.code == llar.ERR_TOO_LARGE
        with pytest.raises(llar.LlarError) as ei:
            buf.allreduce(x, o, 512, "fp16", "fixed_oneshot")
        assert ei.value.code == llar.ERR_UNSUPPORTED
        with pytest.raises(llar.LlarError) as ei:
            buf.allreduce(x, x, 512, "fp16", "ll")  # outputs alias inputs
        assert ei.value.code == llar.ERR_INVALID
        with pytest.raises(llar.LlarError) as ei:
            buf.allreduce(x, o, 512, "fp16", "ll", iters=0)
        assert ei.value.code == llar.ERR_INVALID


# ---------------------------------------------------- fused linear layer
def linear(buf, x, w, dtype, fused=True):
    n, m, k = x.shape
    h = w.shape[2]
    xs = [x[r].contiguous().cuda() for r in range(n)]
    ws = [w[r].contiguous().cuda() for r in range(n)]
    outs = filled_outputs(n, m * h, dtype)
    if fused:
        buf.fused_linear_allreduce(xs, ws, outs, m, k, h, dtype)
    else:
        ps = filled_outputs(n, m * h, dtype)
        llar.llar_linear_partials(xs, ws, ps, m, k, h, dtype)
        buf.allreduce(ps, outs, m * h, dtype, "ll")
    torch.cuda.synchronize()
    assert buf.status()[0] == llar.OK
    return np.stack([inputs.bits_of(o).reshape(m, h) for o in outs])


# the last two give 8 ranks more column tiles than CTAs (40 and 48 tiles of
# 256 columns on the tensor-core path): CTAs with two tiles
SHAPES = [(2, 1, 1, 8), (2, 3, 37, 136), (4, 16, 64, 264), (8, 1, 1024, 512), (8, 5, 200, 8),
          (3, 2, 9, 1000), (8, 8, 64, 10240), (8, 16, 32, 12288)]


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_fused_linear_matches_oracle(shape, dtype):
    n, m, k, h = shape
    x, w = inputs.linear_layer(n, m, k, h, dtype, seed=sum(shape))
    with llar.LLBuffer(n, m * h * inputs.ELEM_BYTES[dtype]) as buf:
        got = linear(buf, x, w, dtype)
        ok, rel = olin.compare_linear(got, inputs.bits_of(x), inputs.bits_of(w), dtype)
        assert ok, rel
        # every rank holds the same result
        assert all(np.array_equal(got[0], got[q]) for q in range(n))
        # and the unfused pipeline (GEMV launch + LL AllReduce launch) gives the same bits
        assert np.array_equal(got, linear(buf, x, w, dtype, fused=False))


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_fused_linear_integers_exact(dtype):
    n, m, k, h = 8, 4, 100, 264
    x, w = inputs.linear_layer(n, m, k, h, dtype, seed=5, integer=True)
    with llar.LLBuffer(n, m * h * 4) as buf:
        got = linear(buf, x, w, dtype)
    assert np.array_equal(got, olin.linear_allreduce(inputs.bits_of(x), inputs.bits_of(w), dtype))


def test_fused_linear_decode_layer_full_size_sampled():
    # 8 ranks, one token, hidden 8192 split 8 ways (K = 1024 per rank), H = 8192
    n, m, k, h, dtype = 8, 1, 1024, 8192, "bf16"
    x, w = inputs.linear_layer(n, m, k, h, dtype, seed=21)
    with llar.LLBuffer(n, m * h * 2) as buf:
        got = linear(buf, x, w, dtype)
        again = linear(buf, x, w, dtype)
    assert np.array_equal(got, again)  # deterministic
    cols = np.random.default_rng(3).choice(h, 512, replace=False)
    xb = inputs.bits_of(x)
    wb = inputs.bits_of(w)[:, :, cols]
    ok, rel = olin.compare_linear(got[:, :, cols], xb, wb, dtype)
    assert ok, rel


def test_fused_linear_argument_errors():
    with llar.LLBuffer(2, 1024) as buf:
        x, w = inputs.linear_layer(2, 1, 8, 1024, "bf16", seed=1)
        xs = [t.cuda() for t in x]
        ws = [t.cuda() for t in w]
        outs = filled_outputs(2, 1024, "bf16")
        with pytest.raises(llar.LlarError) as ei:  # M*H*2 = 2048 > 1024 bytes of capacity
            buf.fused_linear_allreduce(xs, ws, outs, 1, 8, 1024, "bf16")
        assert ei.value.code == llar.ERR_TOO_LARGE
