"""Point-to-point transfers between virtual ranks (llar_sendrecv), LL and
sentinel, against the oracle (a bit copy along the destination map):
rings, pairs, partial maps, fresh data in every back-to-back transfer (so
that a slot reused before its acknowledgement would show), ragged and
maximum sizes, multi-chunk sentinel transfers, errors, and a receiver that
never acknowledges (the sender's wait runs out; no fault)."""

import numpy as np
import pytest
import torch

from oracle import p2p
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import FILL, context, filled_outputs

pytestmark = pytest.mark.gpu


def run(x, dtype, dst, proto, iters=1, chunk=None):
    """x: [iters, N, count] CPU tensor; returns [iters, N, count] bits of recv."""
    it, n, count = x.shape
    e = inputs.ELEM_BYTES[dtype]
    stride = -(-count * e // 16) * 16 // e
    sends = []
    for r in range(n):
        buf = torch.zeros(it * stride, dtype=inputs.TORCH_DTYPE[dtype], device="cuda")
        buf.view(it, stride)[:, :count] = x[:, r, :].cuda()
        sends.append(buf)
    recvs = filled_outputs(n, it * stride, dtype)
    if chunk:
        llar.llar_set_sentinel_chunk(chunk)
    llar.llar_sendrecv(sends, recvs, dst, count, proto, it, stride, stride)
    torch.cuda.synchronize()
    code = llar.llar_get_status()
    assert code[0] == llar.OK, code
    return np.stack([inputs.bits_of(o).reshape(it, stride)[:, :count] for o in recvs], axis=1)


def expected(x, dtype, dst):
    xb = inputs.bits_of(x)
    fill = np.full(xb.shape[1:], FILL[dtype], dtype=xb.dtype)
    return np.stack([p2p.sendrecv(xb[e], dst, fill) for e in range(xb.shape[0])])


MAPS = {
    "ring8": (8, [(r + 1) % 8 for r in range(8)]),
    "pairs4": (4, [1, 0, 3, 2]),
    "pipeline5": (5, [1, 2, 3, 4, -1]),
    "single2": (2, [1, -1]),
    "reverse7": (7, [6, 5, 4, -1, 2, 1, 0]),
}


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("proto", ["ll", "sentinel", "fixed_oneshot"])
@pytest.mark.parametrize("name", sorted(MAPS))
def test_sendrecv_matches_oracle(name, proto, dtype):
    n, dst = MAPS[name]
    with context(n, dtype, 1 << 20):
        for count in (1, 7, 64, 4097, (256 << 10) // inputs.ELEM_BYTES[dtype]):
            x = inputs.normal(n, count, dtype, seed=count + n, iters=3, exclude_sentinel=True)
            assert np.array_equal(run(x, dtype, dst, proto, iters=3), expected(x, dtype, dst)), count


@pytest.mark.parametrize("proto", ["ll", "sentinel"])
def test_back_to_back_fresh_transfers_never_reuse_a_slot_early(proto):
    # 500 transfers with new data each: a slot rewritten before its receiver
    # consumed it would deliver a later transfer's data
    n, count, dtype = 8, 8192, "bf16"
    dst = [(r + 3) % n for r in range(n)]
    with context(n, dtype, 1 << 20):
        x = inputs.normal(n, count, dtype, seed=5, iters=500, exclude_sentinel=True)
        assert np.array_equal(run(x, dtype, dst, proto, iters=500, chunk=4096), expected(x, dtype, dst))


def test_sentinel_multi_chunk_and_slot_state():
    from test_gpu_protocol import staging_bytes
    n, count, dtype = 4, 100003, "fp16"  # 200 KB per transfer in 8 KiB chunks
    dst = [1, 2, 3, 0]
    with context(n, dtype, 1 << 20):
        x = inputs.normal(n, count, dtype, seed=9, iters=4, exclude_sentinel=True)
        assert np.array_equal(run(x, dtype, dst, "sentinel", iters=4, chunk=8192), expected(x, dtype, dst))
        for buf in staging_bytes("sentinel", n):
            assert np.all(buf == 0xFF)


def test_same_buffers_many_iterations_and_graph_replay():
    n, count, dtype = 8, 8192, "bf16"
    dst = [(r + 1) % n for r in range(n)]
    with context(n, dtype, 1 << 20):
        x = inputs.normal(n, count, dtype, seed=11)
        sends = [x[r].cuda() for r in range(n)]
        recvs = filled_outputs(n, count, dtype)
        llar.llar_sendrecv(sends, recvs, dst, count, "ll", 10000)
        torch.cuda.synchronize()
        want = expected(x[None], dtype, dst)[0]
        assert np.array_equal(np.stack([inputs.bits_of(o) for o in recvs]), want)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for proto in ("ll", "sentinel"):
                llar.llar_sendrecv(sends, recvs, dst, count, proto, 1, stream=s)
        for _ in range(3):
            for o in recvs:
                o.view(torch.int16).fill_(FILL[dtype])
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(np.stack([inputs.bits_of(o) for o in recvs]), want)
        assert llar.llar_get_status()[0] == llar.OK


def test_argument_errors():
    n, count, dtype = 4, 1024, "fp32"
    with context(n, dtype, 1 << 16):
        sends = [torch.zeros(count, device="cuda") for _ in range(n)]
        recvs = [torch.zeros(count, device="cuda") for _ in range(n)]
        for bad in ([0, 1, 2, 3], [1, 1, -1, -1], [4, -1, -1, -1], [-2, -1, -1, -1]):
            with pytest.raises(llar.LlarError) as ei:
                llar.llar_sendrecv(sends, recvs, bad, count, "ll")
            assert ei.value.code == llar.ERR_INVALID
        with pytest.raises(llar.LlarError) as ei:  # receive buffer is a send buffer
            llar.llar_sendrecv(sends, [sends[1], sends[0], recvs[2], recvs[3]], [1, 0, -1, -1], count, "ll")
        assert ei.value.code == llar.ERR_INVALID
        with pytest.raises(llar.LlarError) as ei:
            llar.llar_sendrecv(sends, recvs, [1, 0, 3, 2], count, "ll128")
        assert ei.value.code == llar.ERR_UNSUPPORTED
        with pytest.raises(llar.LlarError) as ei:
            llar.llar_sendrecv(sends, recvs, [1, 0, 3, 2], 1 << 20, "ll")
        assert ei.value.code == llar.ERR_TOO_LARGE
        # ranks outside the map may pass no buffers at all
        llar.llar_sendrecv([sends[0], None, None, None], [None, recvs[1], None, None], [1, -1, -1, -1], count, "ll")
        torch.cuda.synchronize()
        assert torch.equal(recvs[1], sends[0])


@pytest.mark.parametrize("proto", ["ll", "sentinel"])
def test_receiver_that_never_acknowledges_times_out(proto):
    # rank 1 is told to stay silent (it never signals): with a ring, the
    # waits around it run out; no fault, and reset recovers
    n, count, dtype = 4, 4096, "bf16"
    dst = [(r + 1) % n for r in range(n)]
    with context(n, dtype, 1 << 20, timeout_ns=20_000_000):
        x = inputs.normal(n, count, dtype, seed=4, iters=6, exclude_sentinel=True)
        llar.llar_debug_inject(1, "skip")
        sends = [x[:, r, :].contiguous().view(-1).cuda() for r in range(n)]
        recvs = filled_outputs(n, 6 * count, dtype)
        llar.llar_sendrecv(sends, recvs, dst, count, proto, 6, count, count)
        torch.cuda.synchronize()
        code, rank, cta, epoch = llar.llar_get_status()
        assert code == llar.ERR_TIMEOUT and 0 <= rank < n
        llar.llar_debug_inject(-1, "none")
        llar.llar_reset()
        assert np.array_equal(run(x, dtype, dst, proto, iters=6), expected(x, dtype, dst))


@pytest.mark.parametrize("name", ["ring8", "pairs4", "pipeline5"])
def test_auto_takes_the_direct_copy(name):
    # AUTO: the receiver's CTAs copy the sender's buffer (measured fastest at
    # every size on one GPU); a bit copy at every size, ragged and empty-tail included
    n, dst = MAPS[name]
    dtype = "bf16"
    with context(n, dtype, 2 << 20):
        for count in (1, 7, 8, 32768 + 3, 131072, (1 << 19) + 5):  # up to 1 MiB + 10 B per rank
            x = inputs.normal(1, n * count, dtype, seed=count + n).view(1, n, count)
            assert np.array_equal(run(x, dtype, dst, "auto"), expected(x, dtype, dst)), count
            assert llar.llar_last_launch()[0] == "fixed_oneshot"
