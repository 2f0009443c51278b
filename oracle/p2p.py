"""CPU oracle for point-to-point transfers between virtual ranks.

TEST INFRASTRUCTURE. Only `tests/`, `__graft_entry__.smoke()` and the CPU
baseline leg of `bench.py` may import this module; the CUDA library never
does.

A pipeline-parallel stage hand-off moves one stage's activations to the
next stage unchanged ("Every Microsecond Matters", summary page: the same
low-latency signalling serves point-to-point transfers; "zcube network
architecture for LLM inference": pipeline stages pass activations from
one to the next). The result is a bit copy: the receiver of rank r's
buffer holds exactly rank r's bits.
"""

import numpy as np


def sources(dst):
    """src[q] = the rank that sends to q, or -1 (dst[r] = -1: r sends nothing)."""
    n = len(dst)
    src = [-1] * n
    for r, d in enumerate(dst):
        if d < 0:
            continue
        if d == r or d >= n or src[d] != -1:
            raise ValueError("invalid destination map")
        src[d] = r
    return src


def sendrecv(send_bits, dst, fill):
    """recv[dst[r]] = send[r]; ranks that receive nothing keep `fill` rows.

    send_bits: [N, count] raw bits. Returns [N, count]."""
    send_bits = np.asarray(send_bits)
    out = np.array(fill, copy=True)
    for q, r in enumerate(sources(dst)):
        if r >= 0:
            out[q] = send_bits[r]
    return out
