"""What the signalling protocols fix about staging, from the pages alone.

TEST INFRASTRUCTURE (same import rule as the rest of `oracle/`).

Source for every item: "Every Microsecond Matters: Achieving Near
Speed-of-Light Latency in GPU Collectives", summary page, the four
techniques that remove the global memory barrier.

* LL (technique 1): an 8-byte flag and 8 bytes of data leave as one
  16-byte store; the receiver knows the data is there when it reads the
  flag. Effective bandwidth is halved and staging doubled.
* Sentinel (technique 2): the receive buffer is prefilled with a value
  that should not occur (the page's example is -NaN); the receiver polls
  until the value changes; the buffer has to be reset after every use; the
  data must never equal the sentinel.
* Two-shot LL128 (technique 4): threads work in groups of 8 on 128-byte
  lines; the group's first thread sets its own element to 1 as the flag;
  the line is complete when the flag has summed to N. Staging is about D/N
  for D bytes per round; the flag costs about 1.5% of bandwidth in FP16
  and about 3% in FP32.

Readings where the pages are silent: the sentinel is the all-ones pattern of
the element type (a NaN with the sign bit set, i.e. a -NaN, in all three
formats); the LL flag is a 64-bit call counter; the LL128 flag is the
line's first element, in the element type.
"""

import numpy as np

from . import fpformats as fp

LL_LINE_BYTES = 16
LL_PAYLOAD_BYTES = 8
LL128_LINE_BYTES = 128
LL128_GROUP_THREADS = 8


def ll_payload_fraction():
    """Share of an LL line that carries data (technique 1: bandwidth halved)."""
    return LL_PAYLOAD_BYTES / LL_LINE_BYTES


def ll_staging_bytes(payload_bytes):
    """Staging an LL transfer of `payload_bytes` needs (technique 1: doubled)."""
    return -(-payload_bytes // LL_PAYLOAD_BYTES) * LL_LINE_BYTES


def sentinel_bits(dtype):
    """The all-ones pattern of `dtype` used to prefill sentinel staging."""
    return {fp.FP32: 0xFFFFFFFF, fp.FP16: 0xFFFF, fp.BF16: 0xFFFF}[dtype]


def ll128_elems_per_line(dtype):
    return LL128_LINE_BYTES // fp.ELEM_BYTES[dtype]


def ll128_payload_elems(dtype):
    """Data elements per 128-byte line: all but the one flag element."""
    return ll128_elems_per_line(dtype) - 1


def ll128_overhead(dtype):
    """Bandwidth share taken by the flag element of each line."""
    return fp.ELEM_BYTES[dtype] / LL128_LINE_BYTES


def ll128_lines(elems, dtype):
    """Lines needed to carry `elems` data elements."""
    return -(-elems // ll128_payload_elems(dtype))


def ll128_round_staging_bytes(count, nranks, dtype):
    """Reduction staging one rank needs for one round of `count` elements.

    Each rank reduces one segment of ceil(count/N) elements, so its line
    staging is ceil(segment / payload) lines: about D/N bytes.
    """
    seg = -(-count // nranks)
    return ll128_lines(seg, dtype) * LL128_LINE_BYTES


def sentinel_refilled(staging_bits, dtype):
    """True if every element of a sentinel staging buffer is the sentinel."""
    return bool(np.all(np.asarray(staging_bits) == sentinel_bits(dtype)))


def ll128_lines_clear(staging_bytes):
    """True if every byte of an LL128 line staging buffer is zero."""
    return bool(np.all(np.asarray(staging_bytes) == 0))
