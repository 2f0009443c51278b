"""Seeded synthetic inputs shaped like tensor-parallel decode activations.

The one module that both the CUDA path's callers (tests, bench) and the
oracle's callers draw inputs from. It holds none of the AllReduce's
arithmetic: it draws random float32 numbers with torch's generator,
casts them to the buffer dtype with torch's own roundTiesToEven cast, and
exposes raw bit views.

Layout of every draw: [iters, N, count] (iteration-major, then rank, then
element), or [N, count] when iters is None.
"""

import numpy as np
import torch

TORCH_DTYPE = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}
ELEM_BYTES = {"fp32": 4, "fp16": 2, "bf16": 2}
# all-ones bit pattern that the sentinel protocol reserves
SENTINEL_BITS = {"fp32": 0xFFFFFFFF, "fp16": 0xFFFF, "bf16": 0xFFFF}


def _shape(nranks, count, iters):
    return (nranks, count) if iters is None else (iters, nranks, count)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def uniform(nranks, count, dtype, seed, lo=-1.0, hi=1.0, iters=None, device="cpu"):
    """Values uniform in [lo, hi)."""
    g = _gen(seed, device)
    x = torch.rand(_shape(nranks, count, iters), generator=g, device=device,
                   dtype=torch.float32)
    x = x * (hi - lo) + lo
    return x.to(TORCH_DTYPE[dtype])


def normal(nranks, count, dtype, seed, scale=1.0, iters=None, device="cpu",
           exclude_sentinel=False):
    """Values N(0, 1) * scale (activation-like)."""
    g = _gen(seed, device)
    x = torch.randn(_shape(nranks, count, iters), generator=g, device=device,
                    dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    x = x.to(TORCH_DTYPE[dtype])
    if exclude_sentinel:
        assert not bool((bits_of(x) == SENTINEL_BITS[dtype]).any()), \
            "draw hit the reserved sentinel pattern"
    return x


def integers(nranks, count, dtype, seed, lo, hi, iters=None, device="cpu"):
    """Integer values uniform in [lo, hi] (inclusive), stored in `dtype`."""
    g = _gen(seed, device)
    x = torch.randint(lo, hi + 1, _shape(nranks, count, iters), generator=g,
                      device=device, dtype=torch.int64)
    return x.to(TORCH_DTYPE[dtype])


def rank_ids(nranks, count, dtype, device="cpu"):
    """Every element of rank r equals r."""
    r = torch.arange(nranks, device=device, dtype=torch.float32)
    return r[:, None].expand(nranks, count).contiguous().to(TORCH_DTYPE[dtype])


def bits_of(t):
    """Raw bit pattern of a tensor as a numpy array (uint32 or uint16)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


def from_bits(bits, dtype):
    """numpy raw bits -> CPU torch tensor of `dtype` (no value conversion)."""
    bits = np.ascontiguousarray(bits)
    if dtype == "fp32":
        return torch.from_numpy(bits.view(np.int32).copy()).view(torch.float32)
    return torch.from_numpy(bits.view(np.int16).copy()).view(TORCH_DTYPE[dtype])


def linear_layer(nranks, m, k, h, dtype, seed, integer=False, device="cpu"):
    """Inputs of a row-parallel linear layer split over `nranks`: activations
    x [N, M, K] ~ N(0, 1) and weights w [N, K, H] ~ N(0, 1) / sqrt(N * K)
    (the scale of an initialised layer with N * K inputs), or, with
    integer=True, x in {-3..3} and w in {-2..2} (every partial sum exact)."""
    g = _gen(seed, device)
    if integer:
        x = torch.randint(-3, 4, (nranks, m, k), generator=g, device=device).to(torch.float32)
        w = torch.randint(-2, 3, (nranks, k, h), generator=g, device=device).to(torch.float32)
    else:
        x = torch.randn((nranks, m, k), generator=g, device=device, dtype=torch.float32)
        w = torch.randn((nranks, k, h), generator=g, device=device, dtype=torch.float32)
        w = w * float((nranks * k) ** -0.5)
    return x.to(TORCH_DTYPE[dtype]), w.to(TORCH_DTYPE[dtype])
