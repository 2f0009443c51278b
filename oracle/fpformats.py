"""Bit-level IEEE formats used by the oracle: fp32, fp16 (binary16), bf16.

TEST INFRASTRUCTURE. Only `tests/`, `__graft_entry__.smoke()` and the CPU
baseline leg of `bench.py` may import this package; the CUDA library never
does, and this package imports nothing from it.

Values travel as raw bit patterns in numpy arrays: uint32 for fp32, uint16
for fp16 and bf16. The three formats are the ones the low-latency
collectives support ("Every Microsecond Matters: Achieving Near
Speed-of-Light Latency in GPU Collectives", summary page, technique 4,
two-shot LL128: add only, FP32/FP16/BF16 only).

Rounding follows IEEE 754 roundTiesToEven ("round to nearest, ties to
even"), written out here from that definition for bf16; fp16 uses numpy's
float32 -> float16 cast, which is an IEEE roundTiesToEven conversion
(library primitive; pinned against torch's CPU cast in tests/).
"""

import numpy as np

FP32, FP16, BF16 = "fp32", "fp16", "bf16"
DTYPES = (FP32, FP16, BF16)

# precision p (significand bits incl. the hidden bit) and minimum normal
# exponent emin of each format (IEEE 754 table 3.2 for binary32/binary16;
# bfloat16 keeps binary32's exponent range with an 8-bit significand).
PRECISION = {FP32: 24, FP16: 11, BF16: 8}
EMIN = {FP32: -126, FP16: -14, BF16: -126}
ELEM_BYTES = {FP32: 4, FP16: 2, BF16: 2}
BITS_DTYPE = {FP32: np.uint32, FP16: np.uint16, BF16: np.uint16}


def decode(bits, dtype):
    """Raw bits -> float32 values (exact: every fp16/bf16 value is a float32)."""
    bits = np.asarray(bits)
    if dtype == FP32:
        return bits.astype(np.uint32).view(np.float32)
    if dtype == FP16:
        return bits.astype(np.uint16).view(np.float16).astype(np.float32)
    if dtype == BF16:
        # a bf16 is the upper half of the float32 with the same value
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    raise ValueError(dtype)


def _bf16_rne(f32):
    """float32 -> bf16 bits, roundTiesToEven, from the definition.

    The bf16 value keeps the upper 16 bits of the float32; the dropped lower
    16 bits are compared with half a unit in the last kept place (0x8000):
    above -> round up, below -> truncate, equal -> round to the even kept
    pattern. A carry out of the significand moves into the exponent, which
    is exactly IEEE's step to the next binade and, from the largest finite
    value, to infinity. NaN maps to a quiet NaN with the same sign.
    """
    u = np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32)
    upper = (u >> np.uint32(16)).astype(np.uint32)
    lower = u & np.uint32(0xFFFF)
    half = np.uint32(0x8000)
    round_up = (lower > half) | ((lower == half) & ((upper & np.uint32(1)) == 1))
    out = upper + round_up.astype(np.uint32)
    is_nan = ((u & np.uint32(0x7F800000)) == np.uint32(0x7F800000)) & (
        (u & np.uint32(0x007FFFFF)) != 0)
    out = np.where(is_nan, (upper & np.uint32(0x8000)) | np.uint32(0x7FC0), out)
    return out.astype(np.uint16)


def encode_rne(f32, dtype):
    """float32 values -> raw bits of `dtype`, one roundTiesToEven rounding."""
    f32 = np.asarray(f32, dtype=np.float32)
    if dtype == FP32:
        return f32.view(np.uint32).copy()
    if dtype == FP16:
        with np.errstate(over="ignore", invalid="ignore"):
            return f32.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        return _bf16_rne(f32)
    raise ValueError(dtype)


def encode_rne64(x64, dtype):
    """float64 values -> raw bits of `dtype`, ONE roundTiesToEven rounding.

    For values that are not float32 numbers (an exact float64 dot product)
    rounding through float32 first could round twice. fp32 and fp16 use
    numpy's direct float64 casts (IEEE conversions, roundTiesToEven); bf16
    is written out from the definition: the value's spacing in bf16 is
    2^(max(floor(log2|x|), emin) - p + 1); x / spacing is rounded to the
    nearest integer, ties to even (np.rint), and scaled back, which is then
    a bf16 number, exact in float32. Magnitudes at or beyond the largest
    finite value plus half its spacing become infinities.
    """
    x = np.asarray(x64, dtype=np.float64)
    if dtype == FP32:
        with np.errstate(over="ignore", invalid="ignore"):
            return x.astype(np.float32).view(np.uint32)
    if dtype == FP16:
        with np.errstate(over="ignore", invalid="ignore"):
            return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        p, emin = PRECISION[BF16], EMIN[BF16]
        ax = np.abs(x)
        with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
            _, e2 = np.frexp(ax)
            expo = np.maximum(np.where(ax > 0, e2 - 1, emin), emin)
            spacing = np.ldexp(1.0, (expo - p + 1).astype(np.int64))
            r = np.rint(x / spacing) * spacing
            big = np.abs(r) > max_finite(BF16)
            r = np.where(big, np.copysign(np.inf, x), r)
            r = np.where(np.isfinite(x), r, x)
        return _bf16_rne(r.astype(np.float32))
    raise ValueError(dtype)


def is_nan_bits(bits, dtype):
    """True where the bit pattern is a NaN of `dtype`."""
    return np.isnan(decode(bits, dtype))


def ulp(x, dtype):
    """Unit in the last place of |x| in `dtype`, as float64.

    ulp(x) = 2^(max(floor(log2|x|), emin) - p + 1); for |x| below the
    smallest normal (and for 0) this is the subnormal spacing 2^(emin-p+1).
    Infinite x gives +inf.
    """
    x = np.abs(np.asarray(x, dtype=np.float64))
    p, emin = PRECISION[dtype], EMIN[dtype]
    with np.errstate(divide="ignore"):
        _, e2 = np.frexp(x)  # x = m * 2^e2 with m in [0.5, 1)
    expo = np.where(x > 0, e2 - 1, emin)  # floor(log2 x)
    expo = np.maximum(expo, emin)
    out = np.ldexp(1.0, (expo - p + 1).astype(np.int64))
    return np.where(np.isinf(x), np.inf, out)


def max_finite(dtype):
    """Largest finite value of `dtype` (float64)."""
    p = PRECISION[dtype]
    emax = {FP32: 127, FP16: 15, BF16: 127}[dtype]
    return (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
