"""CPU oracle for the tensor-parallel row-parallel linear layer whose
AllReduce is fused into the GEMV epilogue.

TEST INFRASTRUCTURE. Only `tests/`, `__graft_entry__.smoke()` and the CPU
baseline leg of `bench.py` may import this module; the CUDA library never
does.

What is computed ("zcube network architecture for LLM inference", section
"Why does Tensor Parallel affect every token": each rank holds a slice of
the layer's input dimension, computes a partial output, and the layer ends
in the sum of the partial outputs over the ranks; "TP All-Reduce and TTFT",
section 2.1, the same per-layer AllReduce):

    p_r = round_dtype( x_r @ w_r )          x_r: [M, K], w_r: [K, H]
    out = AllReduce(p_0 .. p_{N-1})         (rank order, float32, one rounding)

Reading where the pages are silent: the partial is rounded to the buffer's
element type before the AllReduce, as an unfused pipeline stores it; here
the dot product is exact (float64, exact for the products of fp16/bf16 and
fp32 inputs up to the final float64 additions) and rounded once.

The GPU computes each dot product in float32 (fused multiply-adds) with a
split of K the definition does not fix, so its partials may differ from these by the
rounding errors of that computation; `linear_tolerance` bounds the
difference that reaches the output. Inputs whose every partial sum is an
exact float32 number (small integers) give identical results.

Arrays are raw bit patterns (see `fpformats`): x [N, M, K], w [N, K, H].
"""

import numpy as np

from . import allreduce as ar
from . import fpformats as fp

U32 = 2.0 ** -24  # unit roundoff of float32 (round to nearest)
# relative error bound of one float32 addition whatever its rounding: the
# tensor cores accumulate in float32 without stating the rounding of each
# addition (round-toward-zero errs by up to 2^-23)
U_ADD = 2.0 ** -23


def _values(bits, dtype):
    return fp.decode(bits, dtype).astype(np.float64)


def linear_partials(x_bits, w_bits, dtype):
    """p_r = roundTiesToEven(x_r @ w_r) per rank: [N, M, H] bits."""
    x = _values(x_bits, dtype)
    w = _values(w_bits, dtype)
    return fp.encode_rne64(np.matmul(x, w), dtype)


def linear_allreduce(x_bits, w_bits, dtype):
    """Every rank's output: the rank-order AllReduce of the partials, [N, M, H]."""
    p = linear_partials(x_bits, w_bits, dtype)
    n, m, h = p.shape
    return ar.allreduce(p.reshape(n, m * h), dtype).reshape(n, m, h)


def linear_tolerance(x_bits, w_bits, dtype, unit=U_ADD):
    """Per-element bound on |GPU output - linear_allreduce| ([M, H] float64).

    With A_r = sum_k |x_r[m,k] w_r[k,h]| and gamma = K u / (1 - K u): any
    float32 evaluation of a K-term dot product (products rounded and
    added, fused multiply-adds, or tensor-core accumulation; additions in
    any order) is within gamma * A_r of the exact value (Higham, Accuracy
    and Stability of Numerical Algorithms, ch. 3: every term goes through at
    most K roundings, each a relative error of at most u). u = `unit`:
    2^-23 by default, which also covers additions rounded toward zero (the
    tensor cores do not state their rounding); 2^-24 for round to nearest.
    Rounding both to the element type adds at most one ulp at (1 + gamma) A_r,
    so the partials differ by d_r = gamma A_r + ulp((1 + gamma) A_r). The two
    float32 rank-order sums then differ by at most sum_r d_r plus the error
    of each sum, (N - 1) u times its magnitude bound S = sum_r ((1 + gamma)
    A_r + d_r), and the final roundings by one ulp(S).
    """
    x = np.abs(_values(x_bits, dtype))
    w = np.abs(_values(w_bits, dtype))
    n, _, k = x.shape
    a = np.matmul(x, w)  # [N, M, H]
    gamma = k * unit / (1.0 - k * unit)
    d = gamma * a + fp.ulp((1.0 + gamma) * a, dtype)
    s = np.sum((1.0 + gamma) * a + d, axis=0)
    return np.sum(d, axis=0) + 2.0 * (n - 1) * U32 * s + fp.ulp(s, dtype)


def compare_linear(got_bits, x_bits, w_bits, dtype, unit=U_ADD):
    """(ok, max error in tolerances) of a GPU result [N, M, H] against the oracle."""
    want = _values(linear_allreduce(x_bits, w_bits, dtype), dtype)
    got = _values(got_bits, dtype)
    tol = linear_tolerance(x_bits, w_bits, dtype, unit)
    with np.errstate(invalid="ignore"):
        err = np.abs(got - want)
    ok = bool(np.all(np.isfinite(got)) and np.all(err <= tol))
    return ok, float(np.max(err / tol)) if err.size else 0.0
