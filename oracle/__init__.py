"""CPU oracle for the sum AllReduce and its signalling protocols.

TEST INFRASTRUCTURE, not product code. Only `tests/`,
`__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may import,
call or execute anything in this package. The CUDA library in
`tp_allreduce_persistent_b300/` shares no code with it, never imports it,
and fails loudly instead of falling back to it.

Modules:
  fpformats     bit-level fp32/fp16/bf16 decode, roundTiesToEven encode, ulp
  allreduce     one-shot, two-shot (ReduceScatter + AllGather), chained
                sequences, and the tolerance for order-free atomic paths
  atomic_model  a per-order model of the atomic accumulation (pins the
                tolerance only)
  protocol      what the signalling protocols leave behind in staging
                (sentinel refill, zeroed LL128 lines, LL line layout sizes)

Every function is pinned by `-m "not gpu"` tests against closed forms,
invariants, exact rational sums, hand-worked IEEE cases in tests/golden/
and library conversions; none is marked "parity unpinned".
"""
