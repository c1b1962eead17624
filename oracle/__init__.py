"""CPU oracle for the barrier-free AllReduce (test infrastructure only).

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
and the product path never calls it.

The operation follows "Every Microsecond Matters: Achieving Near Speed-of-Light
Latency in GPU Collectives", Sec. III-A: an AllReduce-sum leaves in every rank's
output the element-wise sum of all ranks' inputs.  The same section names the
building blocks ReduceScatter, AllGather, Reduce and Broadcast, which are here
too, and the AllReduce with a residual-add epilogue.  See ``rra_oracle.c`` for the exact evaluation order and precision.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(closed forms, exact integer sums, an order-sensitive binary32 case,
``math.fsum`` error bounds, torch's bfloat16 conversion, hand-built layouts of
the data-movement collectives and the identity AllReduce = AllGather after
ReduceScatter checked element by element against an independent sum).
"""
from .oracle import (  # noqa: F401
    DTYPES,
    all_gather,
    allreduce,
    allreduce_mt,
    allreduce_residual,
    broadcast,
    build,
    f32_to_bf16,
    lib_path,
    reduce,
    reduce_scatter,
    reference_sum,
)
