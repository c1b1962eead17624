"""Run one AllReduce configuration a few times (for profiling one kernel).

    python -m latency_barrier_free_gb300.run_case ALGO NRANKS BYTES_PER_RANK DTYPE REPS [attr=value ...]

e.g. ``python -m latency_barrier_free_gb300.run_case twoshot_dbuf 8 67108864 fp32 4 twoshot_chunk=1048576``.
Inputs are seeded uniform(-1, 1) values generated on the device (no result
check: this is a load generator for profilers).  Exits non-zero if the device
reports an error.
"""
from __future__ import annotations

import sys


def main(argv):
    import torch

    from latency_barrier_free_gb300 import build_ext, rra

    if len(argv) < 5:
        print(__doc__)
        return 2
    algo, n, size, dtype, reps = argv[0], int(argv[1]), int(argv[2]), argv[3], int(argv[4])
    attrs = dict(a.split("=", 1) for a in argv[5:])
    build_ext.build()
    tdt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp64": torch.float64}[dtype]
    es = {"fp32": 4, "bf16": 2, "fp64": 8}[dtype]
    count = size // es
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    xs = [(torch.rand(count, device="cuda", generator=g) * 2 - 1).to(tdt) for _ in range(n)]
    ys = [torch.empty_like(x) for x in xs]
    with rra.Comm(n, size) as c:
        for k, v in attrs.items():
            c.set_attr(k, int(v))
        grid, steps = c.plan_call(count, dtype, algo)
        print("grid %d CTAs, %d steps" % (grid, steps), flush=True)
        for _ in range(reps):
            c.allreduce(xs, ys, algo)
        torch.cuda.synchronize()
        st = c.status()
        print("status", rra.STATUS_NAMES.get(st[0]), flush=True)
        return 0 if st[0] == rra.OK else 1


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
