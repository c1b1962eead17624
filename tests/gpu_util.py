"""Helpers for the GPU tests: move seeded host inputs to the device, read
outputs back, and compare with the oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np

import oracle

TORCH_DT = {"fp32": "float32", "bf16": "bfloat16", "fp64": "float64"}
ELEM = {"fp32": 4, "bf16": 2, "fp64": 8}
FIXED_ORDER = ("oneshot_ll", "oneshot_sentinel", "twoshot_dbuf", "oneshot_barrier", "twoshot_direct",
               "oneshot_cluster", "twoshot_cluster", "twoshot_barrier")
ALGOS = ("oneshot_ll", "oneshot_sentinel", "twoshot_dbuf", "ll128_atomic", "twoshot_direct")
CLUSTER = ("oneshot_cluster", "twoshot_cluster")  # N <= 16


def to_device(arrs, dtype: str):
    import torch

    out = []
    for a in arrs:
        if dtype == "bf16":
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a).copy())
        out.append(t.cuda())
    return out


def to_host(tensors, dtype: str):
    import torch

    out = []
    for t in tensors:
        if dtype == "bf16":
            out.append(t.view(torch.int16).cpu().numpy().view(np.uint16))
        else:
            out.append(t.cpu().numpy())
    return out


def poison_like(tensors):
    """Fresh output buffers filled with a poison pattern (0x7F bytes): a value
    that no correct result of these inputs has."""
    import torch

    outs = []
    for t in tensors:
        o = torch.empty_like(t)
        o.view(torch.uint8).fill_(0x7F)
        outs.append(o)
    return outs


def bits(a: np.ndarray) -> np.ndarray:
    return a.view({2: np.uint16, 4: np.uint32, 8: np.uint64}[a.dtype.itemsize])


def as_float64(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def check_identical_ranks(got):
    for g in got[1:]:
        assert np.array_equal(bits(g), bits(got[0])), "ranks received different bit patterns"


def check_against_oracle(sends_np, got, dtype: str, algo: str):
    """Fixed-order algorithms: bit-exact against the oracle.  LL128-atomic:
    |err| <= N 2^-p sum|x| (+ N 2^-126 for binary32 flush-to-zero atomics,
    + one bfloat16 ulp of the result for bfloat16)."""
    check_identical_ranks(got)
    n = len(sends_np)
    if algo in FIXED_ORDER:
        expect = oracle.allreduce(sends_np, dtype)
        bad = np.nonzero(bits(got[0]) != bits(expect[0]))[0]
        assert bad.size == 0, "%s %s: %d mismatches, first at %d: got %r expect %r" % (
            algo, dtype, bad.size, bad[0], got[0][bad[0]], expect[0][bad[0]])
        return
    ref, absum = oracle.reference_sum(sends_np, dtype)
    g = as_float64(got[0], dtype)
    if dtype == "fp64":
        tol = n * 2.0 ** -52 * absum
    else:
        tol = n * 2.0 ** -23 * absum + n * 2.0 ** -126
        if dtype == "bf16":
            mag = np.maximum(np.abs(ref), 2.0 ** -126)
            tol = tol + 2.0 ** (np.floor(np.log2(mag)) - 7)
    err = np.abs(g - ref)
    bad = np.nonzero(~(err <= tol))[0]
    assert bad.size == 0, "%s %s: %d out of bound, first at %d: got %r ref %r tol %r" % (
        algo, dtype, bad.size, bad[0], g[bad[0]], ref[bad[0]], tol[bad[0]])
