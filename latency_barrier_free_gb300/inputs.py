"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module only draws random numbers and lays them out; it holds none of the
AllReduce arithmetic.  Every generator returns one numpy array per virtual
rank, on the host, so that the oracle and the GPU path see the same bytes.

Seeds follow ``seed = 1000 * workload + iteration``; extra integer tags (size
index, dtype code) are mixed in through ``numpy.random.SeedSequence`` so that
different message sizes of one workload draw independent streams.

Workloads (the shapes and value distributions of the pages' evaluation, see
"Every Microsecond Matters", Sec. I and the microbenchmark figures):
  1  N=2, 32 binary32 integers uniform in [-8, 8] per rank, fresh per call
  2  N=4, 128 B .. 1 MiB per rank (powers of two), binary32/bfloat16 N(0, 1)
  3  N=8, bfloat16 N(0, 1) activations of shape [batch, 8192]
  4  N=64, binary32 N(0, 1), 1 KiB .. 256 KiB per rank
  5  N=8, binary32/binary64 uniform(-1, 1), 4 MiB / 64 MiB / 512 MiB per rank
"""
from __future__ import annotations

import numpy as np

DT_CODE = {"fp32": 0, "bf16": 1, "fp64": 2}
ELEM_BYTES = {"fp32": 4, "bf16": 2, "fp64": 8}
NP_STORAGE = {"fp32": np.float32, "bf16": np.uint16, "fp64": np.float64}

# Workload definitions (sizes are bytes per rank).
W2_SIZES = [1 << k for k in range(7, 21)]             # 128 B .. 1 MiB, 14 sizes
W3_BATCHES = [1, 4, 16, 64]                            # [batch, 8192] bf16
W3_HIDDEN = 8192
W3_CALLS_PER_TOKEN = 160                               # 80 layers x 2 AllReduces
W4_SIZES = [1 << k for k in range(10, 19)]            # 1 KiB .. 256 KiB, 9 sizes
W4_NSWEEP = [2, 4, 8, 16, 32, 64]
W5_SIZES = [4 << 20, 64 << 20, 512 << 20]


def rng(workload: int, iteration: int = 0, *tags: int) -> np.random.Generator:
    seed = np.random.SeedSequence([1000 * int(workload) + int(iteration)] + [int(t) for t in tags])
    return np.random.Generator(np.random.PCG64(seed))


def _bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Take the upper 16 bits of binary32 samples (truncation, no rounding):
    a bfloat16 bit pattern with the same sign/exponent as the sample."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def normal(g: np.random.Generator, nranks: int, count: int, dtype: str):
    out = []
    for _ in range(nranks):
        if dtype == "fp64":
            out.append(g.standard_normal(count, dtype=np.float64))
        else:
            x = g.standard_normal(count, dtype=np.float32)
            out.append(x if dtype == "fp32" else _bf16_bits_from_f32(x))
    return out


def uniform(g: np.random.Generator, nranks: int, count: int, dtype: str, lo=-1.0, hi=1.0):
    out = []
    for _ in range(nranks):
        if dtype == "fp64":
            out.append(lo + (hi - lo) * g.random(count, dtype=np.float64))
        else:
            x = (np.float32(lo) + np.float32(hi - lo) * g.random(count, dtype=np.float32)).astype(np.float32)
            out.append(x if dtype == "fp32" else _bf16_bits_from_f32(x))
    return out


def small_integers(g: np.random.Generator, nranks: int, count: int, dtype: str, lo=-8, hi=8):
    """Integers uniform in [lo, hi], stored in the floating type (exact)."""
    out = []
    for _ in range(nranks):
        k = g.integers(lo, hi + 1, size=count, dtype=np.int64)
        if dtype == "fp64":
            out.append(k.astype(np.float64))
        elif dtype == "fp32":
            out.append(k.astype(np.float32))
        else:
            out.append(_bf16_bits_from_f32(k.astype(np.float32)))  # |k| <= 256 is exact in bf16
    return out


def rank_plus_one(nranks: int, count: int, dtype: str):
    """Rank r filled with the value r + 1 (exact in every dtype for r < 256)."""
    out = []
    for r in range(nranks):
        v = np.full(count, r + 1, dtype=np.float32 if dtype != "fp64" else np.float64)
        out.append(v if dtype != "bf16" else _bf16_bits_from_f32(v))
    return out


def workload1(iteration: int):
    """N=2, 32 binary32 integers in [-8, 8]; a fresh draw per call."""
    return small_integers(rng(1, iteration), 2, 32, "fp32")


def workload2(size_bytes: int, dtype: str, iteration: int = 0):
    n = size_bytes // ELEM_BYTES[dtype]
    return normal(rng(2, iteration, size_bytes, DT_CODE[dtype]), 4, n, dtype)


def workload3(batch: int, iteration: int = 0):
    return normal(rng(3, iteration, batch), 8, batch * W3_HIDDEN, "bf16")


def workload4(size_bytes: int, nranks: int = 64, iteration: int = 0):
    return normal(rng(4, iteration, size_bytes, nranks), nranks, size_bytes // 4, "fp32")


def workload5(size_bytes: int, dtype: str, iteration: int = 0):
    n = size_bytes // ELEM_BYTES[dtype]
    return uniform(rng(5, iteration, size_bytes, DT_CODE[dtype]), 8, n, dtype)
