"""ctypes front end of the C oracle (test infrastructure only).

Arrays are numpy arrays on the host: float32 for binary32, uint16 bit patterns
for bfloat16, float64 for binary64.  Nothing here touches a GPU.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rra_oracle.c")
_LIB = os.path.join(_HERE, "librra_oracle.so")

# dtype name -> (oracle code, numpy storage dtype)
DTYPES = {
    "fp32": (0, np.float32),
    "bf16": (1, np.uint16),
    "fp64": (2, np.float64),
}

_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-Wall", "-Wextra", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vpp = ctypes.POINTER(ctypes.c_void_p)
            lib.rra_oracle_allreduce.argtypes = [ctypes.c_int, vpp, vpp, ctypes.c_size_t, ctypes.c_int]
            lib.rra_oracle_allreduce.restype = ctypes.c_int
            lib.rra_oracle_allreduce_mt.argtypes = [ctypes.c_int, vpp, vpp, ctypes.c_size_t,
                                                    ctypes.c_int, ctypes.c_int]
            lib.rra_oracle_allreduce_mt.restype = ctypes.c_int
            lib.rra_oracle_reference_sum.argtypes = [ctypes.c_int, vpp, ctypes.c_size_t, ctypes.c_int,
                                                     ctypes.c_void_p, ctypes.c_void_p]
            lib.rra_oracle_reference_sum.restype = ctypes.c_int
            lib.rra_oracle_f32_to_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]
            lib.rra_oracle_f32_to_bf16_array.restype = None
            for name in ("rra_oracle_reduce_scatter", "rra_oracle_all_gather"):
                getattr(lib, name).argtypes = [ctypes.c_int, vpp, vpp, ctypes.c_size_t, ctypes.c_int]
                getattr(lib, name).restype = ctypes.c_int
            lib.rra_oracle_allreduce_residual.argtypes = [ctypes.c_int, vpp, vpp, vpp, ctypes.c_size_t,
                                                          ctypes.c_int]
            lib.rra_oracle_allreduce_residual.restype = ctypes.c_int
            for name in ("rra_oracle_broadcast", "rra_oracle_reduce"):
                getattr(lib, name).argtypes = [ctypes.c_int, ctypes.c_int, vpp, vpp, ctypes.c_size_t,
                                               ctypes.c_int]
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptrs(arrays):
    arr = (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def _check_inputs(sends, dtype):
    code, np_dt = DTYPES[dtype]
    if len(sends) < 1:
        raise ValueError("need at least one rank")
    count = sends[0].size
    for s in sends:
        if s.dtype != np_dt or s.size != count or not s.flags.c_contiguous:
            raise ValueError("all ranks need contiguous %s arrays of equal size" % np.dtype(np_dt))
    return code, np_dt, count


def allreduce(sends, dtype: str, recvs=None):
    """Fixed-rank-order AllReduce-sum; returns the list of N outputs."""
    lib = _load()
    code, np_dt, count = _check_inputs(sends, dtype)
    if recvs is None:
        recvs = [np.empty(count, dtype=np_dt) for _ in sends]
    sp, keep_s = _ptrs(sends)
    rp, keep_r = _ptrs(recvs)
    rc = lib.rra_oracle_allreduce(len(sends), sp, rp, count, code)
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    del keep_s, keep_r
    return recvs


def allreduce_mt(sends, dtype: str, nthreads: int, recvs=None):
    """Same result as allreduce(); the element range is split over threads."""
    lib = _load()
    code, np_dt, count = _check_inputs(sends, dtype)
    if recvs is None:
        recvs = [np.empty(count, dtype=np_dt) for _ in sends]
    sp, keep_s = _ptrs(sends)
    rp, keep_r = _ptrs(recvs)
    rc = lib.rra_oracle_allreduce_mt(len(sends), sp, rp, count, code, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    del keep_s, keep_r
    return recvs


def reference_sum(sends, dtype: str):
    """(sum, abs_sum) per element, accumulated in long double, as float64."""
    lib = _load()
    code, _, count = _check_inputs(sends, dtype)
    out_sum = np.empty(count, dtype=np.float64)
    out_abs = np.empty(count, dtype=np.float64)
    sp, keep_s = _ptrs(sends)
    rc = lib.rra_oracle_reference_sum(len(sends), sp, count, code,
                                      out_sum.ctypes.data, out_abs.ctypes.data)
    if rc != 0:
        raise RuntimeError("oracle rejected its arguments")
    del keep_s
    return out_sum, out_abs


def f32_to_bf16(x) -> np.ndarray:
    """Round binary32 values to bfloat16 bit patterns (nearest, ties to even)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.rra_oracle_f32_to_bf16_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def _run(fn, *args):
    if fn(*args) != 0:
        raise RuntimeError("oracle rejected its arguments")


def reduce_scatter(sends, dtype: str):
    """ReduceScatter-sum: sends[p] holds N*count elements; returns N outputs
    of count elements, output r = rank-order sum of the inputs' block r."""
    lib = _load()
    code, np_dt, total = _check_inputs(sends, dtype)
    n = len(sends)
    if total % n:
        raise ValueError("each input must hold N * count elements")
    count = total // n
    recvs = [np.empty(count, dtype=np_dt) for _ in sends]
    sp, keep_s = _ptrs(sends)
    rp, keep_r = _ptrs(recvs)
    _run(lib.rra_oracle_reduce_scatter, n, sp, rp, count, code)
    del keep_s, keep_r
    return recvs


def all_gather(sends, dtype: str):
    """AllGather: every output is the concatenation of the N inputs in rank order."""
    lib = _load()
    code, np_dt, count = _check_inputs(sends, dtype)
    n = len(sends)
    recvs = [np.empty(n * count, dtype=np_dt) for _ in sends]
    sp, keep_s = _ptrs(sends)
    rp, keep_r = _ptrs(recvs)
    _run(lib.rra_oracle_all_gather, n, sp, rp, count, code)
    del keep_s, keep_r
    return recvs


def broadcast(sends, dtype: str, root: int):
    """Broadcast: every output is a copy of sends[root]."""
    lib = _load()
    code, np_dt, count = _check_inputs(sends, dtype)
    recvs = [np.empty(count, dtype=np_dt) for _ in sends]
    sp, keep_s = _ptrs(sends)
    rp, keep_r = _ptrs(recvs)
    _run(lib.rra_oracle_broadcast, len(sends), int(root), sp, rp, count, code)
    del keep_s, keep_r
    return recvs


def reduce(sends, dtype: str, root: int, recvs=None):
    """Reduce-sum to `root`: recvs[root] = rank-order sum; other outputs are
    left as passed (fresh zero arrays when recvs is None)."""
    lib = _load()
    code, np_dt, count = _check_inputs(sends, dtype)
    if recvs is None:
        recvs = [np.zeros(count, dtype=np_dt) for _ in sends]
    sp, keep_s = _ptrs(sends)
    rp, keep_r = _ptrs(recvs)
    _run(lib.rra_oracle_reduce, len(sends), int(root), sp, rp, count, code)
    del keep_s, keep_r
    return recvs


def allreduce_residual(sends, residuals, dtype: str):
    """AllReduce-sum with each rank's residual added to the running value
    before the one rounding: recv[r] = round(sum_p x_p + res[r])."""
    lib = _load()
    code, np_dt, count = _check_inputs(sends, dtype)
    _check_inputs(residuals, dtype)
    if len(residuals) != len(sends) or residuals[0].size != count:
        raise ValueError("one residual of the inputs' size per rank")
    recvs = [np.empty(count, dtype=np_dt) for _ in sends]
    sp, keep_s = _ptrs(sends)
    qp, keep_q = _ptrs(residuals)
    rp, keep_r = _ptrs(recvs)
    _run(lib.rra_oracle_allreduce_residual, len(sends), sp, qp, rp, count, code)
    del keep_s, keep_q, keep_r
    return recvs
