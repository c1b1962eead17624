"""Python binding of the rra C ABI (include/rra.h, include/rra_probe.h).

Argument marshalling only: every step of the AllReduce runs in librra.so's
CUDA kernels.  If librra.so cannot be loaded, every call raises; there is no
fallback.  Torch is used for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librra.so")

OK = 0
STATUS_NAMES = {
    0: "RRA_OK", 1: "RRA_ERR_INVALID_ARG", 2: "RRA_ERR_CUDA", 3: "RRA_ERR_OOM",
    4: "RRA_ERR_NOT_CORESIDENT", 5: "RRA_ERR_TIMEOUT", 6: "RRA_ERR_POISONED",
}
ERR_INVALID_ARG, ERR_CUDA, ERR_OOM, ERR_NOT_CORESIDENT, ERR_TIMEOUT, ERR_POISONED = range(1, 7)

DTYPES = {"fp32": 0, "bf16": 1, "fp64": 2}
ALGOS = {"oneshot_ll": 0, "oneshot_sentinel": 1, "twoshot_dbuf": 2, "ll128_atomic": 3,
         "oneshot_barrier": 4, "twoshot_direct": 5, "auto": 6, "oneshot_cluster": 7,
         "twoshot_cluster": 8, "twoshot_barrier": 9}
ALGO_NAMES = {v: k for k, v in ALGOS.items()}
BARRIER_FREE = ("oneshot_ll", "oneshot_sentinel", "twoshot_dbuf", "ll128_atomic", "twoshot_direct")
ATTRS = {"ctas_per_rank": 0, "poll_timeout_ms": 1, "threads": 2, "twoshot_chunk": 3,
         "ll128_chunk": 4, "oneshot_chunk": 5, "oneshot_wide": 6, "cooperative": 7, "pdl": 8,
         "cluster_slice": 9, "cluster_pipe": 10, "host_zero_copy": 11,
         "coll_split": 12, "cluster_tma": 13}
MAX_RANKS = 64

# Exported symbols, in declaration order of the public headers.
SYMBOLS = [
    "rra_comm_create", "rra_allreduce", "rra_allreduce_host", "rra_host_device_ptrs", "rra_allreduce_mapped",
    "rra_comm_status", "rra_comm_error_site", "rra_comm_last_kernel", "rra_comm_reset",
    "rra_comm_destroy", "rra_comm_set_attr", "rra_comm_get_attr", "rra_comm_layout", "rra_plan_layout",
    "rra_comm_plan_kernel", "rra_select_algo", "rra_comm_plan_call", "rra_comm_max_coresident", "rra_comm_set_timing", "rra_comm_set_trace",
    "rra_comm_inject_drop",
    "rra_comm_barrier_latency", "rra_comm_get_epoch", "rra_comm_set_epoch", "rra_status_string",
    "rra_version",
    "rra_probe_l2_chase", "rra_probe_pingpong", "rra_probe_dsmem_pingpong", "rra_probe_empty_kernel",
    "rra_probe_launch_shape",
    "rra_probe_sm_count", "rra_probe_host_link", "rra_probe_launch_chain",
    "rra_allreduce_static",
    "rra_reduce_scatter", "rra_all_gather", "rra_broadcast", "rra_reduce",
    "rra_allreduce_residual",
]

# The collectives besides AllReduce (all through distributed shared memory).
COLLECTIVES = ("reduce_scatter", "all_gather", "broadcast", "reduce")


class Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) if n != "nranks" else (n, ctypes.c_int) for n in (
        "nranks", "max_bytes", "ll_chunk", "ll_bytes", "os_chunk", "os_bytes", "ts_part", "ts_bytes",
        "la_part", "la_bytes", "window_stride", "ctrl_bytes", "total_bytes", "bf_bytes", "bd_chunk",
        "bd_bytes")]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class RraError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        name = STATUS_NAMES.get(self.status, str(status))
        super().__init__("%s%s: %s" % (what + ": " if what else "", name, status_string(self.status)))


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load librra.so (once).  Raises if it is missing: build it first with
    latency_barrier_free_gb300.build_ext.build()."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError("librra.so not found at %s; run latency_barrier_free_gb300.build_ext.build()" % path)
        lib = ctypes.CDLL(path)
        vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64
        pp = ctypes.POINTER(ctypes.c_void_p)
        ip = ctypes.POINTER(ctypes.c_int)
        sig = {
            "rra_comm_create": ([i32, sz, pp], i32),
            "rra_allreduce": ([vp, pp, pp, sz, i32, i32, vp], i32),
            "rra_allreduce_host": ([vp, pp, pp, sz, i32, i32, vp], i32),
            "rra_host_device_ptrs": ([i32, pp, pp], i32),
            "rra_allreduce_mapped": ([vp, pp, pp, sz, i32, i32, vp], i32),
            "rra_comm_plan_kernel": ([vp, sz, i32, i32, ctypes.POINTER(ctypes.c_char_p)], i32),
            "rra_comm_status": ([vp], i32),
            "rra_comm_error_site": ([vp, ip, ip], i32),
            "rra_comm_last_kernel": ([vp, ctypes.POINTER(ctypes.c_char_p)], i32),
            "rra_comm_reset": ([vp], i32),
            "rra_comm_destroy": ([vp], i32),
            "rra_comm_set_attr": ([vp, i32, i64], i32),
            "rra_comm_get_attr": ([vp, i32, ctypes.POINTER(i64)], i32),
            "rra_comm_layout": ([vp, ctypes.POINTER(Layout)], i32),
            "rra_plan_layout": ([i32, sz, sz, sz, ctypes.POINTER(Layout)], i32),
            "rra_select_algo": ([i32, sz, i32, ip], i32),
            "rra_comm_plan_call": ([vp, sz, i32, i32, ip, ip], i32),
            "rra_comm_max_coresident": ([vp, i32, i32, ip], i32),
            "rra_comm_set_timing": ([vp, vp], i32),
            "rra_comm_set_trace": ([vp, vp], i32),
            "rra_comm_inject_drop": ([vp, i32], i32),
            "rra_comm_barrier_latency": ([vp, i32, ctypes.POINTER(ctypes.c_double)], i32),
            "rra_comm_get_epoch": ([vp, ctypes.POINTER(ctypes.c_uint64)], i32),
            "rra_comm_set_epoch": ([vp, ctypes.c_uint64], i32),
            "rra_status_string": ([i32], ctypes.c_char_p),
            "rra_version": ([], ctypes.c_char_p),
            "rra_probe_l2_chase": ([sz, ctypes.c_uint64, ctypes.c_uint64, ctypes.POINTER(ctypes.c_double)], i32),
            "rra_probe_pingpong": ([i32, i32, i32, ctypes.POINTER(ctypes.c_double), ip, ip], i32),
            "rra_probe_dsmem_pingpong": ([i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                          ip, ip], i32),
            "rra_probe_empty_kernel": ([vp], i32),
            "rra_probe_sm_count": ([ip], i32),
            "rra_probe_host_link": ([sz, i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_double)], i32),
            "rra_probe_launch_shape": ([i32, i32, i32, i32, vp], i32),
            "rra_probe_launch_chain": ([i32, i32, i32, i32, vp], i32),
            "rra_reduce_scatter": ([vp, pp, pp, sz, i32, vp], i32),
            "rra_all_gather": ([vp, pp, pp, sz, i32, vp], i32),
            "rra_broadcast": ([vp, i32, pp, pp, sz, i32, vp], i32),
            "rra_reduce": ([vp, i32, pp, pp, sz, i32, vp], i32),
            "rra_allreduce_residual": ([vp, pp, pp, pp, sz, i32, vp], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(status: int, what: str):
    if status != OK:
        raise RraError(status, what)


def status_string(status: int) -> str:
    return load().rra_status_string(int(status)).decode()


def version() -> str:
    return load().rra_version().decode()


def plan_layout(nranks: int, max_bytes: int, scratch_oneshot: int = 0, scratch_twoshot: int = 0) -> dict:
    """Window layout for (nranks, max_bytes); pure host arithmetic (no GPU)."""
    lay = Layout()
    _check(load().rra_plan_layout(nranks, max_bytes, scratch_oneshot, scratch_twoshot, ctypes.byref(lay)),
           "rra_plan_layout")
    return lay.as_dict()


def select_algo(nranks: int, bytes_per_rank: int, dtype: str = "fp32") -> str:
    """Name of the algorithm RRA_AUTO uses (pure host arithmetic)."""
    v = ctypes.c_int()
    _check(load().rra_select_algo(int(nranks), int(bytes_per_rank), DTYPES[dtype], ctypes.byref(v)),
           "rra_select_algo")
    return ALGO_NAMES[v.value]


def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def _stream_handle(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_of(t) -> int:
    import torch
    m = {torch.float32: 0, torch.bfloat16: 1, torch.float64: 2}
    if t.dtype not in m:
        raise TypeError("unsupported dtype %s (float32, bfloat16, float64)" % t.dtype)
    return m[t.dtype]


class Comm:
    """A communicator of `nranks` virtual ranks on the current CUDA device."""

    def __init__(self, nranks: int, max_bytes: int):
        self._lib = load()
        h = ctypes.c_void_p()
        _check(self._lib.rra_comm_create(int(nranks), int(max_bytes), ctypes.byref(h)), "rra_comm_create")
        self._h = h
        self.nranks = int(nranks)
        self.max_bytes = int(max_bytes)

    # -- lifetime -----------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            st = self._lib.rra_comm_destroy(self._h)
            self._h = None
            _check(st, "rra_comm_destroy")

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- the operation ------------------------------------------------------
    def allreduce_ptrs(self, send_ptrs, recv_ptrs, count: int, dtype: str, algo: str, stream=None) -> None:
        sp, ks = _ptr_array(send_ptrs)
        rp, kr = _ptr_array(recv_ptrs)
        st = self._lib.rra_allreduce(self._h, sp, rp, int(count), DTYPES[dtype], ALGOS[algo],
                                     _stream_handle(stream))
        del ks, kr
        _check(st, "rra_allreduce")

    def prepare(self, send_ptrs, recv_ptrs, count: int, dtype: str, algo: str, stream=None):
        """Build the ctypes arguments of one call once; the returned callable
        enqueues that call (same buffers) with no per-call marshalling."""
        sp, ks = _ptr_array(send_ptrs)
        rp, kr = _ptr_array(recv_ptrs)
        fn = self._lib.rra_allreduce
        args = (self._h, sp, rp, ctypes.c_size_t(int(count)), ctypes.c_int(DTYPES[dtype]),
                ctypes.c_int(ALGOS[algo]), _stream_handle(stream))

        def call(_keep=(ks, kr)):
            st = fn(*args)
            if st != OK:
                raise RraError(st, "rra_allreduce")
        return call

    def allreduce(self, sends, recvs, algo: str, stream=None) -> None:
        """recvs[r][:] = sum over ranks of sends[p][:]; tensors on the GPU,
        one per rank, same dtype and element count, contiguous."""
        if len(sends) != self.nranks or len(recvs) != self.nranks:
            raise ValueError("need one send and one recv tensor per rank")
        dt = _dtype_of(sends[0])
        n = sends[0].numel()
        for t in list(sends) + list(recvs):
            if not t.is_cuda or not t.is_contiguous() or t.numel() != n or _dtype_of(t) != dt:
                raise ValueError("all tensors must be contiguous CUDA tensors of one dtype and size")
        dname = {0: "fp32", 1: "bf16", 2: "fp64"}[dt]
        self.allreduce_ptrs([t.data_ptr() for t in sends], [t.data_ptr() for t in recvs], n, dname, algo, stream)

    # -- AllReduce + residual add ------------------------------------------
    def allreduce_residual_ptrs(self, send_ptrs, resid_ptrs, recv_ptrs, count: int, dtype: str,
                                stream=None) -> None:
        sp, ks = _ptr_array(send_ptrs)
        qp, kq = _ptr_array(resid_ptrs)
        rp, kr = _ptr_array(recv_ptrs)
        st = self._lib.rra_allreduce_residual(self._h, sp, qp, rp, int(count), DTYPES[dtype], _stream_handle(stream))
        del ks, kq, kr
        _check(st, "rra_allreduce_residual")

    def prepare_residual(self, send_ptrs, resid_ptrs, recv_ptrs, count: int, dtype: str, stream=None):
        """As prepare(), for rra_allreduce_residual."""
        sp, ks = _ptr_array(send_ptrs)
        qp, kq = _ptr_array(resid_ptrs)
        rp, kr = _ptr_array(recv_ptrs)
        fn = self._lib.rra_allreduce_residual
        args = (self._h, sp, qp, rp, ctypes.c_size_t(int(count)), ctypes.c_int(DTYPES[dtype]), _stream_handle(stream))

        def call(_keep=(ks, kq, kr)):
            st = fn(*args)
            if st != OK:
                raise RraError(st, "rra_allreduce_residual")
        return call

    def allreduce_residual(self, sends, residuals, recvs, stream=None) -> None:
        """recvs[r] = sum over ranks of sends[p] + residuals[r] (one rounding)."""
        ts = list(sends) + list(residuals) + list(recvs)
        if len(sends) != self.nranks or len(residuals) != self.nranks or len(recvs) != self.nranks:
            raise ValueError("need one send, residual and recv tensor per rank")
        dt, n = _dtype_of(ts[0]), ts[0].numel()
        for t in ts:
            if not t.is_cuda or not t.is_contiguous() or t.numel() != n or _dtype_of(t) != dt:
                raise ValueError("all tensors must be contiguous CUDA tensors of one dtype and size")
        self.allreduce_residual_ptrs([t.data_ptr() for t in sends], [t.data_ptr() for t in residuals],
                                     [t.data_ptr() for t in recvs], n, {0: "fp32", 1: "bf16", 2: "fp64"}[dt],
                                     stream)

    # -- the other collectives ----------------------------------------------
    def _coll_args(self, op, send_ptrs, recv_ptrs, count, dtype, root, stream):
        if op not in COLLECTIVES:
            raise ValueError("collective must be one of %s" % (COLLECTIVES,))
        sp, ks = _ptr_array(send_ptrs)
        rp, kr = _ptr_array(recv_ptrs)
        fn = getattr(self._lib, "rra_" + op)
        tail = (ctypes.c_size_t(int(count)), ctypes.c_int(DTYPES[dtype]), _stream_handle(stream))
        if op in ("broadcast", "reduce"):
            args = (self._h, ctypes.c_int(int(root)), sp, rp) + tail
        else:
            args = (self._h, sp, rp) + tail
        return fn, args, (ks, kr)

    def collective_ptrs(self, op: str, send_ptrs, recv_ptrs, count: int, dtype: str, root: int = 0,
                        stream=None) -> None:
        """One ReduceScatter / AllGather / Broadcast / Reduce on raw device
        pointers (None where the collective ignores an entry)."""
        fn, args, keep = self._coll_args(op, send_ptrs, recv_ptrs, count, dtype, root, stream)
        st = fn(*args)
        del keep
        _check(st, "rra_" + op)

    def prepare_collective(self, op: str, send_ptrs, recv_ptrs, count: int, dtype: str, root: int = 0,
                           stream=None):
        """As prepare(), for one of the other collectives."""
        fn, args, keep = self._coll_args(op, send_ptrs, recv_ptrs, count, dtype, root, stream)

        def call(_keep=keep):
            st = fn(*args)
            if st != OK:
                raise RraError(st, "rra_" + op)
        return call

    def _tensor_call(self, op, sends, recvs, count, root, stream):
        if len(sends) != self.nranks or len(recvs) != self.nranks:
            raise ValueError("need one send and one recv entry per rank (None where unused)")
        ts = [t for t in list(sends) + list(recvs) if t is not None]
        dt = _dtype_of(ts[0])
        for t in ts:
            if not t.is_cuda or not t.is_contiguous() or _dtype_of(t) != dt:
                raise ValueError("all tensors must be contiguous CUDA tensors of one dtype")
        dname = {0: "fp32", 1: "bf16", 2: "fp64"}[dt]
        ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        self.collective_ptrs(op, [ptr(t) for t in sends], [ptr(t) for t in recvs], count, dname, root, stream)

    def reduce_scatter(self, sends, recvs, stream=None) -> None:
        """recvs[r] = sum over ranks of block r of sends[p]; each send holds
        N * recvs[r].numel() elements."""
        self._tensor_call("reduce_scatter", sends, recvs, recvs[0].numel(), 0, stream)

    def all_gather(self, sends, recvs, stream=None) -> None:
        """recvs[r] = concatenation of sends[0..N-1]."""
        self._tensor_call("all_gather", sends, recvs, sends[0].numel(), 0, stream)

    def broadcast(self, sends, recvs, root: int, stream=None) -> None:
        """Every recvs[r] = sends[root] (other sends may be None)."""
        self._tensor_call("broadcast", sends, recvs, recvs[0].numel(), root, stream)

    def reduce(self, sends, recvs, root: int, stream=None) -> None:
        """recvs[root] = sum over ranks of sends[p] (other recvs may be None)."""
        self._tensor_call("reduce", sends, recvs, sends[0].numel(), root, stream)

    def prepare_host(self, send_ptrs, recv_ptrs, count: int, dtype: str, algo: str, stream=None):
        """As prepare(), for host buffers (synchronises per call).  When every
        buffer is pinned, device-mapped host memory and zero copy is on, the
        buffers are resolved once (rra_host_device_ptrs) and each call is
        rra_allreduce_mapped; otherwise each call is rra_allreduce_host.  The
        buffers must stay allocated while the call is in use."""
        n = len(send_ptrs)
        if self.get_attr("host_zero_copy"):
            dev = host_device_ptrs(list(send_ptrs) + list(recv_ptrs))
            if all(d is not None for d in dev):
                sp, ks = _ptr_array(dev[:n])
                rp, kr = _ptr_array(dev[n:])
                fn, name = self._lib.rra_allreduce_mapped, "rra_allreduce_mapped"
            else:
                sp, ks = _ptr_array(send_ptrs)
                rp, kr = _ptr_array(recv_ptrs)
                fn, name = self._lib.rra_allreduce_host, "rra_allreduce_host"
        else:
            sp, ks = _ptr_array(send_ptrs)
            rp, kr = _ptr_array(recv_ptrs)
            fn, name = self._lib.rra_allreduce_host, "rra_allreduce_host"
        args = (self._h, sp, rp, ctypes.c_size_t(int(count)), ctypes.c_int(DTYPES[dtype]),
                ctypes.c_int(ALGOS[algo]), _stream_handle(stream))

        def call(_keep=(ks, kr)):
            st = fn(*args)
            if st != OK:
                raise RraError(st, name)
        return call

    def allreduce_host(self, send_ptrs, recv_ptrs, count: int, dtype: str, algo: str, stream=None) -> None:
        """Host buffers in, host buffers out (H2D, kernel, D2H, synchronise)."""
        sp, ks = _ptr_array(send_ptrs)
        rp, kr = _ptr_array(recv_ptrs)
        st = self._lib.rra_allreduce_host(self._h, sp, rp, int(count), DTYPES[dtype], ALGOS[algo],
                                          _stream_handle(stream))
        del ks, kr
        _check(st, "rra_allreduce_host")

    # -- control ------------------------------------------------------------
    def status(self):
        """(status code, rank, step) -- rra_comm_status, then rra_comm_error_site
        for where the error was recorded; synchronises the device."""
        st = self._lib.rra_comm_status(self._h)
        rank = ctypes.c_int(-1)
        step = ctypes.c_int(-1)
        _check(self._lib.rra_comm_error_site(self._h, ctypes.byref(rank), ctypes.byref(step)),
               "rra_comm_error_site")
        return st, rank.value, step.value

    def last_kernel(self) -> str:
        """Name of the kernel the last call on this communicator launched."""
        name = ctypes.c_char_p()
        _check(self._lib.rra_comm_last_kernel(self._h, ctypes.byref(name)), "rra_comm_last_kernel")
        return name.value.decode()

    def reset(self):
        _check(self._lib.rra_comm_reset(self._h), "rra_comm_reset")

    def set_attr(self, name: str, value: int):
        _check(self._lib.rra_comm_set_attr(self._h, ATTRS[name], int(value)), "rra_comm_set_attr")

    def get_attr(self, name: str) -> int:
        v = ctypes.c_int64()
        _check(self._lib.rra_comm_get_attr(self._h, ATTRS[name], ctypes.byref(v)), "rra_comm_get_attr")
        return v.value

    def layout(self) -> dict:
        lay = Layout()
        _check(self._lib.rra_comm_layout(self._h, ctypes.byref(lay)), "rra_comm_layout")
        return lay.as_dict()

    def plan_call(self, count: int, dtype: str, algo: str):
        g = ctypes.c_int()
        s = ctypes.c_int()
        _check(self._lib.rra_comm_plan_call(self._h, int(count), DTYPES[dtype], ALGOS[algo],
                                            ctypes.byref(g), ctypes.byref(s)), "rra_comm_plan_call")
        return g.value, s.value

    def plan_kernel(self, count: int, dtype: str, algo: str) -> str:
        """Name of the kernel rra_allreduce launches for this call."""
        name = ctypes.c_char_p()
        _check(self._lib.rra_comm_plan_kernel(self._h, int(count), DTYPES[dtype], ALGOS[algo], ctypes.byref(name)),
               "rra_comm_plan_kernel")
        return name.value.decode()

    def max_coresident(self, dtype: str, algo: str) -> int:
        v = ctypes.c_int()
        _check(self._lib.rra_comm_max_coresident(self._h, DTYPES[dtype], ALGOS[algo], ctypes.byref(v)),
               "rra_comm_max_coresident")
        return v.value

    def set_timing(self, dev_ptr):
        _check(self._lib.rra_comm_set_timing(self._h, ctypes.c_void_p(dev_ptr or 0)), "rra_comm_set_timing")

    def barrier_latency(self, iters: int = 1000) -> float:
        """Mean ns per N-way flag barrier (the baseline's barrier)."""
        v = ctypes.c_double()
        _check(self._lib.rra_comm_barrier_latency(self._h, int(iters), ctypes.byref(v)), "rra_comm_barrier_latency")
        return v.value

    def epoch(self) -> int:
        v = ctypes.c_uint64()
        _check(self._lib.rra_comm_get_epoch(self._h, ctypes.byref(v)), "rra_comm_get_epoch")
        return v.value

    def set_epoch(self, epoch: int):
        _check(self._lib.rra_comm_set_epoch(self._h, int(epoch)), "rra_comm_set_epoch")

    def set_trace(self, dev_ptr):
        _check(self._lib.rra_comm_set_trace(self._h, ctypes.c_void_p(dev_ptr or 0)), "rra_comm_set_trace")

    def inject_drop(self, rank: int):
        _check(self._lib.rra_comm_inject_drop(self._h, int(rank)), "rra_comm_inject_drop")


# ------------------------------------------------------------------ probes --
def probe_l2_chase(buf_bytes: int = 8 << 20, hops: int = 200000, seed: int = 1) -> float:
    ns = ctypes.c_double()
    _check(load().rra_probe_l2_chase(int(buf_bytes), int(hops), int(seed), ctypes.byref(ns)), "rra_probe_l2_chase")
    return ns.value


def host_device_ptrs(host_ptrs):
    """Device addresses of pinned, device-mapped host buffers (None where a
    pointer is not such memory)."""
    n = len(host_ptrs)
    hp, keep = _ptr_array(host_ptrs)
    out = (ctypes.c_void_p * max(1, n))()
    _check(load().rra_host_device_ptrs(n, hp, out), "rra_host_device_ptrs")
    del keep
    return [out[i] if out[i] else None for i in range(n)]


def probe_pingpong(cta_a: int, cta_b: int, iters: int = 20000):
    ns = ctypes.c_double()
    a = ctypes.c_int()
    b = ctypes.c_int()
    _check(load().rra_probe_pingpong(int(cta_a), int(cta_b), int(iters), ctypes.byref(ns), ctypes.byref(a),
                                     ctypes.byref(b)), "rra_probe_pingpong")
    return ns.value, a.value, b.value


def probe_empty_kernel(stream=None):
    _check(load().rra_probe_empty_kernel(_stream_handle(stream)), "rra_probe_empty_kernel")


def probe_launch_shape(ctas: int, threads: int, big_params: bool, cooperative: bool, stream=None):
    _check(load().rra_probe_launch_shape(int(ctas), int(threads), int(bool(big_params)), int(bool(cooperative)),
                                         _stream_handle(stream)), "rra_probe_launch_shape")


def probe_launch_chain(ctas: int, threads: int, cluster: int, pdl: bool, stream=None):
    _check(load().rra_probe_launch_chain(int(ctas), int(threads), int(cluster), int(bool(pdl)),
                                         _stream_handle(stream)), "rra_probe_launch_chain")


def probe_sm_count() -> int:
    v = ctypes.c_int()
    _check(load().rra_probe_sm_count(ctypes.byref(v)), "rra_probe_sm_count")
    return v.value


def probe_host_link(nbytes: int = 8 << 20, iters: int = 20):
    """(read, write, copy) GB/s of the device streaming pinned host memory:
    reading one buffer, writing another, and copying one into the other (each
    direction at once)."""
    r = ctypes.c_double()
    w = ctypes.c_double()
    c = ctypes.c_double()
    _check(load().rra_probe_host_link(int(nbytes), int(iters), ctypes.byref(r), ctypes.byref(w), ctypes.byref(c)),
           "rra_probe_host_link")
    return r.value, w.value, c.value


def probe_dsmem_pingpong(iters: int = 20000):
    """(ns per bulk-copy round trip inside a 2-CTA cluster, ns per cluster
    barrier, SM id of CTA 0, SM id of CTA 1)."""
    rt = ctypes.c_double()
    cb = ctypes.c_double()
    a = ctypes.c_int()
    b = ctypes.c_int()
    _check(load().rra_probe_dsmem_pingpong(int(iters), ctypes.byref(rt), ctypes.byref(cb), ctypes.byref(a),
                                           ctypes.byref(b)), "rra_probe_dsmem_pingpong")
    return rt.value, cb.value, a.value, b.value
