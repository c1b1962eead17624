"""The entry point that allocates nothing (rra_allreduce_static), called
through the C ABI and checked against the oracle and against rra_allreduce on
the same inputs.

It exists for callers that cannot allocate device memory when they need an
AllReduce: plug-ins whose host framework owns the allocator, processes whose
device-memory budget is fixed up front, paths that must not pay for an
allocation.  Both entry points run the one-shot LL kernel, which adds the
ranks in order, so the bar is the one the other GPU tests use for it:
identical bits.  Each case runs two calls in a row on the shared static
scratch.

This file is collected last on purpose; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest

import oracle
from latency_barrier_free_gb300 import inputs, rra

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ELEM = {"fp32": 4, "bf16": 2, "fp64": 8}
TDT = {"fp32": "float32", "bf16": "bfloat16", "fp64": "float64"}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    lib = rra.load()
    fn = lib.rra_allreduce_static
    fn.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                   ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return lib


def _dev(arrs, dtype):
    out = []
    for a in arrs:
        if dtype == "bf16":
            out.append(torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda())
        else:
            out.append(torch.from_numpy(a.copy()).cuda())
    return out


def _bits(t):
    return t.view(torch.uint8).cpu().numpy()


def _ptrs(ts):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


@pytest.mark.parametrize("n,count,dtype", [(2, 32, "fp32"), (3, 1001, "fp32"), (4, 4096, "fp32"),
                                           (8, 8192, "bf16"), (8, 2048, "fp64"), (5, 7, "bf16")])
def test_static_entry_matches_allreduce_twice(lib, n, count, dtype):
    stream = torch.cuda.current_stream()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    with rra.Comm(n, count * ELEM[dtype]) as comm:
        for call in range(2):  # two calls in a row, fresh inputs each
            host = inputs.normal(inputs.rng(80, call, n, count), n, count, dtype)
            xs = _dev(host, dtype)
            ref = [torch.empty_like(x) for x in xs]
            comm.allreduce(xs, ref, "oneshot_ll")                   # existing entry point
            got = [torch.empty_like(x).fill_(7) for x in xs]
            sp, ks = _ptrs(xs)
            rp, kr = _ptrs(got)
            st = lib.rra_allreduce_static(n, sp, rp, count, rra.DTYPES[dtype], ctypes.c_void_p(status.data_ptr()),
                                          ctypes.c_void_p(stream.cuda_stream))
            assert st == rra.OK
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            expect = oracle.allreduce(host, dtype)
            for r in range(n):
                assert np.array_equal(_bits(got[r]), expect[r].view(np.uint8)), (call, r)  # the oracle
                assert np.array_equal(_bits(got[r]), _bits(ref[r])), (call, r)  # the existing entry point
            del ks, kr


def test_static_entry_calls_with_changing_rank_counts(lib):
    """Calls with different rank counts share the array's eight windows."""
    stream = torch.cuda.current_stream()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for k, n in enumerate((8, 2, 5, 8, 3, 8)):
        count = 1500
        host = inputs.normal(inputs.rng(81, k, n, count), n, count, "fp32")
        xs = _dev(host, "fp32")
        got = [torch.full_like(x, float("nan")) for x in xs]
        sp, ks = _ptrs(xs)
        rp, kr = _ptrs(got)
        assert lib.rra_allreduce_static(n, sp, rp, count, rra.DTYPES["fp32"], ctypes.c_void_p(status.data_ptr()),
                                        ctypes.c_void_p(stream.cuda_stream)) == rra.OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        expect = oracle.allreduce(host, "fp32")
        for r in range(n):
            assert np.array_equal(_bits(got[r]), expect[r].view(np.uint8)), (k, n, r)
        del ks, kr


def test_static_entry_allocates_no_device_memory(lib):
    """Free device memory is the same before and after two calls (buffers,
    the status word and the first call's set-up are all in place first)."""
    stream = torch.cuda.current_stream()
    n, count = 4, 2048
    host = inputs.normal(inputs.rng(82, 0, n, count), n, count, "fp32")
    xs = _dev(host, "fp32")
    got = [torch.empty_like(x) for x in xs]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp, ks = _ptrs(xs)
    rp, kr = _ptrs(got)
    args = (n, sp, rp, count, rra.DTYPES["fp32"], ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    assert lib.rra_allreduce_static(*args) == rra.OK
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        assert lib.rra_allreduce_static(*args) == rra.OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert int(status.item()) == 0
    expect = oracle.allreduce(host, "fp32")
    for r in range(n):
        assert np.array_equal(_bits(got[r]), expect[r].view(np.uint8))
    del ks, kr


def test_static_entry_rejects_what_does_not_fit(lib):
    x = [torch.zeros(8192, device="cuda") for _ in range(9)]
    sp, ks = _ptrs(x)
    # 16 KiB + 4 bytes per rank: beyond the static slots
    assert lib.rra_allreduce_static(2, sp, sp, 4097, rra.DTYPES["fp32"], None, None) == rra.ERR_INVALID_ARG
    # nine ranks: more windows than the array holds
    assert lib.rra_allreduce_static(9, sp, sp, 16, rra.DTYPES["fp32"], None, None) == rra.ERR_INVALID_ARG
    assert lib.rra_allreduce_static(2, sp, sp, 0, rra.DTYPES["fp32"], None, None) == rra.OK
    del ks
