"""GPU parity of rra_allreduce_residual (the AllReduce with its residual add
fused) against the oracle, bit for bit: both shapes (one-shot, two-shot),
every dtype, ragged sizes, many epochs per cluster (sub-buffer reuse), in
place, graph replay, and a dropped rank.  Up to 16 ranks the one-shot sizes
run the cluster AllReduce's bulk-copy one-shot with the residual add in its
epilogue, the rest the kernel written on the public device API
(include/rra_device.cuh); above 16 ranks the many-rank cluster kernels with
the residual add in their epilogue."""
import numpy as np
import pytest

import oracle
from latency_barrier_free_gb300 import inputs, rra
from tests.gpu_util import ELEM, bits, poison_like, to_device, to_host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _case(n, count, dtype, *tags):
    g = inputs.rng(95, count, n, *tags)
    return inputs.normal(g, n, count, dtype), inputs.normal(g, n, count, dtype)


def _check(comm, sends_np, res_np, dtype, in_place=None):
    sends, res = to_device(sends_np, dtype), to_device(res_np, dtype)
    recvs = {"send": sends, "residual": res}.get(in_place) or poison_like(sends)
    comm.allreduce_residual(sends, res, recvs)
    torch.cuda.synchronize()
    st, rk, step = comm.status()
    assert st == rra.OK, "%s (rank %d epoch %d)" % (rra.STATUS_NAMES.get(st), rk, step)
    expect = oracle.allreduce_residual(sends_np, res_np, dtype)
    for r, got in enumerate(to_host(recvs, dtype)):
        assert np.array_equal(bits(got), bits(expect[r])), r


@pytest.mark.parametrize("tma", [0, -1])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [2, 3, 4, 8, 16, 17, 33, 64])
def test_parity(n, dtype, tma):
    """Sizes on both sides of the one-shot / two-shot switch, ragged tails
    included; st.async sends (tma 0) and, by default, the API's bulk sends
    (up to 16 ranks)."""
    if n > 16 and tma == 0:
        pytest.skip("above 16 ranks the push attribute does not apply")
    with rra.Comm(n, 100003 * ELEM[dtype]) as comm:
        comm.set_attr("cluster_tma", tma)
        for count in (1, 7, 33, 4097, 100003):
            sends_np, res_np = _case(n, count, dtype)
            _check(comm, sends_np, res_np, dtype)


@pytest.mark.parametrize("tma", [0, 1])
@pytest.mark.parametrize("shape_count", [1000, 300001])  # one-shot, two-shot at N=4
@pytest.mark.parametrize("clusters", [1, 3])
@pytest.mark.parametrize("threads", [64, 256])
def test_many_epochs_per_cluster(shape_count, clusters, threads, tma):
    """Few clusters looping over many small slices: every sub-buffer of the
    device API's window is reused many times, each reuse relying on the
    receive-before-resend order; ragged last slice; st.async sends and bulk
    sends."""
    n, dtype = 4, "fp32"
    with rra.Comm(n, shape_count * 4) as comm:
        comm.set_attr("cluster_tma", tma)
        comm.set_attr("ctas_per_rank", clusters)
        comm.set_attr("threads", threads)
        comm.set_attr("cluster_slice", 16 * n * 3)  # 12 vectors per slice
        for it in range(2):
            sends_np, res_np = _case(n, shape_count, dtype, clusters, threads, it, tma)
            _check(comm, sends_np, res_np, dtype)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [2, 3, 8, 16])
def test_kernel_choice(n, dtype):
    """Up to 16 ranks, device inputs at one-shot sizes run the cluster
    AllReduce's bulk-copy one-shot with the residual epilogue; two-shot
    sizes, capped clusters (several slices per cluster) and st.async pushes
    run the device-API kernel.  Every form gives the oracle's bits."""
    small, large = 333, 1200007  # one-shot, two-shot at every N and dtype here, with either push
    with rra.Comm(n, large * ELEM[dtype]) as comm:
        for attrs, count, want in (({}, small, "cluster_tma_kernel<one-shot, residual>"),
                                   ({}, large, "residual_kernel<two-shot, bulk>"),
                                   ({"ctas_per_rank": 1}, small, "residual_kernel<one-shot, bulk>"),
                                   ({"ctas_per_rank": 2}, large, "residual_kernel<two-shot, bulk>"),
                                   ({"cluster_tma": 0}, small, "residual_kernel<one-shot>"),
                                   ({"cluster_tma": 0}, large, "residual_kernel<two-shot>")):
            comm.set_attr("ctas_per_rank", 0)
            comm.set_attr("cluster_tma", -1)
            for k, v in attrs.items():
                comm.set_attr(k, v)
            sends_np, res_np = _case(n, count, dtype, 11, count, *attrs.values())
            _check(comm, sends_np, res_np, dtype)
            assert comm.last_kernel() == want, (attrs, count, comm.last_kernel())


@pytest.mark.parametrize("n", [4, 40])
@pytest.mark.parametrize("in_place", ["send", "residual"])
@pytest.mark.parametrize("count", [3001, 90001])
def test_in_place(in_place, count, n):
    dtype = "bf16"
    with rra.Comm(n, count * 2) as comm:
        sends_np, res_np = _case(n, count, dtype, 7)
        _check(comm, sends_np, res_np, dtype, in_place=in_place)


@pytest.mark.parametrize("n", [8, 24])
def test_zero_residual_equals_allreduce(n):
    count, dtype = 12345, "bf16"
    with rra.Comm(n, count * 2) as comm:
        sends_np, _ = _case(n, count, dtype, 8)
        sends = to_device(sends_np, dtype)
        zeros = [torch.zeros_like(t) for t in sends]
        a, b = poison_like(sends), poison_like(sends)
        comm.allreduce_residual(sends, zeros, a)
        comm.allreduce(sends, b, "oneshot_cluster")
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        for x, y in zip(to_host(a, dtype), to_host(b, dtype)):
            assert np.array_equal(x, y)


def test_graph_replay():
    """160 fused calls (a decode step of an 80-layer model) in one CUDA
    graph, replayed with new inputs."""
    n, count, dtype, calls = 8, 8192, "bf16", 160
    with rra.Comm(n, count * 2) as comm:
        x = torch.empty(n, count, dtype=torch.bfloat16, device="cuda")
        res = torch.empty(n, count, dtype=torch.bfloat16, device="cuda")
        out = torch.empty(calls, n, count, dtype=torch.bfloat16, device="cuda")

        def enqueue():
            for i in range(calls):
                comm.allreduce_residual_ptrs([x[r].data_ptr() for r in range(n)], [res[r].data_ptr() for r in range(n)],
                                             [out[i, r].data_ptr() for r in range(n)], count, dtype)

        enqueue()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                enqueue()
        for rep in range(2):
            sends_np, res_np = _case(n, count, dtype, 9, rep)
            x.copy_(torch.stack(to_device(sends_np, dtype)))
            res.copy_(torch.stack(to_device(res_np, dtype)))
            out.view(torch.int16).fill_(0x7F7F)
            g.replay()
            torch.cuda.synchronize()
            assert comm.status()[0] == rra.OK
            expect = oracle.allreduce_residual(sends_np, res_np, dtype)
            got = out.view(torch.int16).cpu().numpy().view(np.uint16)
            for i in (0, 1, calls - 1):
                for r in range(n):
                    assert np.array_equal(got[i, r], expect[r]), (rep, i, r)


@pytest.mark.parametrize("n,tma", [(4, 0), (4, 1), (20, -1)])
@pytest.mark.parametrize("count", [1000, 300001])
def test_dropped_rank_times_out_and_reset(count, n, tma):
    dtype = "fp32"
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("cluster_tma", tma)
        comm.set_attr("poll_timeout_ms", 20)
        comm.set_attr("ctas_per_rank", 2)
        comm.inject_drop(n - 3)
        sends_np, res_np = _case(n, count, dtype, 10)
        sends, res = to_device(sends_np, dtype), to_device(res_np, dtype)
        recvs = poison_like(sends)
        comm.allreduce_residual(sends, res, recvs)
        st, rank, _ = comm.status()
        assert st == rra.ERR_TIMEOUT and 0 <= rank < n
        comm.reset()
        _check(comm, sends_np, res_np, dtype)


def test_argument_errors():
    with rra.Comm(4, 4096) as comm:
        x = [torch.zeros(1024, device="cuda") for _ in range(4)]
        p = [t.data_ptr() for t in x]
        with pytest.raises(rra.RraError):
            comm.allreduce_residual_ptrs(p, [None] + p[1:], p, 16, "fp32")
        with pytest.raises(rra.RraError):
            comm.allreduce_residual_ptrs(p, [p[0] + 4] + p[1:], p, 16, "fp32")
        with pytest.raises(rra.RraError):
            comm.allreduce_residual_ptrs(p, p, p, 1025, "fp32")
        comm.allreduce_residual_ptrs(p, p, p, 0, "fp32")
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
