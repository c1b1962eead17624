"""GPU tests of the runtime around the kernels: CUDA-graph replay with
device-resident epochs, bounded waits and fault reporting, reset, the
host-buffer entry point, in-kernel timing and the latency probes."""
import numpy as np
import pytest

import oracle
from latency_barrier_free_gb300 import inputs, rra
from tests.gpu_util import ALGOS, CLUSTER, bits, check_against_oracle, poison_like, to_device, to_host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


@pytest.mark.parametrize("algo", ALGOS + CLUSTER)
def test_graph_replay_advances_epochs(algo):
    """Capture 20 calls in a CUDA graph and replay it 5 times with new inputs
    copied in between: every replay must see fresh epochs (LL flags) and
    reset sentinels, so every replay's result is correct."""
    n, count, calls = 4, 3000, 20
    with rra.Comm(n, count * 4) as comm:
        send = torch.zeros(calls, n, count, device="cuda")
        recv = torch.zeros(calls, n, count, device="cuda")

        def enqueue():
            for i in range(calls):
                comm.allreduce_ptrs([send[i, r].data_ptr() for r in range(n)],
                                    [recv[i, r].data_ptr() for r in range(n)], count, "fp32", algo)

        enqueue()  # warm-up outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                enqueue()
        torch.cuda.synchronize()
        for rep in range(5):
            host = [inputs.normal(inputs.rng(70, rep, i), n, count, "fp32") for i in range(calls)]
            send.copy_(torch.from_numpy(np.stack([np.stack(h) for h in host])))
            recv.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert comm.status()[0] == rra.OK
            got = recv.cpu().numpy()
            for i in range(calls):
                check_against_oracle(host[i], list(got[i]), "fp32", algo)


@pytest.mark.parametrize("algo", ALGOS + CLUSTER)
def test_timeout_poison_and_reset(algo):
    """A rank that drops its stores makes its peers' polls run out of time:
    the device records RRA_ERR_TIMEOUT (no fault, no hang), the communicator
    is poisoned, and rra_comm_reset restores a working state.  (Cluster
    kernels here with st.async pushes; the bulk-copy push has its own test.)"""
    n, count = 4, 5000
    sends_np = inputs.normal(inputs.rng(71, 0), n, count, "fp32")
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("cluster_tma", 0)
        comm.set_attr("poll_timeout_ms", 20)
        comm.inject_drop(2)
        sends = to_device(sends_np, "fp32")
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, algo)
        st, rank, step = comm.status()
        assert st == rra.ERR_TIMEOUT
        assert 0 <= rank < n and step == 0
        with pytest.raises(rra.RraError) as e:
            comm.allreduce(sends, recvs, algo)
        assert e.value.status == rra.ERR_POISONED
        comm.reset()
        assert comm.status()[0] == rra.OK
        comm.allreduce(sends, recvs, algo)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", algo)


@pytest.mark.parametrize("algo", CLUSTER)
def test_cluster_many_ranks_timeout_and_reset(algo):
    """N=32 (16-CTA clusters hosting two ranks each) with a dropped rank:
    RRA_ERR_TIMEOUT, no hang; correct after a reset."""
    n, count = 32, 4000
    sends_np = inputs.normal(inputs.rng(77, 0), n, count, "fp32")
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("poll_timeout_ms", 20)
        comm.inject_drop(21)
        sends = to_device(sends_np, "fp32")
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, algo)
        assert comm.status()[0] == rra.ERR_TIMEOUT
        comm.reset()
        comm.allreduce(sends, recvs, algo)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", algo)


@pytest.mark.parametrize("algo", ["oneshot_cluster", "twoshot_cluster"])
def test_bulk_copy_push_timeout_and_reset(algo):
    """Bulk-copy push with a rank that skips its copies to peers: the
    receivers' bounded waits run out (RRA_ERR_TIMEOUT, no hang), every CTA
    still meets the others at the exit barrier, and after a reset the call
    is correct."""
    n, count = 4, 40000
    sends_np = inputs.normal(inputs.rng(78, 0), n, count, "fp32")
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("cluster_tma", 1)
        comm.set_attr("poll_timeout_ms", 20)
        comm.inject_drop(2)
        sends = to_device(sends_np, "fp32")
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, algo)
        st, rank, _ = comm.status()
        assert st == rra.ERR_TIMEOUT and 0 <= rank < n
        comm.reset()
        comm.allreduce(sends, recvs, algo)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", algo)


def test_pipelined_cluster_timeout_and_reset():
    """The persistent cluster two-shot with a rank that drops its pushes:
    waits on data and on credits run out, RRA_ERR_TIMEOUT is recorded, and
    after a reset the same plan gives the oracle's result."""
    n, count = 4, 40000
    sends_np = inputs.normal(inputs.rng(74, 0), n, count, "fp32")
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("cluster_pipe", 1)
        comm.set_attr("ctas_per_rank", 2)
        comm.set_attr("cluster_slice", 1024)
        comm.set_attr("poll_timeout_ms", 20)
        comm.inject_drop(1)
        sends = to_device(sends_np, "fp32")
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, "twoshot_cluster")
        st, rank, step = comm.status()
        assert st == rra.ERR_TIMEOUT
        assert 0 <= rank < n and step in (0, 1)  # the first wait to give up: slice 0 or 1
        comm.reset()
        comm.allreduce(sends, recvs, "twoshot_cluster")
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", "twoshot_cluster")


def test_device_error_makes_later_calls_noops():
    """Calls enqueued after a device-side failure (before the host looks) do
    nothing on the device and do not hang."""
    n, count = 2, 1000
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("poll_timeout_ms", 10)
        comm.inject_drop(0)
        x = [torch.ones(count, device="cuda") for _ in range(n)]
        y = poison_like(x)
        for _ in range(5):
            comm.allreduce(x, y, "oneshot_ll")
        st, _, _ = comm.status()
        assert st == rra.ERR_TIMEOUT
        comm.reset()
        comm.allreduce(x, y, "oneshot_ll")
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        assert torch.equal(y[0], torch.full_like(y[0], 2.0))


def test_argument_errors():
    with rra.Comm(4, 4096) as comm:
        x = [torch.zeros(1024, device="cuda") for _ in range(4)]
        ptrs = [t.data_ptr() for t in x]
        with pytest.raises(rra.RraError) as e:  # larger than max_bytes
            comm.allreduce_ptrs(ptrs, ptrs, 2048, "fp32", "oneshot_ll")
        assert e.value.status == rra.ERR_INVALID_ARG
        with pytest.raises(rra.RraError):       # misaligned pointer
            comm.allreduce_ptrs([p + 4 for p in ptrs], ptrs, 16, "fp32", "oneshot_ll")
        with pytest.raises(rra.RraError):       # null pointer
            comm.allreduce_ptrs([0] * 4, ptrs, 16, "fp32", "oneshot_ll")
        with pytest.raises(rra.RraError):
            comm.set_attr("threads", 96)
    with pytest.raises(rra.RraError):
        rra.Comm(1, 4096)
    with pytest.raises(rra.RraError):
        rra.Comm(65, 4096)


@pytest.mark.parametrize("algo", ALGOS)
def test_host_buffer_entry_point(algo):
    n, count = 8, 10000
    sends_np = inputs.normal(inputs.rng(72, 0), n, count, "fp32")
    recvs_np = [np.full(count, np.nan, np.float32) for _ in range(n)]
    with rra.Comm(n, count * 4) as comm:
        for _ in range(2):
            comm.allreduce_host([a.ctypes.data for a in sends_np], [a.ctypes.data for a in recvs_np],
                                count, "fp32", algo)
            check_against_oracle(sends_np, recvs_np, "fp32", algo)


@pytest.mark.parametrize("zero_copy", [1, 0])
@pytest.mark.parametrize("algo", ALGOS + CLUSTER)
def test_host_entry_pinned_buffers(algo, zero_copy):
    """Pinned host buffers: with zero copy the kernel reads and writes host
    memory directly; without it the call stages through device buffers.
    Both give the oracle's result, twice in a row."""
    n, count = 4, 70001
    sends_np = inputs.normal(inputs.rng(73, 0), n, count, "fp32")
    hs = [torch.from_numpy(a).pin_memory() for a in sends_np]
    hr = [torch.full((count,), float("nan")).pin_memory() for _ in range(n)]
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("host_zero_copy", zero_copy)
        for _ in range(2):
            comm.allreduce_host([t.data_ptr() for t in hs], [t.data_ptr() for t in hr], count, "fp32", algo)
            check_against_oracle(sends_np, [t.numpy() for t in hr], "fp32", algo)
            for t in hr:
                t.fill_(float("nan"))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("n", [3, 8, 16])
def test_host_zero_copy_two_shot(n, dtype):
    """The cluster two-shot on pinned host buffers (zero copy) takes its own
    slices (4 KiB, aligned up to N partitions): the oracle's result at a size
    of many slices and a ragged tail, for N that do and do not divide a
    slice."""
    count = 300001
    sends_np = inputs.normal(inputs.rng(77, n), n, count, dtype)
    tdt = torch.float32 if dtype == "fp32" else torch.bfloat16
    hs = [torch.from_numpy(a.view(np.int16) if dtype == "bf16" else a).view(tdt).pin_memory() for a in sends_np]
    hr = [torch.full((count,), float("nan"), dtype=tdt).pin_memory() for _ in range(n)]
    with rra.Comm(n, count * 4) as comm:
        call = comm.prepare_host([t.data_ptr() for t in hs], [t.data_ptr() for t in hr], count, dtype,
                                 "twoshot_cluster")
        for _ in range(2):
            call()
            got = [t.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else t.numpy() for t in hr]
            check_against_oracle(sends_np, got, dtype, "twoshot_cluster")
            for t in hr:
                t.fill_(float("nan"))


@pytest.mark.parametrize("algo", ["auto", "oneshot_cluster", "twoshot_cluster", "oneshot_sentinel", "ll128_atomic"])
def test_host_buffers_resolved_once(algo):
    """Pinned host buffers resolved once (rra_host_device_ptrs), then
    rra_allreduce_mapped per call: the oracle's result on every call; a
    pageable buffer does not resolve; a device error comes back from the call
    itself and a reset clears it."""
    n, count = 4, 30001
    sends_np = inputs.normal(inputs.rng(76, 0), n, count, "fp32")
    hs = [torch.from_numpy(a).pin_memory() for a in sends_np]
    hr = [torch.full((count,), float("nan")).pin_memory() for _ in range(n)]
    dev = rra.host_device_ptrs([t.data_ptr() for t in hs + hr] + [sends_np[0].ctypes.data, None])
    assert all(d is not None for d in dev[:2 * n])
    assert dev[2 * n] is None and dev[2 * n + 1] is None
    with rra.Comm(n, count * 4) as comm:
        call = comm.prepare_host([t.data_ptr() for t in hs], [t.data_ptr() for t in hr], count, "fp32", algo)
        for _ in range(3):
            call()
            check_against_oracle(sends_np, [t.numpy() for t in hr], "fp32", algo)
            for t in hr:
                t.fill_(float("nan"))
        comm.set_attr("poll_timeout_ms", 20)
        comm.inject_drop(2)
        with pytest.raises(rra.RraError) as e:
            call()
        assert e.value.status == rra.ERR_TIMEOUT
        comm.inject_drop(-1)
        comm.reset()
        call()
        check_against_oracle(sends_np, [t.numpy() for t in hr], "fp32", algo)


def test_plan_kernel_names_the_launched_kernel():
    """rra_comm_plan_kernel names the __global__ function a call launches:
    the automatic choice per size and rank count, the push attribute, the
    global-memory kernels and their wide variants."""
    with rra.Comm(4, 1 << 20) as comm:
        assert comm.plan_kernel(32, "fp32", "auto") == "cluster_tma_kernel<one-shot>"
        assert comm.plan_kernel(1 << 18, "fp32", "auto") == "cluster_tma_kernel<two-shot>"  # N^2 M = 16 MiB
        assert comm.plan_kernel(1 << 16, "fp32", "twoshot_cluster") == "cluster_tma_kernel<two-shot>"
        assert comm.plan_kernel(32, "fp32", "oneshot_sentinel") == "oneshot_kernel<sentinel>"
        assert comm.plan_kernel(32, "fp32", "twoshot_direct") == "twoshot_kernel<direct>"
        comm.set_attr("cluster_tma", 0)
        assert comm.plan_kernel(32, "fp32", "auto") == "cluster_kernel<one-shot>"
        comm.set_attr("cluster_pipe", 1)
        assert comm.plan_kernel(1 << 18, "fp32", "twoshot_cluster") == "cluster_pipe_kernel"
    with rra.Comm(16, 1 << 16) as comm:
        assert comm.plan_kernel(256, "fp32", "ll128_atomic") == "ll128_wide_kernel"
        assert comm.plan_kernel(256, "fp32", "oneshot_ll") == "oneshot_wide_kernel<LL>"
    with rra.Comm(32, 1 << 16) as comm:
        assert comm.plan_kernel(256, "fp32", "auto") == "cluster_multi_kernel<one-shot, bulk>"
        assert comm.plan_kernel(1 << 14, "fp32", "auto") == "cluster_multi_kernel<two-shot, bulk>"  # 16 N M = 32 MiB
        comm.set_attr("cluster_tma", 0)
        assert comm.plan_kernel(256, "fp32", "auto") == "cluster_multi_kernel<one-shot>"
        assert comm.plan_kernel(1 << 14, "fp32", "auto") == "cluster_multi_kernel<two-shot>"


def test_in_kernel_timing():
    n, count = 4, 1 << 16
    with rra.Comm(n, count * 4) as comm:
        grid, _ = comm.plan_call(count, "fp32", "oneshot_sentinel")
        buf = torch.zeros(2 * grid, dtype=torch.int64, device="cuda")
        comm.set_timing(buf.data_ptr())
        x = [torch.randn(count, device="cuda") for _ in range(n)]
        y = poison_like(x)
        comm.allreduce(x, y, "oneshot_sentinel")
        torch.cuda.synchronize()
        comm.set_timing(0)
        t = buf.view(grid, 2).cpu().numpy()
        assert np.all(t[:, 0] > 0) and np.all(t[:, 1] >= t[:, 0])
        assert t[:, 1].max() - t[:, 0].min() < 10_000_000  # < 10 ms


@pytest.mark.parametrize("algo,n", [("oneshot_ll", 2), ("oneshot_ll", 4), ("oneshot_sentinel", 2),
                                    ("oneshot_sentinel", 4), ("oneshot_cluster", 4)])
def test_trace_points(algo, n):
    """rra_comm_set_trace: the call launches the traced variant, its result is
    still exact, and every CTA's six stamps are set and in order; with the
    buffer switched off a call leaves it untouched."""
    count = 32
    sends_np = inputs.normal(inputs.rng(102, n), n, count, "fp32")
    with rra.Comm(n, count * 4) as comm:
        grid, _ = comm.plan_call(count, "fp32", algo)
        buf = torch.zeros(6 * grid, dtype=torch.int64, device="cuda")
        comm.set_trace(buf.data_ptr())
        sends = to_device(sends_np, "fp32")
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, algo)
        torch.cuda.synchronize()
        comm.set_trace(0)
        assert comm.status()[0] == rra.OK
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", algo)
        t = buf.view(grid, 6).cpu().numpy()
        assert np.all(t > 0), t
        assert np.all(np.diff(t, axis=1) >= 0), t
        assert t[:, 5].max() - t[:, 0].min() < 10_000_000  # < 10 ms
        buf.fill_(-1)
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, algo)
        torch.cuda.synchronize()
        assert bool((buf == -1).all())
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", algo)


def test_probes():
    ns = rra.probe_l2_chase(4 << 20, 20000, 3)
    assert 50.0 < ns < 10000.0
    sms = rra.probe_sm_count()
    rtt, sa, sb = rra.probe_pingpong(0, sms - 1, 2000)
    assert sa != sb and 50.0 < rtt < 100000.0
    # bulk-copy ping-pong inside a 2-CTA cluster: SM ids, a round trip and a
    # cluster barrier in a plausible range
    brtt, bar, s0, s1 = rra.probe_dsmem_pingpong(2000)
    assert 0 <= s0 < sms and 0 <= s1 < sms
    assert 20.0 < brtt < 100000.0 and 1.0 < bar < 100000.0
    rra.probe_empty_kernel()
    torch.cuda.synchronize()


def test_probe_launch_chain():
    """Empty kernels launched in clusters and with programmatic dependent
    launch run to completion on a stream and inside a captured graph; shapes
    the probe does not take are refused."""
    for cluster, pdl in ((4, True), (4, False), (1, True), (8, True)):
        rra.probe_launch_chain(8, 32, cluster, pdl)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for _ in range(8):
                rra.probe_launch_chain(4, 32, 4, True, s)
    g.replay()
    torch.cuda.synchronize()
    for ctas, threads, cluster in ((6, 32, 4), (4, 16, 1), (4, 32, 0), (16, 32, 16)):
        with pytest.raises(rra.RraError):
            rra.probe_launch_chain(ctas, threads, cluster, True)


def test_probe_host_link():
    """The host-link probe: three positive rates below any plausible link
    (the probe itself checks that its copy arrived whole), and its argument
    checks."""
    r, w, c = rra.probe_host_link(1 << 20, 5)
    for x in (r, w, c):
        assert 1.0 < x < 5000.0
    for nbytes, iters in ((1000, 5), (1 << 20, 0), ((1 << 20) + 8, 5)):
        with pytest.raises(rra.RraError):
            rra.probe_host_link(nbytes, iters)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("start", [2 ** 31 - 5, 2 ** 32 - 3, 3 * 2 ** 31 - 1])
def test_epoch_scrub_at_boundary(algo, start):
    """Calls whose epochs reach a multiple of 2^31 first zero every LL flag
    region (grid-wide, one bounded barrier) and restart the epoch one past the
    multiple; results stay exact across the boundary, also where the low 32
    bits of the epoch wrap."""
    n, count = 4, 50000
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("oneshot_chunk", 4096)
        comm.set_attr("twoshot_chunk", 8192)
        comm.set_attr("ll128_chunk", 8192)
        _, steps = comm.plan_call(count, "fp32", algo)
        assert steps >= 5
        comm.set_epoch(start)
        for it in range(3):
            sends_np = inputs.normal(inputs.rng(73, it), n, count, "fp32")
            sends = to_device(sends_np, "fp32")
            recvs = poison_like(sends)
            comm.allreduce(sends, recvs, algo)
            torch.cuda.synchronize()
            assert comm.status()[0] == rra.OK
            check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", algo)
        boundary = (start | (2 ** 31 - 1)) + 1
        assert comm.epoch() == boundary + 1 + 3 * steps


def test_barrier_latency_and_baseline_timeout():
    """The flag barrier of the baselines is measurable for N = 2..64, and a
    rank that never signals makes both baselines time out like the others."""
    for n in (2, 8, 64):
        with rra.Comm(n, 4096) as comm:
            ns = comm.barrier_latency(200)
            assert 50.0 < ns < 1e6
            x = [torch.ones(1024, device="cuda") for _ in range(n)]
            y = poison_like(x)
            for algo in ("oneshot_barrier", "twoshot_barrier"):
                comm.allreduce(x, y, algo)
                torch.cuda.synchronize()
                assert comm.status()[0] == rra.OK
                assert torch.equal(y[n - 1], torch.full_like(y[0], float(n)))
                comm.set_attr("poll_timeout_ms", 20)
                comm.inject_drop(1)
                comm.allreduce(x, y, algo)
                assert comm.status()[0] == rra.ERR_TIMEOUT
                comm.reset()
                comm.set_attr("poll_timeout_ms", 1000)
                comm.allreduce(x, y, algo)
                torch.cuda.synchronize()
                assert comm.status()[0] == rra.OK


@pytest.mark.parametrize("algo", ALGOS)
def test_plain_launch_matches_cooperative(algo):
    """With the cooperative attribute off, the same occupancy-checked grid runs
    as a plain launch and gives the same results."""
    n, count = 4, 100000
    sends_np = inputs.normal(inputs.rng(74, 0), n, count, "fp32")
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("cooperative", 0)
        sends = to_device(sends_np, "fp32")
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, algo)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", algo)


@pytest.mark.parametrize("algo", ALGOS + ("oneshot_barrier", "twoshot_barrier"))
def test_programmatic_dependent_launch(algo):
    """With programmatic dependent launch each kernel waits for its
    predecessor before touching memory: back-to-back calls (stream and graph)
    stay exact."""
    n, count, calls = 4, 20000, 12
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("pdl", 1)
        for coop in (1, 0):
            comm.set_attr("cooperative", coop)
            host = [inputs.normal(inputs.rng(75, coop, i), n, count, "fp32") for i in range(calls)]
            send = [to_device(h, "fp32") for h in host]
            recv = [poison_like(s) for s in send]
            for i in range(calls):
                comm.allreduce(send[i], recv[i], algo)
            torch.cuda.synchronize()
            assert comm.status()[0] == rra.OK
            for i in range(calls):
                check_against_oracle(host[i], to_host(recv[i], "fp32"), "fp32", algo)
