"""GPU parity: the CUDA AllReduce through the C ABI against the CPU oracle.

Fixed-order algorithms (one-shot LL, one-shot sentinel, two-shot) must match
the oracle bit for bit; LL128-atomic must stay within N 2^-23 sum|x| (binary32)
and every rank must receive the same bits.  Inputs come from the seeded
workload generators (latency_barrier_free_gb300.inputs).
"""
import numpy as np
import pytest

import oracle
from latency_barrier_free_gb300 import inputs, rra
from tests.gpu_util import ALGOS, CLUSTER, ELEM, FIXED_ORDER, bits, check_against_oracle, poison_like, to_device, to_host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def run(comm, sends_np, dtype, algo, in_place=False):
    sends = to_device(sends_np, dtype)
    recvs = sends if in_place else poison_like(sends)
    comm.allreduce(sends, recvs, algo)
    torch.cuda.synchronize()
    st, rk, step = comm.status()
    assert st == rra.OK, "%s: device status %s (rank %d step %d)" % (algo, rra.STATUS_NAMES.get(st), rk, step)
    return to_host(recvs, dtype)


# ---------------------------------------------------------------- workload 1
@pytest.mark.parametrize("algo", ["oneshot_ll", "oneshot_sentinel", "oneshot_cluster", "twoshot_cluster"])
def test_workload1_1000_back_to_back(algo):
    """N=2, 32 binary32 integers in [-8, 8], a fresh draw for each of 1000
    back-to-back calls (distinct buffers, one stream): every result exact."""
    iters = 1000
    host = np.stack([np.stack(inputs.workload1(i)) for i in range(iters)])  # [iters, 2, 32]
    send = torch.from_numpy(host).cuda()
    recv = torch.full_like(send, float("nan"))
    with rra.Comm(2, 128) as comm:
        for i in range(iters):
            comm.allreduce_ptrs([send[i, 0].data_ptr(), send[i, 1].data_ptr()],
                                [recv[i, 0].data_ptr(), recv[i, 1].data_ptr()], 32, "fp32", algo)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
    got = recv.cpu().numpy()
    exact = host.astype(np.int64).sum(axis=1)  # integer sums, exact
    for i in range(iters):
        for r in range(2):
            assert np.array_equal(got[i, r], exact[i].astype(np.float32)), (i, r)


@pytest.mark.parametrize("algo", ["oneshot_ll", "oneshot_sentinel", "twoshot_cluster"])
def test_workload1_same_buffers(algo):
    """1000 calls reusing one send/recv pair, new inputs copied in between."""
    with rra.Comm(2, 128) as comm:
        send = [torch.empty(32, device="cuda") for _ in range(2)]
        recv = [torch.empty(32, device="cuda") for _ in range(2)]
        for i in range(1000):
            x = inputs.workload1(i)
            for r in range(2):
                send[r].copy_(torch.from_numpy(x[r]))
            comm.allreduce(send, recv, algo)
            if i % 97 == 0 or i == 999:
                expect = x[0].astype(np.int64) + x[1].astype(np.int64)
                for r in range(2):
                    assert np.array_equal(recv[r].cpu().numpy(), expect.astype(np.float32)), (i, r)
        assert comm.status()[0] == rra.OK


# ---------------------------------------------------------------- workload 2
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("algo", ALGOS + CLUSTER)
def test_workload2_size_sweep(algo, dtype):
    """N=4, 128 B .. 1 MiB per rank, N(0,1) inputs."""
    with rra.Comm(4, 1 << 20) as comm:
        for size in inputs.W2_SIZES:
            sends_np = inputs.workload2(size, dtype)
            got = run(comm, sends_np, dtype, algo)
            check_against_oracle(sends_np, got, dtype, algo)


# ---------------------------------------------------------------- workload 4
@pytest.mark.parametrize("algo", ALGOS)
def test_workload4_64_ranks(algo):
    """N=64, binary32 N(0,1), 1 KiB .. 256 KiB per rank."""
    with rra.Comm(64, 256 << 10) as comm:
        for size in inputs.W4_SIZES:
            sends_np = inputs.workload4(size, 64)
            got = run(comm, sends_np, "fp32", algo)
            check_against_oracle(sends_np, got, "fp32", algo)


@pytest.mark.parametrize("algo", ["ll128_atomic", "oneshot_sentinel"])
def test_workload4_rank_sweep(algo):
    """N in {2, 4, 8, 16, 32, 64} at 16 KiB per rank."""
    for n in inputs.W4_NSWEEP:
        with rra.Comm(n, 16 << 10) as comm:
            sends_np = inputs.workload4(16 << 10, n)
            got = run(comm, sends_np, "fp32", algo)
            check_against_oracle(sends_np, got, "fp32", algo)


# ------------------------------------------------------------- edge cases
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("algo", ALGOS + CLUSTER)
def test_ragged_counts_and_odd_ranks(algo, dtype):
    """Counts that are not a multiple of a 16-byte vector, odd N."""
    for n in (2, 3, 5):
        with rra.Comm(n, 8192 * ELEM[dtype]) as comm:
            for count in (1, 2, 3, 5, 7, 9, 33, 255, 1001, 4097, 8191):
                sends_np = inputs.normal(inputs.rng(60, count, n), n, count, dtype)
                got = run(comm, sends_np, dtype, algo)
                check_against_oracle(sends_np, got, dtype, algo)


@pytest.mark.parametrize("algo", ALGOS + CLUSTER)
def test_count_zero_is_noop(algo):
    with rra.Comm(4, 1024) as comm:
        x = [torch.ones(4, device="cuda") for _ in range(4)]
        comm.allreduce_ptrs([t.data_ptr() for t in x], [t.data_ptr() for t in x], 0, "fp32", algo)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        assert all(torch.equal(t, torch.ones(4, device="cuda")) for t in x)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("algo", ALGOS + CLUSTER)
def test_in_place(algo, dtype):
    with rra.Comm(4, 1 << 16) as comm:
        for count in (7, 1000, (1 << 16) // ELEM[dtype]):
            sends_np = inputs.normal(inputs.rng(61, count), 4, count, dtype)
            got = run(comm, sends_np, dtype, algo, in_place=True)
            check_against_oracle(sends_np, got, dtype, algo)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("algo", ALGOS + CLUSTER)
def test_closed_form_every_dtype(algo, dtype):
    """Rank r filled with r + 1 sums to N(N+1)/2 (exact for these N)."""
    for n in (2, 4, 8):
        count = 4096 + 3
        with rra.Comm(n, count * ELEM[dtype]) as comm:
            got = run(comm, inputs.rank_plus_one(n, count, dtype), dtype, algo)
            expect = oracle.allreduce(inputs.rank_plus_one(n, count, dtype), dtype)
            for g in got:
                assert np.array_equal(bits(g), bits(expect[0]))


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("ctas", [1, 2, 3, 7])
@pytest.mark.parametrize("threads", [64, 256])
def test_many_steps_credit_chain(algo, ctas, threads):
    """Small chunks force many double-buffered steps per call (>= 3, so the
    step fences and the receive-as-credit chain are exercised), with several
    CTAs per rank and a ragged last step."""
    n, dtype = 4, "fp32"
    count = 40000 + 13
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("ctas_per_rank", ctas)
        comm.set_attr("threads", threads)
        comm.set_attr("oneshot_chunk", 2048)
        comm.set_attr("twoshot_chunk", 4096)
        comm.set_attr("ll128_chunk", 4096)
        _, steps = comm.plan_call(count, dtype, algo)
        assert steps >= 3
        for it in range(3):
            sends_np = inputs.normal(inputs.rng(62, it, ctas, threads), n, count, dtype)
            got = run(comm, sends_np, dtype, algo)
            check_against_oracle(sends_np, got, dtype, algo)


def test_mixed_algorithms_interleaved():
    """Alternate all algorithms and dtypes on one communicator, 70 calls
    enqueued back to back, all checked at the end."""
    n = 4
    rng_sizes = np.random.Generator(np.random.PCG64(5))
    with rra.Comm(n, 1 << 18) as comm:
        pending = []
        for i in range(70):
            algo = (ALGOS + CLUSTER)[i % len(ALGOS + CLUSTER)]
            dtype = ("fp32", "bf16", "fp64")[i % 3]
            count = int(rng_sizes.integers(1, (1 << 18) // ELEM[dtype]))
            sends_np = inputs.normal(inputs.rng(63, i), n, count, dtype)
            sends = to_device(sends_np, dtype)
            recvs = poison_like(sends)
            comm.allreduce(sends, recvs, algo)
            pending.append((sends_np, sends, recvs, dtype, algo))
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        for sends_np, _, recvs, dtype, algo in pending:
            check_against_oracle(sends_np, to_host(recvs, dtype), dtype, algo)


def test_inputs_equal_to_rank_index_pattern_fp64_halves():
    """binary64 values whose low 32 bits are all ones must not be mistaken for
    the sentinel (the sentinel test is per 64-bit value)."""
    n, count = 4, 1000
    vals = []
    for r in range(n):
        u = np.full(count, 0x3FF00000FFFFFFFF + r, dtype=np.uint64)
        u[::2] = 0xBFF00001FFFFFFFF
        vals.append(u.view(np.float64))
    with rra.Comm(n, count * 8) as comm:
        for algo in ALGOS:
            got = run(comm, vals, "fp64", algo)
            check_against_oracle(vals, got, "fp64", algo)


@pytest.mark.parametrize("algo", ["oneshot_ll", "oneshot_sentinel"])
@pytest.mark.parametrize("wide", [0, 1])
@pytest.mark.parametrize("n", [2, 5, 16, 64])
def test_oneshot_wide_and_narrow_variants(algo, wide, n):
    """Both one-shot receive variants (thread per position / threads split a
    position's sources and stage in shared memory) give the oracle's bits,
    single-step and multi-step, for every dtype."""
    for dtype, counts in (("fp32", (1, 33, 4097, 70001)), ("bf16", (7, 5000)), ("fp64", (3, 3001))):
        with rra.Comm(n, 70001 * 4) as comm:
            comm.set_attr("oneshot_wide", wide)
            for count in counts:
                sends_np = inputs.normal(inputs.rng(64, count, n, wide), n, count, dtype)
                got = run(comm, sends_np, dtype, algo)
                check_against_oracle(sends_np, got, dtype, algo)
            comm.set_attr("oneshot_chunk", 1024)
            comm.set_attr("ctas_per_rank", 2)
            count = 20000 // ELEM[dtype] * 4 + 5
            _, steps = comm.plan_call(count, dtype, algo)
            assert steps >= 3
            sends_np = inputs.normal(inputs.rng(65, n, wide), n, count, dtype)
            got = run(comm, sends_np, dtype, algo)
            check_against_oracle(sends_np, got, dtype, algo)


@pytest.mark.parametrize("wide", [0, 1])
@pytest.mark.parametrize("n", [2, 5, 16, 64])
def test_ll128_wide_and_narrow_variants(wide, n):
    """Both LL128-atomic variants (a thread walks a position's owners / the
    CTA's threads split the (owner, position) items of the atomic adds and
    of the AllGather polls) stay within the atomic-order bound, single-step
    and multi-step, for every dtype; ragged partitions and tails."""
    for dtype, counts in (("fp32", (1, 33, 4097, 70001)), ("bf16", (7, 5000)), ("fp64", (3, 3001))):
        with rra.Comm(n, 70001 * 4) as comm:
            comm.set_attr("oneshot_wide", wide)
            for count in counts:
                sends_np = inputs.normal(inputs.rng(66, count, n, wide), n, count, dtype)
                got = run(comm, sends_np, dtype, "ll128_atomic")
                check_against_oracle(sends_np, got, dtype, "ll128_atomic")
            comm.set_attr("ll128_chunk", 16 * 40 * n)  # 40 positions per owner and step
            comm.set_attr("ctas_per_rank", 2)
            count = 16 * 40 * n * 3 // ELEM[dtype] + 5
            _, steps = comm.plan_call(count, dtype, "ll128_atomic")
            assert steps >= 3
            sends_np = inputs.normal(inputs.rng(67, n, wide), n, count, dtype)
            got = run(comm, sends_np, dtype, "ll128_atomic")
            check_against_oracle(sends_np, got, dtype, "ll128_atomic")


@pytest.mark.parametrize("algo", ["oneshot_barrier", "twoshot_barrier"])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
def test_barrier_baseline_parity(dtype, algo):
    """The barrier-based baselines (plain stores + two flag barriers per step)
    add in rank order too, so they are bit-exact against the oracle; several
    steps, several CTAs per rank, ragged partitions, in place."""
    for n in (2, 4, 7, 64):
        with rra.Comm(n, 70000 * ELEM[dtype]) as comm:
            for count in (1, 33, 4097, 70000):
                sends_np = inputs.normal(inputs.rng(66, count, n), n, count, dtype)
                got = run(comm, sends_np, dtype, algo)
                check_against_oracle(sends_np, got, dtype, algo)
            comm.set_attr("oneshot_chunk", 1024)
            comm.set_attr("twoshot_chunk", 16 * 8 * n)  # partitions of 8 vectors
            comm.set_attr("ctas_per_rank", 3)
            sends_np = inputs.normal(inputs.rng(67, n), n, 9000, dtype)
            assert comm.plan_call(9000, dtype, algo)[1] >= 3
            got = run(comm, sends_np, dtype, algo)
            check_against_oracle(sends_np, got, dtype, algo)
            got = run(comm, sends_np, dtype, algo, in_place=True)
            check_against_oracle(sends_np, got, dtype, algo)


@pytest.mark.parametrize("n", [2, 4, 8, 16, 64])
def test_auto_algorithm(n):
    """RRA_AUTO runs the algorithm rra_select_algo names, with its results."""
    max_bytes = 1 << 20
    with rra.Comm(n, max_bytes) as comm:
        for size in (128, 4096, 65536, 262144, 393216, 524288, 1 << 20):
            count = size // 4
            algo = rra.select_algo(n, size, "fp32")
            sends_np = inputs.normal(inputs.rng(68, n, size), n, count, "fp32")
            got = run(comm, sends_np, "fp32", "auto")
            check_against_oracle(sends_np, got, "fp32", algo)


@pytest.mark.parametrize("algo", CLUSTER)
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [2, 3, 4, 8, 16, 17, 32, 64])
def test_cluster_kernels(n, dtype, algo):
    """One-shot and two-shot through distributed shared memory (one cluster
    of N CTAs per slice) with st.async pushes: bit-exact, for ragged sizes
    (two-shot partitions that are partly or wholly empty), many slices, and
    in place.  (The bulk-copy push, on by default, has its own test.)"""
    with rra.Comm(n, 300000 * ELEM[dtype]) as comm:
        comm.set_attr("cluster_tma", 0)
        for count in (1, 7, 33, 4097, 70001, 300000):
            sends_np = inputs.normal(inputs.rng(69, count, n), n, count, dtype)
            got = run(comm, sends_np, dtype, algo)
            check_against_oracle(sends_np, got, dtype, algo)
        sends_np = inputs.normal(inputs.rng(69, 1, n), n, 5000, dtype)
        got = run(comm, sends_np, dtype, algo, in_place=True)
        check_against_oracle(sends_np, got, dtype, algo)


@pytest.mark.parametrize("algo", CLUSTER)
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [2, 3, 4, 8, 16, 17, 32, 64])
def test_cluster_kernels_bulk_copy_push(n, dtype, algo):
    """The cluster kernels with the push made by TMA bulk copies
    (RRA_ATTR_CLUSTER_TMA; above 16 ranks one copy per hosted rank and
    owner): bit-exact for ragged sizes (a last vector only partly inside
    the input; empty two-shot partitions), several slice sizes, and in
    place."""
    with rra.Comm(n, 300000 * ELEM[dtype]) as comm:
        comm.set_attr("cluster_tma", 1)
        for count in (1, 7, 33, 4097, 70001, 300000):
            sends_np = inputs.normal(inputs.rng(68, count, n), n, count, dtype)
            got = run(comm, sends_np, dtype, algo)
            check_against_oracle(sends_np, got, dtype, algo)
        for slice_bytes in (16 * n, 4096, 96 << 10):
            comm.set_attr("cluster_slice", slice_bytes)
            sends_np = inputs.normal(inputs.rng(68, slice_bytes, n), n, 20001, dtype)
            got = run(comm, sends_np, dtype, algo)
            check_against_oracle(sends_np, got, dtype, algo)
        comm.set_attr("cluster_slice", 0)
        sends_np = inputs.normal(inputs.rng(68, 1, n), n, 5000, dtype)
        got = run(comm, sends_np, dtype, algo, in_place=True)
        check_against_oracle(sends_np, got, dtype, algo)


@pytest.mark.parametrize("tma", [0, 1])
@pytest.mark.parametrize("algo", CLUSTER)
@pytest.mark.parametrize("threads", [64, 128, 256])
def test_cluster_slice_sizes(algo, threads, tma):
    """Slices from one vector per rank to the full 96 KiB stage, so that a
    thread pushes up to several batches of inputs; ragged last slice; with
    st.async pushes and with the bulk-copy push."""
    dtype = "fp32"
    for n in (2, 4, 16):
        count = 200000 + 5
        with rra.Comm(n, count * 4) as comm:
            comm.set_attr("threads", threads)
            comm.set_attr("cluster_tma", tma)
            for slice_bytes in (16, 16 * n, 4096, 48 << 10, 96 << 10):
                for pipe in ((0, 1) if algo == "twoshot_cluster" else (0,)):
                    comm.set_attr("cluster_slice", slice_bytes)
                    comm.set_attr("cluster_pipe", pipe)
                    grid, _ = comm.plan_call(count, dtype, algo)
                    assert grid % n == 0
                    sends_np = inputs.normal(inputs.rng(72, n, slice_bytes, threads, pipe, tma), n, count, dtype)
                    got = run(comm, sends_np, dtype, algo)
                    check_against_oracle(sends_np, got, dtype, algo)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [2, 3, 4, 8, 16])
@pytest.mark.parametrize("clusters", [1, 3, 0])
def test_cluster_twoshot_pipelined(n, dtype, clusters):
    """The persistent, double-buffered two-shot: one cluster looping over
    hundreds of slices (every buffer reused ~100 times, each reuse gated by
    the receivers' credits), three clusters, and as many as fit; ragged
    message tails and slices; bit-exact."""
    with rra.Comm(n, 70001 * ELEM[dtype]) as comm:
        comm.set_attr("cluster_pipe", 1)
        comm.set_attr("ctas_per_rank", clusters)
        comm.set_attr("cluster_slice", 16 * n * 4)
        for count in (70001, 5, 4097):
            grid, steps = comm.plan_call(count, dtype, "twoshot_cluster")
            if clusters:
                assert grid == n * min(clusters, steps)
            sends_np = inputs.normal(inputs.rng(73, count, n, clusters), n, count, dtype)
            got = run(comm, sends_np, dtype, "twoshot_cluster")
            check_against_oracle(sends_np, got, dtype, "twoshot_cluster")
        sends_np = inputs.normal(inputs.rng(73, 2, n, clusters), n, 70001, dtype)
        got = run(comm, sends_np, dtype, "twoshot_cluster", in_place=True)
        check_against_oracle(sends_np, got, dtype, "twoshot_cluster")


@pytest.mark.parametrize("algo", CLUSTER)
def test_cluster_rank_sweep(algo):
    """N in {2, 4, 8, 16} at 16 KiB and 1 MiB per rank (workload 4's sweep,
    up to the cluster limit)."""
    for n in (2, 4, 8, 16):
        with rra.Comm(n, 1 << 20) as comm:
            for size in (16 << 10, 1 << 20):
                sends_np = inputs.workload4(size, n)
                got = run(comm, sends_np, "fp32", algo)
                check_against_oracle(sends_np, got, "fp32", algo)


@pytest.mark.parametrize("algo", CLUSTER)
@pytest.mark.parametrize("n", [20, 33, 48])
def test_cluster_more_ranks_than_ctas(n, algo):
    """N > 16: clusters of 16 CTAs, CTA j hosting ranks j, j + 16, ...
    (uneven: some CTAs host one more rank); slices from one vector to the
    stage limit; bit-exact."""
    count = 50000 + 3
    with rra.Comm(n, count * 4) as comm:
        for slice_bytes in (0, 16 * 16, 4096):
            comm.set_attr("cluster_slice", slice_bytes)
            sends_np = inputs.normal(inputs.rng(76, n, slice_bytes), n, count, "fp32")
            got = run(comm, sends_np, "fp32", algo)
            check_against_oracle(sends_np, got, "fp32", algo)
