"""GPU parity of ReduceScatter, AllGather, Broadcast and Reduce (through
distributed shared memory) against the oracle, bit for bit: every rank,
every dtype, ragged and unaligned block sizes, several roots, in place,
CUDA-graph replay, a dropped rank, and argument errors; up to 16 ranks one
CTA per rank, above that 16-CTA clusters whose CTAs act for several ranks."""
import numpy as np
import pytest

import oracle
from latency_barrier_free_gb300 import inputs, rra
from tests.gpu_util import ELEM, bits, poison_like, to_device, to_host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

COUNTS = (1, 3, 5, 33, 4096, 4097, 20000, 20001)  # 4096, 20000: blocks of whole 16-byte vectors


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _same_bits(got, expect, what):
    g, w = bits(got), bits(expect)
    bad = np.nonzero(g != w)[0]
    if bad.size:
        poison = np.frombuffer(b"\x7f" * g.itemsize, dtype=g.dtype)[0]
        raise AssertionError("%r: %d of %d elements differ, first at %s; got %s expect %s; %d still poison" % (
            what, bad.size, g.size, bad[:8].tolist(), [hex(int(v)) for v in g[bad[:4]]],
            [hex(int(v)) for v in w[bad[:4]]], int((g[bad] == poison).sum())))


def _run(comm, op, sends_np, out_count, dtype, root=0, send_mask=None, recv_mask=None):
    """Device copies of sends_np, poisoned outputs of out_count elements;
    entries masked off are passed as NULL.  Returns host outputs (None where
    masked) and the poisoned pattern for untouched checks."""
    n = len(sends_np)
    sends = to_device(sends_np, dtype)
    tdt = sends[0].dtype
    recvs = [torch.empty(out_count, dtype=tdt, device="cuda") for _ in range(n)]
    for t in recvs:
        t.view(torch.uint8).fill_(0x7F)
    sp = [None if send_mask and not send_mask[r] else sends[r].data_ptr() for r in range(n)]
    rp = [None if recv_mask and not recv_mask[r] else recvs[r].data_ptr() for r in range(n)]
    count = out_count if op != "all_gather" else out_count // n
    if op == "reduce":
        count = sends_np[0].size
    comm.collective_ptrs(op, sp, rp, count, dtype, root)
    torch.cuda.synchronize()
    st, rk, step = comm.status()
    assert st == rra.OK, "%s: %s (rank %d step %d)" % (op, rra.STATUS_NAMES.get(st), rk, step)
    return to_host(recvs, dtype)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [2, 3, 4, 8, 16, 17, 33, 64])
def test_reduce_scatter(n, dtype):
    with rra.Comm(n, n * max(COUNTS) * ELEM[dtype]) as comm:
        for count in COUNTS:
            sends_np = inputs.normal(inputs.rng(80, count, n), n, n * count, dtype)
            got = _run(comm, "reduce_scatter", sends_np, count, dtype)
            expect = oracle.reduce_scatter(sends_np, dtype)
            for r in range(n):
                _same_bits(got[r], expect[r], (count, r))


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [2, 3, 4, 8, 16, 17, 33, 64])
def test_all_gather(n, dtype):
    with rra.Comm(n, n * max(COUNTS) * ELEM[dtype]) as comm:
        for count in COUNTS:
            sends_np = inputs.normal(inputs.rng(81, count, n), n, count, dtype)
            got = _run(comm, "all_gather", sends_np, n * count, dtype)
            expect = oracle.all_gather(sends_np, dtype)
            for r in range(n):
                _same_bits(got[r], expect[r], (count, r))


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [2, 3, 8, 16, 17, 64])
def test_broadcast(n, dtype):
    """Only send[root] is passed; the other send entries are NULL."""
    with rra.Comm(n, max(COUNTS) * ELEM[dtype]) as comm:
        for count in COUNTS:
            for root in sorted({0, n // 2, n - 1}):
                sends_np = inputs.normal(inputs.rng(82, count, n, root), n, count, dtype)
                got = _run(comm, "broadcast", sends_np, count, dtype, root,
                           send_mask=[r == root for r in range(n)])
                expect = oracle.broadcast(sends_np, dtype, root)
                for r in range(n):
                    _same_bits(got[r], expect[r], (count, root, r))


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [2, 3, 8, 16, 17, 64])
def test_reduce(n, dtype):
    """recv[root] is the oracle's sum; the other outputs keep their poison
    (one run passes them, one passes NULL)."""
    with rra.Comm(n, max(COUNTS) * ELEM[dtype]) as comm:
        for count in COUNTS:
            for root in sorted({0, n - 1, 16 % n}):
                sends_np = inputs.normal(inputs.rng(83, count, n, root), n, count, dtype)
                expect = oracle.reduce(sends_np, dtype, root)[root]
                got = _run(comm, "reduce", sends_np, count, dtype, root)
                _same_bits(got[root], expect, (count, root))
                poison = np.full(got[0].nbytes, 0x7F, np.uint8)
                for r in range(n):
                    if r != root:
                        assert np.array_equal(got[r].view(np.uint8), poison), (count, root, r)
                got = _run(comm, "reduce", sends_np, count, dtype, root, recv_mask=[r == root for r in range(n)])
                _same_bits(got[root], expect, (count, root, "null"))


@pytest.mark.parametrize("split", [1, -1])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [2, 3, 4, 8, 16])
def test_two_hop_broadcast_and_reduce(n, dtype, split):
    """Broadcast and Reduce in two hops (forced, and chosen automatically for
    a message of at least 256 KiB): the same bits as the oracle; ragged
    parts; Broadcast with NULL non-root inputs, Reduce with NULL non-root
    outputs."""
    big = (300 << 10) // ELEM[dtype]
    counts = (1, 5, 33, 4097, 20001, big) if split == 1 else (big,)
    with rra.Comm(n, big * ELEM[dtype]) as comm:
        comm.set_attr("coll_split", split)
        for count in counts:
            for root in sorted({0, n - 1}):
                sends_np = inputs.normal(inputs.rng(89, count, n, root), n, count, dtype)
                got = _run(comm, "broadcast", sends_np, count, dtype, root,
                           send_mask=[r == root for r in range(n)])
                expect = oracle.broadcast(sends_np, dtype, root)
                for r in range(n):
                    _same_bits(got[r], expect[r], ("bc", count, root, r))
                got = _run(comm, "reduce", sends_np, count, dtype, root, recv_mask=[r == root for r in range(n)])
                _same_bits(got[root], oracle.reduce(sends_np, dtype, root)[root], ("rd", count, root))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_reduce_scatter_then_all_gather_is_allreduce(dtype):
    """AllGather(ReduceScatter(x)) equals the fixed-order AllReduce bit for
    bit on the GPU too (the composition of Sec. III-A)."""
    n, count = 4, 3001
    sends_np = inputs.normal(inputs.rng(84, 0), n, n * count, dtype)
    with rra.Comm(n, n * count * ELEM[dtype]) as comm:
        sends = to_device(sends_np, dtype)
        mids = [torch.empty(count, dtype=sends[0].dtype, device="cuda") for _ in range(n)]
        outs = poison_like(sends)
        comm.reduce_scatter(sends, mids)
        comm.all_gather(mids, outs)
        ar = poison_like(sends)
        comm.allreduce(sends, ar, "twoshot_cluster")
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        for a, b in zip(to_host(outs, dtype), to_host(ar, dtype)):
            _same_bits(a, b, "RS+AG vs AR")


@pytest.mark.parametrize("n", [4, 33])
@pytest.mark.parametrize("dtype", ["fp32", "fp64"])
def test_in_place(dtype, n):
    """ReduceScatter into recv[r] = send[r] + r*count and AllGather from
    send[r] = recv[r] + r*count (16-byte aligned blocks)."""
    count = 2048
    with rra.Comm(n, n * count * ELEM[dtype]) as comm:
        sends_np = inputs.normal(inputs.rng(85, 0), n, n * count, dtype)
        bufs = to_device(sends_np, dtype)
        comm.reduce_scatter(bufs, [bufs[r][r * count:(r + 1) * count] for r in range(n)])
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        expect = oracle.reduce_scatter(sends_np, dtype)
        for r, b in enumerate(to_host(bufs, dtype)):
            _same_bits(b[r * count:(r + 1) * count], expect[r], ("rs", r))
        ag_np = inputs.normal(inputs.rng(85, 1), n, count, dtype)
        bufs = [torch.empty(n * count, dtype=bufs[0].dtype, device="cuda") for _ in range(n)]
        for r in range(n):
            bufs[r][r * count:(r + 1) * count].copy_(to_device([ag_np[r]], dtype)[0])
        comm.all_gather([bufs[r][r * count:(r + 1) * count] for r in range(n)], bufs)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        expect = oracle.all_gather(ag_np, dtype)
        for r, b in enumerate(to_host(bufs, dtype)):
            _same_bits(b, expect[r], ("ag", r))


@pytest.mark.parametrize("n", [4, 40])
@pytest.mark.parametrize("op", rra.COLLECTIVES)
@pytest.mark.parametrize("slice_bytes", [16, 4096, 96 << 10])
def test_slice_sizes(op, slice_bytes, n):
    """From one vector per slice to the full stage (several input batches
    per thread, ragged last slice; the planner clips a slice to the stage)."""
    count, dtype = 30001 if n <= 16 else 3001, "fp32"
    with rra.Comm(n, n * count * 4) as comm:
        comm.set_attr("cluster_slice", slice_bytes)
        if op == "reduce_scatter":
            sends_np = inputs.normal(inputs.rng(86, slice_bytes), n, n * count, dtype)
            got, expect = _run(comm, op, sends_np, count, dtype), oracle.reduce_scatter(sends_np, dtype)
        elif op == "all_gather":
            sends_np = inputs.normal(inputs.rng(86, slice_bytes), n, count, dtype)
            got, expect = _run(comm, op, sends_np, n * count, dtype), oracle.all_gather(sends_np, dtype)
        elif op == "broadcast":
            sends_np = inputs.normal(inputs.rng(86, slice_bytes), n, count, dtype)
            got, expect = _run(comm, op, sends_np, count, dtype, 1), oracle.broadcast(sends_np, dtype, 1)
        else:
            sends_np = inputs.normal(inputs.rng(86, slice_bytes), n, count, dtype)
            got = _run(comm, op, sends_np, count, dtype, 2)
            expect = oracle.reduce(sends_np, dtype, 2)
            got, expect = got[2:3], expect[2:3]
        for g, e in zip(got, expect):
            _same_bits(g, e, (op, slice_bytes))


@pytest.mark.parametrize("n", [4, 24])
def test_graph_replay(n):
    """All four collectives captured in one CUDA graph, replayed with new
    inputs: every replay's results match the oracle."""
    count, dtype = 5000, "fp32"
    with rra.Comm(n, n * count * 4) as comm:
        rs_in = [torch.empty(n * count, device="cuda") for _ in range(n)]
        rs_out = [torch.empty(count, device="cuda") for _ in range(n)]
        x = [torch.empty(count, device="cuda") for _ in range(n)]
        ag_out = [torch.empty(n * count, device="cuda") for _ in range(n)]
        bc_out = [torch.empty(count, device="cuda") for _ in range(n)]
        rd_out = [torch.empty(count, device="cuda") for _ in range(n)]

        def enqueue():
            comm.reduce_scatter(rs_in, rs_out)
            comm.all_gather(x, ag_out)
            comm.broadcast(x, bc_out, 3)
            comm.reduce(x, rd_out, 1)

        enqueue()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                enqueue()
        for rep in range(3):
            a = inputs.normal(inputs.rng(87, rep, 0), n, n * count, dtype)
            b = inputs.normal(inputs.rng(87, rep, 1), n, count, dtype)
            for r in range(n):
                rs_in[r].copy_(torch.from_numpy(a[r]))
                x[r].copy_(torch.from_numpy(b[r]))
            g.replay()
            torch.cuda.synchronize()
            assert comm.status()[0] == rra.OK
            for r in range(n):
                _same_bits(rs_out[r].cpu().numpy(), oracle.reduce_scatter(a, dtype)[r], ("rs", rep))
                _same_bits(ag_out[r].cpu().numpy(), oracle.all_gather(b, dtype)[r], ("ag", rep))
                _same_bits(bc_out[r].cpu().numpy(), oracle.broadcast(b, dtype, 3)[r], ("bc", rep))
            _same_bits(rd_out[1].cpu().numpy(), oracle.reduce(b, dtype, 1)[1], ("rd", rep))


@pytest.mark.parametrize("n,split", [(4, 0), (4, 1), (20, -1)])
@pytest.mark.parametrize("op", rra.COLLECTIVES)
def test_dropped_rank_times_out_and_reset(op, n, split):
    """A rank that skips its pushes makes its receivers' bounded waits run
    out: RRA_ERR_TIMEOUT, no hang; after a reset the call is correct (one-
    and two-hop Broadcast / Reduce; at 20 ranks the dropped rank shares
    its CTA with another)."""
    count, dtype = 3000, "fp32"
    root = 0
    drop = n - 2 if op != "broadcast" else root  # a Broadcast's only first-hop sender is the root
    with rra.Comm(n, n * count * 4) as comm:
        comm.set_attr("coll_split", split)
        comm.set_attr("poll_timeout_ms", 20)
        comm.inject_drop(drop)
        m = n * count if op == "reduce_scatter" else count
        sends_np = inputs.normal(inputs.rng(88, 0), n, m, dtype)
        sends = to_device(sends_np, dtype)
        out = count if op != "all_gather" else n * count
        recvs = [torch.empty(out, device="cuda") for _ in range(n)]
        cnt = sends[0].numel() if op in ("all_gather", "reduce") else out
        comm.collective_ptrs(op, [t.data_ptr() for t in sends], [t.data_ptr() for t in recvs], cnt, dtype, root)
        st, rank, _ = comm.status()
        assert st == rra.ERR_TIMEOUT
        assert 0 <= rank < n
        comm.reset()
        comm.collective_ptrs(op, [t.data_ptr() for t in sends], [t.data_ptr() for t in recvs], cnt, dtype, root)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        got = to_host(recvs, dtype)
        expect = {"reduce_scatter": lambda: oracle.reduce_scatter(sends_np, dtype),
                  "all_gather": lambda: oracle.all_gather(sends_np, dtype),
                  "broadcast": lambda: oracle.broadcast(sends_np, dtype, root),
                  "reduce": lambda: oracle.reduce(sends_np, dtype, root)}[op]()
        ranks = [root] if op == "reduce" else range(n)
        for r in ranks:
            _same_bits(got[r], expect[r], (op, r))


def test_argument_errors():
    with rra.Comm(4, 4096) as comm:
        x = [torch.zeros(1024, device="cuda") for _ in range(4)]
        p = [t.data_ptr() for t in x]
        for bad_root in (-1, 4):
            for op in ("broadcast", "reduce"):
                with pytest.raises(rra.RraError):
                    comm.collective_ptrs(op, p, p, 16, "fp32", bad_root)
        with pytest.raises(rra.RraError):  # 4 blocks of 512 floats exceed 4096 bytes
            comm.collective_ptrs("reduce_scatter", p, p, 512, "fp32")
        with pytest.raises(rra.RraError):  # a NULL input that the collective needs
            comm.collective_ptrs("all_gather", [None] + p[1:], p, 16, "fp32")
        with pytest.raises(rra.RraError):  # misaligned
            comm.collective_ptrs("broadcast", [p[0] + 4] + p[1:], p, 16, "fp32", 0)
        for op in rra.COLLECTIVES:  # count 0: nothing launched, nothing checked on the device
            comm.collective_ptrs(op, p, p, 0, "fp32", 0)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
