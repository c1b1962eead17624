"""GPU tests of where the bulk-copy push (TMA bulk copies with cluster
multicast, read straight from the callers' inputs) may run: only on inputs in
device memory of this GPU.  Host buffers -- the host entry points, and
device-mapped pinned host memory passed to the device entry points -- get the
st.async kernels, with the same results.  rra_comm_last_kernel names the
kernel each call launched."""
import numpy as np
import pytest

import oracle
from latency_barrier_free_gb300 import inputs, rra
from tests.gpu_util import bits, check_against_oracle, poison_like, to_device, to_host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _pinned(arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in arrs]


@pytest.mark.parametrize("algo,count", [("oneshot_cluster", 32), ("twoshot_cluster", 70000), ("auto", 32),
                                        ("auto", 300000)])
def test_device_buffers_take_the_bulk_copy_push(algo, count):
    n = 4
    sends_np = inputs.normal(inputs.rng(90, count), n, count, "fp32")
    with rra.Comm(n, count * 4) as comm:
        assert comm.last_kernel() == "none"
        sends = to_device(sends_np, "fp32")
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, algo)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        assert comm.last_kernel().startswith("cluster_tma_kernel<")
        assert comm.last_kernel() == comm.plan_kernel(count, "fp32", algo)
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", "oneshot_cluster")


@pytest.mark.parametrize("algo,count", [("oneshot_cluster", 32), ("twoshot_cluster", 70000), ("auto", 1000)])
def test_host_entry_never_takes_the_bulk_copy_push(algo, count):
    """rra_allreduce_host and rra_allreduce_mapped with the bulk-copy push
    switched on explicitly: the kernel reads host memory, so the push is
    st.async (cluster_kernel), and the sums are exact."""
    n = 4
    sends_np = inputs.normal(inputs.rng(91, count), n, count, "fp32")
    hs = _pinned(sends_np)
    hr = [torch.full((count,), float("nan")).pin_memory() for _ in range(n)]
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("cluster_tma", 1)
        comm.allreduce_host([t.data_ptr() for t in hs], [t.data_ptr() for t in hr], count, "fp32", algo)
        assert comm.last_kernel().startswith("cluster_kernel<"), comm.last_kernel()
        check_against_oracle(sends_np, [t.numpy() for t in hr], "fp32", "oneshot_cluster")
        for t in hr:
            t.fill_(float("nan"))
        call = comm.prepare_host([t.data_ptr() for t in hs], [t.data_ptr() for t in hr], count, "fp32", algo)
        call()
        assert comm.last_kernel().startswith("cluster_kernel<"), comm.last_kernel()
        check_against_oracle(sends_np, [t.numpy() for t in hr], "fp32", "oneshot_cluster")


def test_mapped_host_pointers_on_the_device_entry_get_st_async():
    """Device addresses of pinned host memory handed to rra_allreduce itself
    (not through the host entry) still fail the device-memory check."""
    n, count = 4, 4096
    sends_np = inputs.normal(inputs.rng(92, 0), n, count, "fp32")
    hs = _pinned(sends_np)
    dev_send = rra.host_device_ptrs([t.data_ptr() for t in hs])
    assert all(d is not None for d in dev_send)
    recvs = [torch.full((count,), float("nan"), device="cuda") for _ in range(n)]
    with rra.Comm(n, count * 4) as comm:
        comm.allreduce_ptrs(dev_send, [t.data_ptr() for t in recvs], count, "fp32", "oneshot_cluster")
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        assert comm.last_kernel() == "cluster_kernel<one-shot>"
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", "oneshot_cluster")
        # one rank's input on the device, the others in host memory: still st.async
        first = to_device([sends_np[0]], "fp32")[0]  # kept alive: the call reads it
        mixed = [first.data_ptr()] + dev_send[1:]
        comm.allreduce_ptrs(mixed, [t.data_ptr() for t in recvs], count, "fp32", "oneshot_cluster")
        torch.cuda.synchronize()
        assert comm.last_kernel() == "cluster_kernel<one-shot>"
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", "oneshot_cluster")


@pytest.mark.parametrize("n", [20, 64])
@pytest.mark.parametrize("algo,count", [("oneshot_cluster", 40), ("twoshot_cluster", 30001), ("auto", 64)])
def test_many_ranks_choose_their_push_by_source_memory(n, algo, count):
    """Above 16 ranks (16-CTA clusters, each CTA hosting several ranks):
    device inputs take the bulk copies, pinned host buffers and the
    attribute switched off the st.async pushes; every result exact."""
    sends_np = inputs.normal(inputs.rng(99, n, count), n, count, "fp32")
    with rra.Comm(n, count * 4) as comm:
        sends = to_device(sends_np, "fp32")
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, algo)
        torch.cuda.synchronize()
        assert comm.status()[0] == rra.OK
        kind = comm.last_kernel()
        assert kind.startswith("cluster_multi_kernel<") and kind.endswith(", bulk>"), kind
        assert kind == comm.plan_kernel(count, "fp32", algo)
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", "oneshot_cluster")
        hs = _pinned(sends_np)
        hr = [torch.full((count,), float("nan")).pin_memory() for _ in range(n)]
        comm.allreduce_host([t.data_ptr() for t in hs], [t.data_ptr() for t in hr], count, "fp32", algo)
        assert comm.last_kernel() == kind[:-len(", bulk>")] + ">", comm.last_kernel()
        check_against_oracle(sends_np, [t.numpy() for t in hr], "fp32", "oneshot_cluster")
        comm.set_attr("cluster_tma", 0)
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, algo)
        torch.cuda.synchronize()
        assert comm.last_kernel() == kind[:-len(", bulk>")] + ">", comm.last_kernel()
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", "oneshot_cluster")
        assert comm.status()[0] == rra.OK


def test_bulk_copy_attribute_off():
    n, count = 4, 32
    sends_np = inputs.normal(inputs.rng(93, 0), n, count, "fp32")
    with rra.Comm(n, count * 4) as comm:
        comm.set_attr("cluster_tma", 0)
        sends = to_device(sends_np, "fp32")
        recvs = poison_like(sends)
        comm.allreduce(sends, recvs, "oneshot_cluster")
        torch.cuda.synchronize()
        assert comm.last_kernel() == "cluster_kernel<one-shot>"
        check_against_oracle(sends_np, to_host(recvs, "fp32"), "fp32", "oneshot_cluster")


@pytest.mark.parametrize("m", [1000, 1024, 1025, 65536, 65537])
def test_collectives_choose_their_push_by_source_memory(m):
    """AllGather and Broadcast push by bulk copies from device inputs, by
    st.async from inputs in host memory; with device inputs and outputs and
    blocks of whole 16-byte vectors of at least 4 KiB (AllGather) or 256 KiB
    (Broadcast) they also write the outputs by bulk copies.  The results are
    the oracle's."""
    n = 4
    small_np = [inputs.normal(inputs.rng(94, r), 1, m, "fp32")[0] for r in range(n)]
    want_ag = oracle.all_gather(small_np, "fp32")
    want_bc = oracle.broadcast(small_np, "fp32", 2)
    hs = _pinned(small_np)
    dev_host = rra.host_device_ptrs([t.data_ptr() for t in hs])
    on_device = to_device(small_np, "fp32")  # kept alive: the calls read it
    store_ag = ", bulk store" if m % 4 == 0 and m * 4 >= 4096 else ""
    store_bc = ", bulk store" if m % 4 == 0 and m * 4 >= 262144 else ""
    with rra.Comm(n, n * m * 4) as comm:
        for where, src in (("device", [t.data_ptr() for t in on_device]), ("host", dev_host)):
            out = [torch.full((n * m,), float("nan"), device="cuda") for _ in range(n)]
            comm.collective_ptrs("all_gather", src, [t.data_ptr() for t in out], m, "fp32", 0)
            torch.cuda.synchronize()
            kind = comm.last_kernel()
            assert kind == ("coll_bulk_kernel<all_gather%s>" % store_ag if where == "device"
                            else "coll_kernel<all_gather>"), kind
            for g, w in zip(out, want_ag):
                assert np.array_equal(bits(g.cpu().numpy()), bits(w))
            bc = [torch.full((m,), float("nan"), device="cuda") for _ in range(n)]
            comm.collective_ptrs("broadcast", src, [t.data_ptr() for t in bc], m, "fp32", 2)
            torch.cuda.synchronize()
            kind = comm.last_kernel()
            if where == "device" and store_bc:
                want_kind = "coll_bulk_kernel<broadcast, bulk store>"
            elif m * 4 >= 262144:  # from 256 KiB a Broadcast without bulk stores takes two hops
                want_kind = "coll_split_kernel<broadcast>"
            else:
                want_kind = "coll_bulk_kernel<broadcast>" if where == "device" else "coll_kernel<broadcast>"
            assert kind == want_kind, kind
            for g, w in zip(bc, want_bc):
                assert np.array_equal(bits(g.cpu().numpy()), bits(w))
        assert comm.status()[0] == rra.OK


@pytest.mark.parametrize("m", [1000, 1001])
def test_reduce_scatter_chooses_its_push_by_source_memory(m):
    """ReduceScatter pushes by bulk copies (one per owner) from device inputs
    whose blocks are whole 16-byte vectors (m = 1000 fp32), by st.async
    otherwise and from host memory; the sums are the oracle's bits."""
    n = 4
    sends_np = inputs.normal(inputs.rng(97, m), n, n * m, "fp32")
    want = oracle.reduce_scatter(sends_np, "fp32")
    hs = _pinned(sends_np)
    dev_host = rra.host_device_ptrs([t.data_ptr() for t in hs])
    on_device = to_device(sends_np, "fp32")  # kept alive: the calls read it
    with rra.Comm(n, n * m * 4) as comm:
        for where, src in (("device", [t.data_ptr() for t in on_device]), ("host", dev_host)):
            out = [torch.full((m,), float("nan"), device="cuda") for _ in range(n)]
            comm.collective_ptrs("reduce_scatter", src, [t.data_ptr() for t in out], m, "fp32", 0)
            torch.cuda.synchronize()
            kind = comm.last_kernel()
            bulk = where == "device" and m % 4 == 0
            assert kind == ("coll_bulk_kernel<reduce_scatter>" if bulk else "coll_kernel<reduce_scatter>"), kind
            for g, w in zip(out, want):
                assert np.array_equal(bits(g.cpu().numpy()), bits(w))
        assert comm.status()[0] == rra.OK


@pytest.mark.parametrize("m", [1000, 1001, 1024, 70001, 70000])
def test_reduce_chooses_its_push_by_source_memory(m):
    """Reduce pushes partition q of every rank's slice to CTA q by bulk
    copies from device inputs (any count: each input starts aligned), the
    owners storing their sums into the root's output; from host memory it
    keeps the st.async kernels (two hops from 256 KiB).  The sums are the
    oracle's bits."""
    n, root = 4, 2
    sends_np = inputs.normal(inputs.rng(98, m), n, m, "fp32")
    want = oracle.reduce(sends_np, "fp32", root)
    hs = _pinned(sends_np)
    dev_host = rra.host_device_ptrs([t.data_ptr() for t in hs])
    on_device = to_device(sends_np, "fp32")  # kept alive: the calls read it
    with rra.Comm(n, m * 4) as comm:
        for where, src in (("device", [t.data_ptr() for t in on_device]), ("host", dev_host)):
            out = [torch.full((m,), float("nan"), device="cuda") for _ in range(n)]
            comm.collective_ptrs("reduce", src, [t.data_ptr() for t in out], m, "fp32", root)
            torch.cuda.synchronize()
            kind = comm.last_kernel()
            if where == "device":
                assert kind == "coll_bulk_kernel<reduce>", kind
            else:
                assert kind == ("coll_split_kernel<reduce>" if m * 4 >= 262144 else "coll_kernel<reduce>"), kind
            assert np.array_equal(bits(out[root].cpu().numpy()), bits(want[root]))
            for r in range(n):  # only the root's output is written
                if r != root:
                    assert torch.isnan(out[r]).all()
        assert comm.status()[0] == rra.OK


@pytest.mark.parametrize("n", [20, 64])
@pytest.mark.parametrize("m", [1000, 1001])
def test_many_rank_collectives_choose_their_push(n, m):
    """Above 16 ranks all four collectives push by bulk copies from device
    inputs (ReduceScatter only for blocks of whole 16-byte vectors), by
    st.async with the attribute off; the results are the oracle's bits."""
    root = n - 3
    rs_np = inputs.normal(inputs.rng(100, n, m), n, n * m, "fp32")
    one_np = inputs.normal(inputs.rng(101, n, m), n, m, "fp32")
    want = {"reduce_scatter": oracle.reduce_scatter(rs_np, "fp32"), "all_gather": oracle.all_gather(one_np, "fp32"),
            "broadcast": oracle.broadcast(one_np, "fp32", root), "reduce": oracle.reduce(one_np, "fp32", root)}
    rs_dev = to_device(rs_np, "fp32")
    one_dev = to_device(one_np, "fp32")
    with rra.Comm(n, n * m * 4) as comm:
        for tma in (-1, 0):
            comm.set_attr("cluster_tma", tma)
            for op in rra.COLLECTIVES:
                src = rs_dev if op == "reduce_scatter" else one_dev
                out_n = n * m if op == "all_gather" else m
                out = [torch.full((out_n,), float("nan"), device="cuda") for _ in range(n)]
                comm.collective_ptrs(op, [t.data_ptr() for t in src], [t.data_ptr() for t in out], m, "fp32", root)
                torch.cuda.synchronize()
                bulk = tma != 0 and (op != "reduce_scatter" or m % 4 == 0)
                kind = comm.last_kernel()
                want_kind = "coll_reduce_multi_bulk_kernel" if (bulk and op == "reduce") else \
                    "coll_multi_kernel<%s%s>" % (op, ", bulk" if bulk else "")
                assert kind == want_kind, kind
                ranks = [root] if op == "reduce" else range(n)
                for r in ranks:
                    assert np.array_equal(bits(out[r].cpu().numpy()), bits(want[op][r])), (op, tma, r)
        assert comm.status()[0] == rra.OK


def test_many_rank_bulk_stores():
    """Above 16 ranks, AllGather (4 KiB blocks) and Broadcast (256 KiB) on
    device buffers write their outputs by bulk copies too; the results are
    the oracle's bits."""
    n, root = 20, 7
    with rra.Comm(n, n * 65536 * 4) as comm:
        for op, m in (("all_gather", 1024), ("broadcast", 65536)):
            src_np = [inputs.normal(inputs.rng(103, r, m), 1, m, "fp32")[0] for r in range(n)]
            want = oracle.all_gather(src_np, "fp32") if op == "all_gather" else oracle.broadcast(src_np, "fp32", root)
            src = to_device(src_np, "fp32")
            out_n = n * m if op == "all_gather" else m
            out = [torch.full((out_n,), float("nan"), device="cuda") for _ in range(n)]
            comm.collective_ptrs(op, [t.data_ptr() for t in src], [t.data_ptr() for t in out], m, "fp32", root)
            torch.cuda.synchronize()
            assert comm.last_kernel() == "coll_multi_kernel<%s, bulk, bulk store>" % op, comm.last_kernel()
            for g, w in zip(out, want):
                assert np.array_equal(bits(g.cpu().numpy()), bits(w)), op
        assert comm.status()[0] == rra.OK


def test_collective_outputs_in_host_memory_get_vector_stores():
    """Device inputs, outputs in pinned host memory: the push is by bulk
    copies, the outputs are written by vector stores (no bulk copy writes
    host memory)."""
    n, m = 4, 65536
    small_np = [inputs.normal(inputs.rng(96, r), 1, m, "fp32")[0] for r in range(n)]
    want_ag = oracle.all_gather(small_np, "fp32")
    want_bc = oracle.broadcast(small_np, "fp32", 1)
    on_device = to_device(small_np, "fp32")
    ho = [torch.full((n * m,), float("nan")).pin_memory() for _ in range(n)]
    hb = [torch.full((m,), float("nan")).pin_memory() for _ in range(n)]
    dev_ho = rra.host_device_ptrs([t.data_ptr() for t in ho])
    dev_hb = rra.host_device_ptrs([t.data_ptr() for t in hb])
    with rra.Comm(n, n * m * 4) as comm:
        src = [t.data_ptr() for t in on_device]
        comm.collective_ptrs("all_gather", src, dev_ho, m, "fp32", 0)
        torch.cuda.synchronize()
        assert comm.last_kernel() == "coll_bulk_kernel<all_gather>"
        comm.collective_ptrs("broadcast", src, dev_hb, m, "fp32", 1)
        torch.cuda.synchronize()
        assert comm.last_kernel() == "coll_split_kernel<broadcast>"  # no bulk stores: two hops at 256 KiB
        assert comm.status()[0] == rra.OK
    for g, w in zip(ho, want_ag):
        assert np.array_equal(bits(g.numpy()), bits(w))
    for g, w in zip(hb, want_bc):
        assert np.array_equal(bits(g.numpy()), bits(w))


def test_fused_residual_chooses_its_push_by_source_memory():
    n, count = 4, 2000
    sends_np = inputs.normal(inputs.rng(95, 0), n, count, "fp32")
    res_np = inputs.normal(inputs.rng(95, 1), n, count, "fp32")
    want = oracle.allreduce_residual(sends_np, res_np, "fp32")
    hs = _pinned(sends_np)
    dev_host = rra.host_device_ptrs([t.data_ptr() for t in hs])
    res = to_device(res_np, "fp32")
    on_device = to_device(sends_np, "fp32")  # kept alive: the calls read it
    with rra.Comm(n, count * 4) as comm:
        for where, src in (("device", [t.data_ptr() for t in on_device]), ("host", dev_host)):
            out = [torch.full((count,), float("nan"), device="cuda") for _ in range(n)]
            comm.allreduce_residual_ptrs(src, [t.data_ptr() for t in res], [t.data_ptr() for t in out], count, "fp32")
            torch.cuda.synchronize()
            kind = comm.last_kernel()
            # device inputs: the cluster AllReduce's bulk-copy one-shot with the
            # residual epilogue; host inputs: the device-API kernel on st.async
            want_kind = "cluster_tma_kernel<one-shot, residual>" if where == "device" else "residual_kernel<one-shot>"
            assert kind == want_kind, kind
            for g, w in zip(out, want):
                assert np.array_equal(bits(g.cpu().numpy()), bits(w))
        assert comm.status()[0] == rra.OK
