"""GPU parity on workload 3 (Llama-3.1-70B-shaped decode, 160 AllReduces per
token in one CUDA graph) and workload 5 (the bandwidth end, up to 512 MiB per
rank, every element compared with the oracle)."""
import os

import numpy as np
import pytest

import oracle
from latency_barrier_free_gb300 import inputs, rra
from tests.gpu_util import bits, check_against_oracle, to_device, to_host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


@pytest.mark.parametrize("algo", ["twoshot_dbuf", "oneshot_ll", "twoshot_direct", "oneshot_sentinel",
                                  "oneshot_cluster", "twoshot_cluster", "auto"])
@pytest.mark.parametrize("batch", inputs.W3_BATCHES)
def test_workload3_decode_graph(batch, algo):
    """One token = 160 AllReduces of bf16 [batch, 8192] over N=8, captured in
    one CUDA graph.  Each call has its own output buffers (inputs cycle over 8
    distinct draws); the graph is replayed twice with new inputs."""
    n, calls, distinct = 8, inputs.W3_CALLS_PER_TOKEN, 8
    count = batch * inputs.W3_HIDDEN
    with rra.Comm(n, count * 2) as comm:
        send = torch.empty(distinct, n, count, dtype=torch.bfloat16, device="cuda")
        recv = torch.empty(calls, n, count, dtype=torch.bfloat16, device="cuda")

        def enqueue():
            for i in range(calls):
                j = i % distinct
                comm.allreduce_ptrs([send[j, r].data_ptr() for r in range(n)],
                                    [recv[i, r].data_ptr() for r in range(n)], count, "bf16", algo)

        enqueue()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                enqueue()
        for rep in range(2):
            host = [inputs.workload3(batch, iteration=100 * rep + j) for j in range(distinct)]
            for j in range(distinct):
                for r in range(n):
                    send[j, r].copy_(to_device([host[j][r]], "bf16")[0])
            recv.view(torch.int16).fill_(0x7F7F)
            g.replay()
            torch.cuda.synchronize()
            assert comm.status()[0] == rra.OK
            expect = [oracle.allreduce(h, "bf16")[0] for h in host]
            got = recv.view(torch.int16).cpu().numpy().view(np.uint16)
            for i in range(calls):
                for r in range(n):
                    assert np.array_equal(got[i, r], expect[i % distinct]), (rep, i, r)


def test_workload3_same_buffer_variant():
    """All 160 calls of a token on the same send/recv buffers."""
    n, batch = 8, 16
    count = batch * inputs.W3_HIDDEN
    host = inputs.workload3(batch)
    expect = oracle.allreduce(host, "bf16")[0]
    with rra.Comm(n, count * 2) as comm:
        for algo in ("twoshot_dbuf", "oneshot_ll"):
            xs = to_device(host, "bf16")
            ys = [torch.empty_like(x) for x in xs]
            for _ in range(inputs.W3_CALLS_PER_TOKEN):
                comm.allreduce(xs, ys, algo)
            torch.cuda.synchronize()
            assert comm.status()[0] == rra.OK
            for y in to_host(ys, "bf16"):
                assert np.array_equal(y, expect)


def _expected_full(host, dtype):
    """The oracle's AllReduce of the whole message (every rank's output is the
    same, so one array is written N times)."""
    out = np.empty_like(host[0])
    oracle.allreduce_mt(host, dtype, os.cpu_count() or 1, recvs=[out] * len(host))
    return out


def _full_check(expect, recv0, dtype, algo, piece):
    """Every element of rank 0's output bit-exact against the oracle, copied
    back in pieces (the other ranks are compared with rank 0 on the device)."""
    for off in range(0, expect.size, piece):
        m = min(piece, expect.size - off)
        got = recv0[off:off + m].cpu().numpy()
        bad = np.nonzero(bits(got) != bits(expect[off:off + m]))[0]
        assert bad.size == 0, "%s %s: %d mismatches in [%d, %d), first at %d: got %r expect %r" % (
            algo, dtype, bad.size, off, off + m, off + bad[0], got[bad[0]], expect[off + bad[0]])


def _bounded_check(host, recv0, dtype, algo, piece):
    """LL128-atomic (unordered sums): every element within the stated bound,
    piece by piece."""
    for off in range(0, host[0].size, piece):
        m = min(piece, host[0].size - off)
        check_against_oracle([h[off:off + m] for h in host], [recv0[off:off + m].cpu().numpy()], dtype, algo)


@pytest.mark.parametrize("dtype", ["fp32", "fp64"])
@pytest.mark.parametrize("size", inputs.W5_SIZES)
def test_workload5_bandwidth_end(size, dtype):
    """N=8 at 4 MiB / 64 MiB / 512 MiB per rank with the two-shot kernels (the
    cluster two-shot is the one the bench times at the bandwidth end, and the
    automatic choice), uniform(-1,1) inputs from the seeded generator: every
    rank's output equal on the device, and every element of it bit-exact
    against the oracle (one pass of the oracle over the whole message)."""
    n = 8
    elem = 4 if dtype == "fp32" else 8
    count = size // elem
    np_dt = np.float32 if dtype == "fp32" else np.float64
    g = inputs.rng(5, 0, size, inputs.DT_CODE[dtype])
    piece = (64 << 20) // elem
    host = []
    for r in range(n):
        h = np.empty(count, dtype=np_dt)
        for off in range(0, count, piece):
            m = min(piece, count - off)
            h[off:off + m] = inputs.uniform(g, 1, m, dtype)[0].astype(np_dt)
        host.append(h)
    expect = _expected_full(host, dtype)
    sends = [torch.from_numpy(h).cuda() for h in host]
    recvs = [torch.empty_like(s) for s in sends]
    with rra.Comm(n, size) as comm:
        for algo in ("twoshot_dbuf", "twoshot_direct", "twoshot_cluster", "auto"):
            for t in recvs:
                t.view(torch.uint8).fill_(0x7F)
            comm.allreduce(sends, recvs, algo)
            torch.cuda.synchronize()
            assert comm.status()[0] == rra.OK
            for r in range(1, n):
                assert torch.equal(recvs[r].view(torch.uint8), recvs[0].view(torch.uint8))
            _full_check(expect, recvs[0], dtype, algo, piece)
        for algo in ("oneshot_sentinel", "ll128_atomic"):
            if size > (64 << 20):
                continue
            for t in recvs:
                t.view(torch.uint8).fill_(0x7F)
            comm.allreduce(sends, recvs, algo)
            torch.cuda.synchronize()
            assert comm.status()[0] == rra.OK
            for r in range(1, n):
                assert torch.equal(recvs[r].view(torch.uint8), recvs[0].view(torch.uint8))
            if algo == "oneshot_sentinel":
                _full_check(expect, recvs[0], dtype, algo, piece)
            else:
                _bounded_check(host, recvs[0], dtype, algo, piece)
    del sends, recvs
    torch.cuda.empty_cache()
