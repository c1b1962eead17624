"""GPU parity on workload 3 (Llama-3.1-70B-shaped decode, 160 AllReduces per
token in one CUDA graph) and workload 5 (the bandwidth end, up to 512 MiB per
rank, checked on sampled elements that the oracle computes one by one)."""
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


def _sampled_check(sends, recvs, dtype, algo, nsample=20000, seed=0):
    count = sends[0].numel()
    g = np.random.Generator(np.random.PCG64(seed))
    idx = np.unique(np.concatenate([g.integers(0, count, nsample), [0, 1, count - 2, count - 1]]))
    tidx = torch.from_numpy(idx).cuda()
    s_np = [s[tidx].cpu().numpy() for s in sends]
    r_np = [r[tidx].cpu().numpy() for r in recvs]
    check_against_oracle(s_np, r_np, dtype, algo)


@pytest.mark.parametrize("dtype", ["fp32", "fp64"])
@pytest.mark.parametrize("size", inputs.W5_SIZES)
def test_workload5_bandwidth_end(size, dtype):
    """N=8 at 4 MiB / 64 MiB / 512 MiB per rank with the two-shot kernels (the
    cluster two-shot is the one the bench times at the bandwidth end, and the
    automatic choice), uniform(-1,1) inputs from
    the seeded generator; every rank's output equal, sampled elements
    bit-exact against the oracle."""
    n = 8
    elem = 4 if dtype == "fp32" else 8
    count = size // elem
    np_dt = np.float32 if dtype == "fp32" else np.float64
    sends = []
    g = inputs.rng(5, 0, size, inputs.DT_CODE[dtype])
    piece = (64 << 20) // elem
    for r in range(n):
        t = torch.empty(count, dtype=torch.float32 if dtype == "fp32" else torch.float64, device="cuda")
        for off in range(0, count, piece):
            m = min(piece, count - off)
            t[off:off + m].copy_(torch.from_numpy(inputs.uniform(g, 1, m, dtype)[0].astype(np_dt)))
        sends.append(t)
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
            _sampled_check(sends, recvs, dtype, rra.select_algo(n, size, dtype) if algo == "auto" else algo)
        for algo in ("oneshot_sentinel", "ll128_atomic"):
            if size > (64 << 20):
                continue
            comm.allreduce(sends, recvs, algo)
            torch.cuda.synchronize()
            assert comm.status()[0] == rra.OK
            _sampled_check(sends, recvs, dtype, algo, seed=1)
    del sends, recvs
    torch.cuda.empty_cache()
