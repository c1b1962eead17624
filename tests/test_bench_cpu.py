"""CPU tests of bench.py's host logic: replica aggregation over ranks (gloo,
world size 2), clock-record parsing and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vals = bench.max_over_ranks(dist, [1.0 + rank, 10.0 - rank, 5.0])
    bench.barrier(dist)
    q.put((rank, vals))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        assert res[r] == [2.0, 10.0, 5.0]


def test_single_rank_aggregation_is_identity():
    assert bench.max_over_ranks(None, [1.5, 2.5]) == [1.5, 2.5]


def test_clock_parsing(tmp_path):
    c = bench.ClockSampler(0)
    c.path = str(tmp_path / "clocks.csv")
    with open(c.path, "w") as f:
        f.write("0, 1900, 2070, 800.1, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1950, 2070, 900.2, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 2000, 2070, 950.3, 0x0, Not Active, Not Active, Not Active, Not Active\n")

    class P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    c.proc = P()
    c.f = open(os.devnull, "w")
    out = c.stop()
    assert out["sm_mhz"] == 1950.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ)
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "us/call" and d["higher_is_better"] is False
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["warmup"] >= 3


def test_source_hash_ignores_comments_not_code():
    """The hash that ties a committed DRAM-traffic figure to the device code:
    a comment or blank-line edit keeps it, any code edit changes it."""
    src = "int a; // note\n/* block\n comment */\n\n__device__ int f() { return 1; }\n"
    same = "int a;\n// another note\n__device__ int f() { return 1; }   \n"
    other = "int a;\n__device__ int f() { return 2; }\n"
    assert bench.strip_comments(src) == bench.strip_comments(same)
    assert bench.strip_comments(src) != bench.strip_comments(other)
    assert bench.strip_comments('asm volatile("mov.u32 %0, 1;");') == 'asm volatile("mov.u32 %0, 1;");'
    h = bench.kernel_source_sha()
    assert len(h) == 16 and h == bench.kernel_source_sha()
    entries = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))["entries"]
    assert entries and all(len(e["source_sha"]) == 16 for e in entries)
