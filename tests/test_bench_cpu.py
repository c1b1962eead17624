"""CPU tests of bench.py's host logic: the compact last line, the refusal of
multi-GPU runs, clock-record parsing and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _fake_detail():
    """A full result of the shape run_ours builds (every table present, values
    made up), as large as a default run's."""
    sizes = [128 << k for k in range(14)]
    cases = ["%s/%d" % (dt, m) for dt in ("fp32", "bf16") for m in sizes]
    algos = list(bench.ALGOS)
    kern = {"N%d/%s" % (n, a): 1.234 for n in (2, 4) for a in algos}
    bw = {"%s/%s/%dMiB" % (a, dt, m): {"ms": 1.0, "GB/s": 6000.0, "frac": 0.9, "busbw_GB/s": 5000.0,
                                       "status": "RRA_OK"}
          for a in ("twoshot_dbuf", "twoshot_direct", "twoshot_cluster") for dt in ("fp32", "fp64")
          for m in (4, 64, 512)}
    return {
        "metric": bench.METRIC, "value": 1.854, "unit": "us/call", "n_gpus": 1, "steps": 20, "warmup": 5,
        "ms_per_step": 0.889, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32+bf16", "data": "synthetic (seeded N(0,1), no dataset)",
        "config": {"workload": bench.WORKLOAD, "nranks": 4, "sizes_bytes": sizes, "inner_calls": 16,
                   "l2": "flushed (256 MiB write) between steps; calls in a step reuse L2-resident buffers",
                   "parallelism": "single GPU", "gpu": "NVIDIA GB300", "sms": 152},
        "gpu_launches": 8960,
        "roofline": {"bound": "hbm", "achieved": 646.5, "peak": 6779.0, "unit": "GB/s", "frac": 0.0954,
                     "traffic": 608654, "kernel": "cluster_tma_kernel", "config": "x" * 60,
                     "launches_per_step": 448, "bytes_per_launch": 1198299.4, "us_per_launch": 1.854,
                     "share_of_step": 1.0, "peak_source": "measured", "note": "y" * 200,
                     "launched": {c: "cluster_tma_kernel<one-shot>" for c in cases},
                     "largest_launch": {"config": "z" * 40, "kernel": "k", "achieved": 1.0, "frac": 0.1,
                                        "traffic": None}},
        "latency_floor": {"l2_rtt_ns": 150.5, "store_poll_ns": 427.9, "pingpong_rtt_ns": [850.0] * 32,
                          "pingpong_sms": [[0, 5]] * 32, "floor_us": 0.729, "floor_dsmem_us": 0.4,
                          "in_kernel_us_128B": kern, "best_in_kernel": "N2/oneshot_cluster",
                          "best_over_floor": 0.83, "empty_kernel_us": 2.0, "graph_node_us": 0.7, "method": "m" * 300},
        "bandwidth": {"nranks": 8, "bytes": "2*N*M per call", "sizes": bw, "note": "n" * 100},
        "e2e": {"value": 18.75, "unit": "us/call", "h2d_bytes_per_step": 16776192, "d2h_bytes_per_step": 16776192,
                "api": "a" * 300, "per_case_us": [12.5] * 28},
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 16},
        "auto_us": {c: 1.5 for c in cases}, "auto_algo": {c: "oneshot_cluster" for c in cases},
        "per_size_us": {c: {a: 3.4 for a in algos} for c in cases},
        "cpu_baseline": {"value": 865.384, "unit": "us/call", "cores": 16, "kind": "oracle", "sample": "s" * 150},
    }


def test_summary_line_is_compact_and_complete(tmp_path):
    """The last stdout line stays well under 4 KB (a driver keeps only the
    tail of stdout) and carries every key the measurement contract names."""
    d = _fake_detail()
    line = json.dumps(bench.summary_line(d, str(tmp_path / "bench_detail.json")))
    assert len(line) < 3500, len(line)
    out = json.loads(line)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "gpu_launches"):
        assert out[k] == d[k], k
    assert out["config"]["workload"] == bench.WORKLOAD
    r = out["roofline"]
    assert r["bound"] == "hbm" and r["frac"] == 0.0954 and r["traffic"] == 608654 and r["peak"] == 6779.0
    assert out["e2e"]["h2d_bytes_per_step"] > 0 and out["e2e"]["d2h_bytes_per_step"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] == 16
    assert out["clocks"]["sm_mhz"] == 2070.0 and out["clocks"]["reasons"] == []
    lf = out["latency_floor"]
    assert lf["in_kernel_us_128B"]["N2/oneshot_ll"] == 1.234
    assert lf["x_floor"]["N2/oneshot_ll"] == round(1.234 / 0.729, 2)
    assert lf["x_floor"]["N4/oneshot_cluster"] == round(1.234 / 0.4, 2)  # the DSMEM floor for the cluster kernel
    assert "N2/twoshot_direct" not in lf["in_kernel_us_128B"]
    assert out["bandwidth_hbm_frac"]["twoshot_dbuf/fp32/512MiB"] == 0.9


def test_multi_gpu_request_prints_unavailable():
    """--gpus 2 (or a torchrun rank with WORLD_SIZE=2) does no GPU work: rank 0
    prints one JSON line with the reason, every rank exits 0."""
    for extra_env, want_line in (({}, True), ({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"}, False)):
        env = dict(os.environ, **extra_env)
        p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                           capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
        assert p.returncode == 0, p.stderr
        lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
        if not want_line:
            assert lines == []
            continue
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["n_gpus"] == 2 and "one GPU only" in d["unavailable"] and d["metric"] == bench.METRIC


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
