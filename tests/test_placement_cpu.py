"""CPU test of the rule that decides where the bulk-copy push (TMA bulk copies
with cluster multicast) may read: only when every source lies in device
memory of the current GPU, over the whole range the copies read (rounded up
to 16-byte vectors), and the process drives no other GPU.  The rule is plain
host C++ (csrc/placement.h); tests/placement_check.cpp runs it against a fake
memory map."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bulk_copy_placement_rule(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    exe = str(tmp_path / "placement_check")
    subprocess.run([gxx, "-std=c++17", "-O1", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "latency_barrier_free_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "placement_check.cpp"), "-o", exe], check=True)
    run = subprocess.run([exe], capture_output=True, text=True)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip().endswith("0 failed"), run.stdout
