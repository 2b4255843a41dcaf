"""The work decomposition shared by the planner and the kernels, checked on the
CPU: tests/schedule_cover_check.cpp includes csrc/gqa_schedule.h directly and
brute-forces coverage (every KV tile of every item exactly once, no empty unit,
partial slots exactly where the merge kernel reads them) over many chunk shapes,
grid sizes, numbers of whole rounds and tail splits."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_schedule_covers_every_tile_once(tmp_path):
    exe = tmp_path / "schedule_cover_check"
    src = os.path.join(ROOT, "tests", "schedule_cover_check.cpp")
    inc = os.path.join(ROOT, "gqa_chunked_prefill_gb300", "csrc")
    subprocess.run(["g++", "-O2", "-std=c++17", "-D__host__=", "-D__device__=", "-I", inc, src,
                    "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad=0" in r.stdout
