"""Paged K/V addressing checked on the CPU: tests/paged_rows_check.cpp includes
csrc/gqa_paged.h (the code the attention kernel's TMA producer runs) and
brute-forces, key by key, which cache row every box of every KV tile is copied
from, over many page sizes, sequence lengths and block tables (including entries
outside the cache)."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_paged_rows_map_every_key(tmp_path):
    exe = tmp_path / "paged_rows_check"
    src = os.path.join(ROOT, "tests", "paged_rows_check.cpp")
    inc = os.path.join(ROOT, "gqa_chunked_prefill_gb300", "csrc")
    subprocess.run(["g++", "-O2", "-std=c++17", "-D__host__=", "-D__device__=", "-I", inc, src,
                    "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad=0" in r.stdout
