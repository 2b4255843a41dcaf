"""The FP8 quantisers' division-free quotient equals the IEEE division everywhere.

The quantisers (Q, K per vector; V per channel) define each code as
E4M3(RN(x / s)) with s = RN(max|x| / 448). They compute RN(x / s) from one
correctly rounded reciprocal per vector and Markstein's correction
(csrc/fp8_quotient.cuh). Inputs are BF16, so every pair (x, maximum) they can
meet is enumerable: tests/fp8_quotient_check.cu compares the correction with
CUDA's IEEE division on all of them (~1.04e9 with |x| <= maximum): the E4M3
codes agree everywhere, and so do the FP32 quotients wherever either is 2^-11
or more. (Below that they may differ in low bits when x is subnormal, where
the remainder of the correction is no longer exact; E4M3 rounds both to zero.)
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def expected_pairs() -> int:
    """Pairs the checker visits: m = BF16 0x0001..0x7F7F with RN(m / 448) >= 2^-100,
    and for each, the 2 (m_bits + 1) BF16 values x with |x| <= m (both signs)."""
    bits = np.arange(1, 0x7F80, dtype=np.uint32)
    m = (bits << 16).view(np.float32)
    s = m / np.float32(448.0)  # IEEE float32 division, as on the device
    keep = s >= np.float32(2.0 ** -100)
    return int((2 * (bits[keep].astype(np.int64) + 1)).sum())


def test_quotient_matches_ieee_division_on_every_bf16_pair(tmp_path):
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = shutil.which("nvcc") or "nvcc"
    exe = tmp_path / "fp8_quotient_check"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(ROOT, "gqa_chunked_prefill_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "fp8_quotient_check.cu"), "-o", str(exe)],
                   check=True, capture_output=True, timeout=600)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    f = r.stdout.split()
    got = dict(zip(f[0::2], f[1::2]))
    assert int(got["checked"]) == expected_pairs()
    assert int(got["code_mismatch"]) == 0, r.stdout
    assert int(got["fp32_mismatch_from_2^-11"]) == 0, r.stdout
