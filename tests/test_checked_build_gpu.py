"""The parity suite on the bounds-checked build (libgqa_prefill_checked.so).

That build checks, inside the kernels, every row the epilogue stores (output, LSE,
split partials) and every partial row the merge pass reads or writes against its
buffer; a row outside records GQA_ERR_BOUNDS in the device status word and skips the
access. The GPU parity tests assert the status word is 0 after every call, so
running them on this build (in a child process that loads it through
GQA_PREFILL_LIB) checks both the results and that no access left its buffer: dense
shapes with ragged tails, forced uniform and balanced split tails, decode shapes,
items cut into 16 or more pieces (the block-per-row merge), and paged, batched and FP8 calls."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_on_the_bounds_checked_build(cuda_device):
    lib = os.path.join(ROOT, "gqa_chunked_prefill_gb300", "libgqa_prefill_checked.so")
    assert os.path.exists(lib), "build() makes the bounds-checked library"
    env = dict(os.environ, GQA_PREFILL_LIB=lib)
    sel = ("small_shapes or split_tail or balanced or whole_items or decode or many_pieces or paged "
           "or varlen or fp8")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-k", sel,
                        "-p", "no:cacheprovider",
                        "tests/test_parity_gpu.py", "tests/test_paged_gpu.py",
                        "tests/test_varlen_gpu.py", "tests/test_fp8qk_gpu.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
