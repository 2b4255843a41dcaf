"""gqa_prefill_attn_noalloc: the entry point for callers that cannot allocate
device memory during a call (engines that reserve the whole memory budget at
start-up, code that must not risk cudaFree's implicit synchronisation, hosts
whose allocator belongs to another framework). It keeps split-KV partials in a
64 MiB scratch array compiled into the library instead of allocating them.

Checks, through the C ABI: on workloads whose plan splits work items along
the KV range (so the scratch really holds partials), two calls in a row each
match the allocating entry point within the suite's tolerance; a call whose
partials would not fit is refused with GQA_ERR_SCRATCH and writes nothing (on
devices where such a plan exists); and calls with growing split partials leave
the device's free memory unchanged. This file is collected last, and it also
passes when run alone in a fresh process."""
import pytest
import torch

from gqa_inputs import WORKLOADS, make_qkv, make_workload
from tests.gpu_helpers import check_close

pytestmark = pytest.mark.gpu
SCRATCH_BYTES = 64 << 20


def _run(fn, qd, kd, vd, scale):
    q_len, hq, d = qd.shape
    kv_len, hkv, _ = kd.shape
    out = torch.full_like(qd, float("nan"))
    lse = torch.full((q_len, hq), float("nan"), dtype=torch.float32, device=qd.device)
    fn(qd, kd, vd, out, lse, q_len, kv_len, hq, hkv, d, scale)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("case", ["q512_kv4096_kbias", "q512_kv32768", "small_forced"])
def test_noalloc_matches_allocating_entry_on_two_calls(cuda_device, case):
    import gqa_chunked_prefill_gb300 as gqa
    if case == "small_forced":
        q, k, v = make_qkv(129, 1000, seed=77)
        scale = 1 / 16
    else:
        w = WORKLOADS[case]
        q, k, v = make_workload(w)
        scale = w.scale
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, plan = gqa.gqa_prefill_make_plan(q.shape[0], k.shape[0], 24, 4, 256, sms)
    assert plan["workspace_bytes"] <= SCRATCH_BYTES
    ref_o, ref_l = _run(gqa.gqa_prefill_attn, qd, kd, vd, scale)
    for _ in range(2):
        o, l = _run(gqa.gqa_prefill_attn_noalloc, qd, kd, vd, scale)
        assert gqa.gqa_prefill_poll() == 0
        check_close(o.double().cpu().numpy(), l.double().cpu().numpy(),
                    ref_o.double().cpu().numpy(), ref_l.double().cpu().numpy(), f"noalloc {case}")


def test_noalloc_uses_scratch_on_a_split_plan(cuda_device):
    """At least one of the shapes above really exercises the scratch array."""
    import gqa_chunked_prefill_gb300 as gqa
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plans = [gqa.gqa_prefill_make_plan(WORKLOADS[n].q_len, WORKLOADS[n].kv_len, 24, 4, 256, sms)[1]
             for n in ("q512_kv4096_kbias", "q512_kv32768")]
    assert any(p["tail_splits"] != 1 and 0 < p["workspace_bytes"] <= SCRATCH_BYTES
               for p in plans)


def test_noalloc_refuses_partials_larger_than_scratch(cuda_device):
    import gqa_chunked_prefill_gb300 as gqa
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    big = None
    for q_len, kv_len in ((4096, 32768), (4096, 16384), (2048, 65536), (4096, 65536), (168, 262144)):
        _, plan = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, sms)
        if plan["workspace_bytes"] > SCRATCH_BYTES:
            big = (q_len, kv_len)
            break
    if big is None:
        pytest.skip("no candidate shape needs more split scratch than the array on this device")
    q_len, kv_len = big
    q = torch.zeros(q_len, 24, 256, device="cuda", dtype=torch.bfloat16)
    kv = torch.zeros(kv_len, 4, 256, device="cuda", dtype=torch.bfloat16)
    out = torch.full_like(q, 3.0)
    rc = gqa.gqa_prefill_attn_noalloc(q, kv, kv, out, None, q_len, kv_len, 24, 4, 256, 1 / 16,
                                      check=False)
    assert rc == gqa.GqaStatus.ERR_SCRATCH
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)


_NO_ALLOC_CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import gqa_chunked_prefill_gb300 as gqa
from gqa_inputs import make_qkv
dev = torch.device("cuda:0")
cases = [(129, 1000), (512, 4096), (512, 32768)]  # split plans, growing partials
sms, pairs = gqa.gqa_prefill_device_info()
ws = [gqa.gqa_prefill_make_plan(a, b, 24, 4, 256, sms, max_pairs=pairs)[1]["workspace_bytes"]
      for a, b in cases]
assert 0 < ws[0] < ws[-1], ws
bufs = []
for q_len, kv_len in cases:
    q, k, v = (t.to(dev) for t in make_qkv(q_len, kv_len, seed=q_len))
    out = torch.empty_like(q)
    lse = torch.empty((q_len, 24), dtype=torch.float32, device=dev)
    bufs.append((q, k, v, out, lse, q_len, kv_len))
torch.cuda.synchronize()
q, k, v, out, lse, q_len, kv_len = bufs[0]
gqa.gqa_prefill_attn_noalloc(q, k, v, out, lse, q_len, kv_len, 24, 4, 256, 1 / 16)  # set-up
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
for q, k, v, out, lse, q_len, kv_len in bufs:
    for _ in range(2):
        gqa.gqa_prefill_attn_noalloc(q, k, v, out, lse, q_len, kv_len, 24, 4, 256, 1 / 16)
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
assert gqa.gqa_prefill_poll() == 0
print("free", free0, free1, "workspace", ws)
assert free1 == free0, (free0, free1)
"""


def test_noalloc_allocates_no_device_memory(cuda_device):
    """The promise itself: in a fresh process (no earlier call has grown any pool;
    every kernel loaded up front), after one warm-up call that does the one-time
    set-up, calls whose split partials grow from the smallest to the largest of
    three plans leave the device's free memory exactly unchanged. A version that
    took the partials from an allocator would have to grow it for the larger plans."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    # Eager module loading: every kernel of the library is resident before the
    # measurement, so a first launch cannot take device memory for its code.
    env = dict(os.environ, CUDA_MODULE_LOADING="EAGER")
    r = subprocess.run([sys.executable, "-c", _NO_ALLOC_CHILD, root], capture_output=True,
                       text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
