"""GPU invariants of the CUDA path: determinism, causality (bit-exact), agreement
of whole and cut work items, the ABI's refusals and empty chunks, and the route check (the plan
the library reports for the call that ran)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gqa_inputs import WORKLOADS, make_qkv, make_workload
from tests.gpu_helpers import check_close, run_gpu

pytestmark = pytest.mark.gpu
SCALE = 1.0 / 16.0


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("variant", [0, 1, 2])
def test_run_twice_bit_identical(cuda_device, name, variant):
    """Every workload at full size, on the planner's choice (0) and on each kernel
    variant forced: two calls on the same inputs give the same bits (split pieces
    are merged in a fixed order; nothing depends on which CTA finishes first)."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    o1, l1, p1 = run_gpu(q, k, v, w.scale, force_variant=variant)
    o2, l2, p2 = run_gpu(q, k, v, w.scale, force_variant=variant)
    assert p1 == p2
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("q_len,kv_len,t_star", [(100, 700, 40), (300, 300, 150), (512, 4096, 200)])
@pytest.mark.parametrize("splits,grid,variant", [(0, 0, 1), (3, 9, 1), (0, 0, 2), (3, 10, 2),
                                                 (-1, 0, 1), (-1, 10, 2)])
def test_future_keys_leave_earlier_rows_bit_identical(cuda_device, q_len, kv_len, t_star, splits,
                                                      grid, variant):
    q, k, v = make_qkv(q_len, kv_len, seed=q_len + kv_len)
    o1, l1, _ = run_gpu(q, k, v, SCALE, force_splits=splits, force_grid=grid,
                        force_variant=variant)
    p_star = kv_len - q_len + t_star
    k2, v2 = k.clone(), v.clone()
    k2[p_star + 1:] = (k2[p_star + 1:].float() * 3.0 + 1.0).to(torch.bfloat16)
    v2[p_star + 1:] = (-v2[p_star + 1:].float() + 2.0).to(torch.bfloat16)
    o2, l2, _ = run_gpu(q, k2, v2, SCALE, force_splits=splits, force_grid=grid,
                        force_variant=variant)
    assert torch.equal(o1[: t_star + 1], o2[: t_star + 1])
    assert torch.equal(l1[: t_star + 1], l2[: t_star + 1])
    assert not torch.equal(o1[t_star + 1:], o2[t_star + 1:])


@pytest.mark.parametrize("name", ["q512_kv4096_kbias", "q4096_kv8192"])
@pytest.mark.parametrize("variant", [1, 2])
def test_whole_and_cut_items_agree(cuda_device, name, variant):
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    o1, l1, p1 = run_gpu(q, k, v, SCALE, force_splits=1, force_variant=variant)
    o2, l2, p2 = run_gpu(q, k, v, SCALE, force_splits=4, force_variant=variant)
    assert p1["tail_splits"] == 1 and p1["kernels_per_call"] == 1
    assert p2["tail_splits"] == 4 and p2["tail_items"] > 0 and p2["kernels_per_call"] == 2
    check_close(o2.double().cpu().numpy(), l2.double().cpu().numpy(),
                o1.double().cpu().numpy(), l1.double().cpu().numpy(), "cut vs whole items")


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_route_check_reports_planned_kernel(cuda_device, name):
    """The plan a call reports is the one the host-only planner makes from the
    device's SM count and co-resident CTA pairs (as the library measures them)."""
    import gqa_chunked_prefill_gb300 as gqa
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    _, _, plan = run_gpu(q, k, v, w.scale)
    sms, pairs = gqa.gqa_prefill_device_info()
    assert sms == torch.cuda.get_device_properties(0).multi_processor_count
    assert 0 <= pairs <= sms // 2
    _, host_plan = gqa.gqa_prefill_make_plan(w.q_len, w.kv_len, 24, 4, 256, sms, max_pairs=pairs)
    assert plan == host_plan
    assert plan["variant"] in (1, 2) and plan["num_sms"] == sms and plan["grid"] <= sms


def test_empty_chunk_is_a_no_op(cuda_device):
    import gqa_chunked_prefill_gb300 as gqa
    k = torch.randn(10, 4, 256, device="cuda").to(torch.bfloat16)
    rc = gqa.gqa_prefill_attn(None, k, k, None, None, 0, 10, 24, 4, 256, SCALE, check=False)
    assert rc == 0


def test_refusals_launch_nothing(cuda_device):
    import gqa_chunked_prefill_gb300 as gqa
    from gqa_chunked_prefill_gb300 import GqaStatus as S
    q = torch.zeros(8, 24, 256, device="cuda", dtype=torch.bfloat16)
    kv = torch.zeros(16, 4, 256, device="cuda", dtype=torch.bfloat16)
    out = torch.full_like(q, 7.0)
    f = lambda *a: gqa.gqa_prefill_attn(*a, check=False)
    assert f(q, kv, kv, out, None, 8, 7, 24, 4, 256, SCALE) == S.ERR_SHAPE
    assert f(q, kv, kv, out, None, 8, 16, 24, 4, 128, SCALE) == S.ERR_UNSUPPORTED
    assert f(q, kv, kv, out, None, 8, 16, 24, 8, 256, SCALE) == S.ERR_UNSUPPORTED
    assert f(q, kv, kv, out, None, 8, 16, 24, 4, 256, -1.0) == S.ERR_SHAPE
    assert f(q, None, kv, out, None, 8, 16, 24, 4, 256, SCALE) == S.ERR_NULL
    assert f(q.data_ptr() + 2, kv, kv, out, None, 8, 16, 24, 4, 256, SCALE) == S.ERR_ALIGN
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)  # nothing was launched


def test_non_default_stream(cuda_device):
    q, k, v = make_qkv(200, 900, seed=9)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1, _ = run_gpu(q, k, v, SCALE, stream=s)
    o0, l0, _ = run_gpu(q, k, v, SCALE)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
