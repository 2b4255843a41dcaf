"""GPU parity of the paged-K/V entry point (gqa_prefill_attn_paged).

Each case checks two things: the paged call equals the dense call on the same
logical K/V bit for bit (same plan and kernel variant: both put identical tiles
in shared memory), and it matches the FP64 oracle reading the same caches
through the block table, at the acceptance tolerance. Caches place the
sequence's pages in a seeded random order among spare pages and fill every
slot the sequence does not use with NaN, so a slot past kv_len that reached a
result would show.
"""
import pytest
import torch

import oracle
from gqa_inputs import (SERVING_PAGE_SIZE, WORKLOADS, make_paged_cache, make_qkv, make_workload,
                        sample_rows)
from tests.gpu_helpers import check_close, gather_rows, item_cover_rows, run_gpu, unchecked_items

pytestmark = pytest.mark.gpu
SCALE = 1.0 / 16.0


def run_paged(q, k_cache, v_cache, table, kv_len, scale, force_splits=0, force_grid=0,
              force_variant=0):
    """Returns (out, lse, plan, device status word after the call)."""
    import gqa_chunked_prefill_gb300 as gqa
    dev = torch.device("cuda:0")
    qd = q.to(dev).contiguous()
    kc, vc = k_cache.to(dev).contiguous(), v_cache.to(dev).contiguous()
    td = table.to(device=dev, dtype=torch.int32).contiguous()
    q_len = qd.shape[0]
    out = torch.empty_like(qd)
    lse = torch.empty((q_len, qd.shape[1]), dtype=torch.float32, device=dev)
    _, plan = gqa.gqa_prefill_attn_paged_ex(
        qd, kc, vc, td, kc.shape[0], kc.shape[1], out, lse, q_len, kv_len, qd.shape[1],
        kc.shape[2], kc.shape[3], scale, force_splits=force_splits, force_grid=force_grid,
        force_variant=force_variant)
    torch.cuda.synchronize()
    return out, lse, plan, gqa.gqa_prefill_poll()


def check_paged(q, k, v, page_size, seed, what, rows=None, **force):
    kc, vc, table = make_paged_cache(k, v, page_size, seed)
    out_p, lse_p, plan_p, status = run_paged(q, kc, vc, table, k.shape[0], SCALE, **force)
    assert status == 0, f"{what}: device status {status}"
    # Paged calls may prefer the CTA pair where dense ones would not: the dense
    # call runs the variant the paged plan chose (the same plan, so the same tiles).
    dense_force = dict(force)
    if not dense_force.get("force_variant"):
        dense_force["force_variant"] = plan_p["variant"]
    out_d, lse_d, plan_d = run_gpu(q, k, v, SCALE, **dense_force)
    assert plan_p == plan_d
    assert torch.equal(out_p, out_d) and torch.equal(lse_p, lse_d), f"{what}: paged != dense"
    if rows is None:
        ref_o, ref_l = oracle.paged_attention(q, kc, vc, table, k.shape[0], SCALE)
        check_close(out_p.double().cpu().numpy(), lse_p.double().cpu().numpy(), ref_o, ref_l, what)
    else:
        ref_o, ref_l = oracle.paged_attention(q, kc, vc, table, k.shape[0], SCALE, rows=rows)
        got_o, got_l = gather_rows(out_p, lse_p, rows)
        check_close(got_o, got_l, ref_o, ref_l, what)
    return plan_p


PAGE_SIZES = [16, 32, 48, 64, 128, SERVING_PAGE_SIZE, 1024]
SHAPES = [(1, 1), (5, 300), (43, 300), (100, 100), (129, 1000), (22, 2000)]


@pytest.mark.parametrize("page_size", PAGE_SIZES)
@pytest.mark.parametrize("q_len,kv_len", SHAPES)
@pytest.mark.parametrize("variant", [1, 2])
def test_paged_small_shapes_every_element(cuda_device, page_size, q_len, kv_len, variant):
    q, k, v = make_qkv(q_len, kv_len, seed=3 * q_len + kv_len + page_size)
    plan = check_paged(q, k, v, page_size, seed=kv_len + page_size,
                       what=f"{q_len}x{kv_len} page {page_size}", force_variant=variant)
    assert plan["variant"] == variant


@pytest.mark.parametrize("page_size", [16, SERVING_PAGE_SIZE])
@pytest.mark.parametrize("splits,grid,variant", [(3, 0, 1), (3, 5, 1), (2, 0, 2), (3, 6, 2),
                                                 (-1, 0, 1), (-1, 5, 1), (-1, 0, 2), (-1, 6, 2)])
def test_paged_split_tail_every_element(cuda_device, page_size, splits, grid, variant):
    q, k, v = make_qkv(129, 1000, seed=91)
    plan = check_paged(q, k, v, page_size, seed=92, what=f"split {splits} grid {grid}",
                       force_splits=splits, force_grid=grid, force_variant=variant)
    assert plan["variant"] == variant


def test_one_page_longer_than_the_sequence(cuda_device):
    q, k, v = make_qkv(43, 300, seed=5)
    check_paged(q, k, v, 4096, seed=6, what="page 4096")


@pytest.mark.parametrize("name,page_size", [("q4096_kv32768", SERVING_PAGE_SIZE),
                                            ("q4096_kv32768", 16),
                                            ("q512_kv32768", SERVING_PAGE_SIZE),
                                            ("q4096_kv8192", 48),
                                            ("q512_kv4096_kbias", SERVING_PAGE_SIZE)])
def test_paged_workload_full_size(cuda_device, name, page_size):
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    rows = item_cover_rows(w.q_len, w.n_q_heads, sample_rows(w.q_len, w.n_q_heads, 1200, seed=8))
    plan = check_paged(q, k, v, page_size, seed=w.seed, what=f"{name} page {page_size}", rows=rows)
    assert unchecked_items(rows, w.q_len, 21 * plan["variant"]) == []


@pytest.mark.parametrize("q_len,kv_len", [(512, 32768), (512, 4096), (43, 300), (1, 2000)])
def test_paged_plan_is_the_host_plan(cuda_device, q_len, kv_len):
    """The plan a paged call reports is the host-only paged planner's for the
    device's SM count and co-resident pairs (paged calls may prefer the pair)."""
    import gqa_chunked_prefill_gb300 as gqa
    q, k, v = make_qkv(q_len, kv_len, seed=q_len + kv_len)
    kc, vc, table = make_paged_cache(k, v, SERVING_PAGE_SIZE, seed=31)
    _, _, plan, status = run_paged(q, kc, vc, table, kv_len, SCALE)
    assert status == 0
    sms, pairs = gqa.gqa_prefill_device_info()
    _, host_plan = gqa.gqa_prefill_make_plan_paged_varlen([0, q_len], [kv_len], 24, 4, 256, sms,
                                                          max_pairs=pairs)
    assert plan == host_plan


@pytest.mark.parametrize("bad", ["past_end", "negative"])
@pytest.mark.parametrize("variant", [1, 2])
def test_block_table_entry_outside_cache_reads_zeros(cuda_device, bad, variant):
    """An entry outside [0, num_pages) is not followed: the device records
    GQA_ERR_PAGE_TABLE and the page's keys and values read as zeros, so the result
    equals the dense call on K/V with those rows zeroed."""
    q_len, kv_len, page_size, page = 43, 1000, 128, 3
    q, k, v = make_qkv(q_len, kv_len, seed=17)
    kc, vc, table = make_paged_cache(k, v, page_size, seed=18)
    table = table.clone()
    table[page] = kc.shape[0] + 5 if bad == "past_end" else -1
    out_p, lse_p, _, status = run_paged(q, kc, vc, table, kv_len, SCALE, force_variant=variant)
    assert status == 8
    k0, v0 = k.clone(), v.clone()
    k0[page * page_size:(page + 1) * page_size] = 0
    v0[page * page_size:(page + 1) * page_size] = 0
    out_d, lse_d, _ = run_gpu(q, k0, v0, SCALE, force_variant=variant)
    assert torch.equal(out_p, out_d) and torch.equal(lse_p, lse_d)
    import gqa_chunked_prefill_gb300 as gqa
    assert gqa.gqa_prefill_poll() == 0  # the poll cleared the word
