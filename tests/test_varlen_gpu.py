"""GPU parity of the batched (varlen) entry points.

A batch packs several chunks end to end (decode rows, short chunks over long
prefixes, empty sequences, long chunks). Checks: every output element against
the oracle applied per sequence; bit-identity with one call per sequence when
items are not split (each item is then computed by one CTA or pair over the
same tiles in the same order, wherever it lands in the batch); split tails
across sequences; the paged batch (one shared cache, seeded page order, NaN in
unused slots, out-of-range padding in unused table entries that a read would
report) bit-identical to the dense batch.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_inputs import make_paged_batch, make_varlen
from tests.gpu_helpers import check_close, run_gpu

pytestmark = pytest.mark.gpu
SCALE = 1.0 / 16.0

BATCHES = {
    "mixed": [(43, 300), (1, 4096), (0, 50), (129, 1000), (22, 22)],
    "decode": [(1, 1000)] * 7 + [(4, 5000)],
    "chunks": [(512, 4096), (300, 6000), (700, 700)],
    "many": [(1 + (7 * i) % 60, 61 + (37 * i) % 900) for i in range(40)],
}


def run_varlen(q, k, v, cu_q, cu_k, **force):
    import gqa_chunked_prefill_gb300 as gqa
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev).contiguous() for t in (q, k, v))
    out = torch.full_like(qd, float("nan"))
    lse = torch.full((qd.shape[0], 24), float("nan"), dtype=torch.float32, device=dev)
    _, plan = gqa.gqa_prefill_attn_varlen_ex(qd, kd, vd, out, lse, cu_q, cu_k, 24, 4, 256, SCALE,
                                             **force)
    torch.cuda.synchronize()
    assert gqa.gqa_prefill_poll() == 0
    return out, lse, plan


@pytest.mark.parametrize("name", list(BATCHES))
@pytest.mark.parametrize("variant", [1, 2])
def test_varlen_every_element(cuda_device, name, variant):
    q, k, v, cu_q, cu_k = make_varlen(BATCHES[name], seed=300)
    out, lse, plan = run_varlen(q, k, v, cu_q, cu_k, force_variant=variant)
    assert plan["variant"] == variant
    ref_o, ref_l = oracle.varlen_attention(q, k, v, cu_q, cu_k, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l, name)


@pytest.mark.parametrize("name", ["mixed", "chunks", "many"])
@pytest.mark.parametrize("variant", [1, 2])
def test_varlen_matches_one_call_per_sequence_bit_for_bit(cuda_device, name, variant):
    q, k, v, cu_q, cu_k = make_varlen(BATCHES[name], seed=400)
    out, lse, _ = run_varlen(q, k, v, cu_q, cu_k, force_splits=1, force_variant=variant)
    for b in range(len(cu_q) - 1):
        if cu_q[b + 1] == cu_q[b]:
            continue
        ob, lb, _ = run_gpu(q[cu_q[b]:cu_q[b + 1]], k[cu_k[b]:cu_k[b + 1]], v[cu_k[b]:cu_k[b + 1]],
                            SCALE, force_splits=1, force_variant=variant)
        assert torch.equal(out[cu_q[b]:cu_q[b + 1]], ob), f"sequence {b}"
        assert torch.equal(lse[cu_q[b]:cu_q[b + 1]], lb), f"sequence {b}"


@pytest.mark.parametrize("splits,grid,variant", [(3, 0, 1), (3, 7, 1), (2, 0, 2), (4, 6, 2),
                                                 (32, 0, 1), (-1, 0, 1), (-1, 7, 1), (-1, 0, 2),
                                                 (-1, 6, 2)])
def test_varlen_split_tails_every_element(cuda_device, splits, grid, variant):
    q, k, v, cu_q, cu_k = make_varlen(BATCHES["decode"] + [(43, 300)], seed=500)
    out, lse, plan = run_varlen(q, k, v, cu_q, cu_k, force_splits=splits, force_grid=grid,
                                force_variant=variant)
    # A balanced tail on a small grid may find worker boundaries on item boundaries
    # (nothing split, no workspace); on the full grid it cuts items.
    assert plan["workspace_bytes"] > 0 or (splits < 0 and grid > 0)
    assert plan["kernels_per_call"] == (2 if plan["workspace_bytes"] else 1)
    assert (plan["tail_splits"] == 0) == (splits < 0)
    ref_o, ref_l = oracle.varlen_attention(q, k, v, cu_q, cu_k, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                f"split {splits} grid {grid}")


@pytest.mark.parametrize("page_size", [16, 784])
@pytest.mark.parametrize("name", ["mixed", "decode", "chunks"])
@pytest.mark.parametrize("variant", [1, 2])
def test_paged_varlen_matches_dense_and_oracle(cuda_device, page_size, name, variant):
    import gqa_chunked_prefill_gb300 as gqa
    q, k, v, cu_q, cu_k = make_varlen(BATCHES[name], seed=600)
    kc, vc, table, kv_lens = make_paged_batch(k, v, cu_k, page_size, seed=601)
    dev = torch.device("cuda:0")
    qd = q.to(dev)
    out = torch.empty_like(qd)
    lse = torch.empty((qd.shape[0], 24), dtype=torch.float32, device=dev)
    _, plan = gqa.gqa_prefill_attn_paged_varlen_ex(qd, kc.to(dev), vc.to(dev), table.to(dev),
                                                   table.shape[1], kc.shape[0], page_size, out, lse,
                                                   cu_q, kv_lens, 24, 4, 256, SCALE,
                                                   force_variant=variant)
    torch.cuda.synchronize()
    assert gqa.gqa_prefill_poll() == 0  # no table entry past a sequence's pages was read
    out_d, lse_d, plan_d = run_varlen(q, k, v, cu_q, cu_k, force_variant=variant)
    assert plan == plan_d
    assert torch.equal(out, out_d) and torch.equal(lse, lse_d)
    ref_o, ref_l = oracle.paged_varlen_attention(q, kc, vc, table, cu_q, kv_lens, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                f"paged {name} page {page_size}")


def test_largest_batch(cuda_device):
    lens = [(1 + i % 5, 1 + i % 5 + (13 * i) % 200) for i in range(128)]
    q, k, v, cu_q, cu_k = make_varlen(lens, seed=700)
    out, lse, plan = run_varlen(q, k, v, cu_q, cu_k)
    ref_o, ref_l = oracle.varlen_attention(q, k, v, cu_q, cu_k, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l, "128 seqs")


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("splits", [0, 3, -1])
@pytest.mark.parametrize("poison", [float("nan"), float("inf")])
def test_a_sequences_values_do_not_reach_its_neighbours(cuda_device, variant, splits, poison):
    """Sequences are independent (the single-sequence definition, applied per
    sequence): one sequence whose Q, K and V hold Inf or NaN leaves every other
    sequence's output and LSE bit-identical to the clean run. K/V lengths are not
    multiples of the 128-key tile, so the last tile of each sequence reaches into the
    next sequence's rows."""
    lens = [(43, 300), (5, 1000), (129, 1001), (22, 22), (7, 700), (1, 33)]
    q, k, v, cu_q, cu_k = make_varlen(lens, seed=900)
    force = dict(force_variant=variant, force_splits=splits)
    out_c, lse_c, _ = run_varlen(q, k, v, cu_q, cu_k, **force)
    ref_o, ref_l = oracle.varlen_attention(q, k, v, cu_q, cu_k, SCALE)
    check_close(out_c.double().cpu().numpy(), lse_c.double().cpu().numpy(), ref_o, ref_l, "clean")
    for bad in range(len(lens)):
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        q2[cu_q[bad]:cu_q[bad + 1]] = poison
        k2[cu_k[bad]:cu_k[bad + 1]] = poison
        v2[cu_k[bad]:cu_k[bad + 1]] = poison
        out_p, lse_p, _ = run_varlen(q2, k2, v2, cu_q, cu_k, **force)
        for b in range(len(lens)):
            if b == bad:
                continue
            r = slice(cu_q[b], cu_q[b + 1])
            assert torch.equal(out_p[r], out_c[r]), f"sequence {b} changed when {bad} was poisoned"
            assert torch.equal(lse_p[r], lse_c[r]), f"sequence {b} LSE changed ({bad} poisoned)"
