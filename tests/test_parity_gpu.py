"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle.

Small shapes are compared on every output element; they span several 21-token
query tiles and 128-key KV tiles with ragged tails (q_len not a multiple of 21,
kv_len not a multiple of 128), tiles straddling the causal diagonal, and the
single-token/single-key degenerate cases. The seven workload shapes run at full
size in the same launch configuration as the benchmark and are compared on a
row sample that checks every work item: the first and last token of every
21-token query tile in every KV group (the last token depends on every KV piece
of a split item), plus a stratified random sample; an assertion counts the items
(one-CTA and CTA-pair tiling) the sample leaves unchecked and requires none.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_inputs import WORKLOADS, make_qkv, make_workload, sample_rows
from tests.gpu_helpers import check_close, gather_rows, item_cover_rows, run_gpu, unchecked_items

pytestmark = pytest.mark.gpu
SCALE = 1.0 / 16.0

Q_LENS = [1, 2, 5, 6, 7, 21, 22, 42, 43, 127, 128, 129]
KV_EXTRA = ["q", "q+1", 255, 256, 257, 1000]


def _kv(q_len, spec):
    if spec == "q":
        return q_len
    if spec == "q+1":
        return q_len + 1
    return spec


CASES = sorted({(ql, _kv(ql, s)) for ql in Q_LENS for s in KV_EXTRA if _kv(ql, s) >= ql})


@pytest.mark.parametrize("q_len,kv_len", CASES)
@pytest.mark.parametrize("variant", [1, 2])
def test_small_shapes_every_element(cuda_device, q_len, kv_len, variant):
    q, k, v = make_qkv(q_len, kv_len, seed=7 * q_len + kv_len)
    out, lse, plan = run_gpu(q, k, v, SCALE, force_variant=variant)
    assert plan["variant"] == variant and plan["q_tiles"] == -(-q_len // (21 * variant))
    ref_o, ref_l = oracle.attention(q, k, v, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                f"{q_len}x{kv_len}")


@pytest.mark.parametrize("q_len,kv_len", [(22, 1000), (129, 1000), (43, 257), (7, 700), (300, 300)])
@pytest.mark.parametrize("splits,grid,variant", [(2, 0, 1), (3, 0, 1), (7, 0, 1), (3, 5, 1),
                                                 (2, 11, 1), (4, 1, 1), (2, 0, 2), (3, 0, 2),
                                                 (3, 6, 2), (2, 10, 2), (5, 2, 2)])
def test_split_tail_every_element(cuda_device, q_len, kv_len, splits, grid, variant):
    """Items split into KV pieces and merged: all items (grid >= items) or only the
    items after whole rounds on a few CTAs (small grid); one CTA or a CTA pair per item."""
    q, k, v = make_qkv(q_len, kv_len, seed=11 * q_len + kv_len)
    out, lse, plan = run_gpu(q, k, v, SCALE, force_splits=splits, force_grid=grid,
                             force_variant=variant)
    assert plan["grid"] <= (grid or plan["num_sms"]) and plan["variant"] == variant
    assert plan["kernels_per_call"] == (2 if plan["tail_splits"] > 1 and plan["tail_items"] else 1)
    ref_o, ref_l = oracle.attention(q, k, v, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                f"{q_len}x{kv_len} splits {splits} grid {grid}")


@pytest.mark.parametrize("q_len,kv_len", [(22, 4096), (129, 2200), (300, 4096)])
@pytest.mark.parametrize("splits,grid,variant", [(16, 0, 1), (31, 0, 1), (17, 9, 1), (16, 0, 2),
                                                 (20, 6, 2)])
def test_many_pieces_every_element(cuda_device, q_len, kv_len, splits, grid, variant):
    """16 or more KV pieces per item: the merge takes a block per output row, its
    warps each combining a subset of the pieces (the decode-sized merge)."""
    q, k, v = make_qkv(q_len, kv_len, seed=23 * q_len + kv_len)
    out, lse, plan = run_gpu(q, k, v, SCALE, force_splits=splits, force_grid=grid,
                             force_variant=variant)
    # S is capped at the fewest KV tiles of an item (17 for 129x2200)
    assert plan["tail_items"] > 0 and 16 <= plan["tail_splits"] <= splits
    assert plan["kernels_per_call"] == 2
    ref_o, ref_l = oracle.attention(q, k, v, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                f"{q_len}x{kv_len} splits {splits} grid {grid}")


BALANCED = -1  # force_splits value of the balanced tail (GQA_FORCE_BALANCED_TAIL)


@pytest.mark.parametrize("q_len,kv_len", [(22, 1000), (129, 1000), (43, 257), (7, 700), (300, 300),
                                          (1, 129), (512, 4096)])
@pytest.mark.parametrize("grid,variant", [(0, 1), (0, 2), (5, 1), (3, 1), (6, 2), (10, 2), (152, 1),
                                          (38, 1), (76, 2)])
def test_balanced_tail_every_element(cuda_device, q_len, kv_len, grid, variant):
    """The balanced tail: the tail items' tiles laid end to end and cut into equal
    shares, one per CTA (pair), whole rounds first where they fit; items cut at
    any tile, pieces merged from per-worker slots."""
    q, k, v = make_qkv(q_len, kv_len, seed=19 * q_len + kv_len)
    out, lse, plan = run_gpu(q, k, v, SCALE, force_splits=BALANCED, force_grid=grid,
                             force_variant=variant)
    assert plan["variant"] == variant and plan["grid"] <= (grid or plan["num_sms"])
    assert plan["tail_splits"] == 0
    ref_o, ref_l = oracle.attention(q, k, v, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                f"{q_len}x{kv_len} balanced grid {grid}")


@pytest.mark.parametrize("q_len,kv_len", [(129, 1000), (300, 300)])
@pytest.mark.parametrize("grid,variant", [(1, 1), (5, 1), (2, 2), (6, 2)])
def test_whole_items_on_few_ctas(cuda_device, q_len, kv_len, grid, variant):
    """No split, more items than CTAs: each CTA (pair) walks many whole items in turn."""
    q, k, v = make_qkv(q_len, kv_len, seed=13 * q_len + kv_len)
    out, lse, plan = run_gpu(q, k, v, SCALE, force_splits=1, force_grid=grid,
                             force_variant=variant)
    assert plan["tail_splits"] == 1 and plan["kernels_per_call"] == 1 and plan["grid"] == grid
    ref_o, ref_l = oracle.attention(q, k, v, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                f"{q_len}x{kv_len} whole items on {grid} CTAs")


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("variant,splits", [(0, 0), (1, 0), (2, 0), (2, -1)])
def test_workload_full_size_every_item(cuda_device, name, variant, splits):
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    out, lse, plan = run_gpu(q, k, v, w.scale, force_variant=variant, force_splits=splits)
    rows = item_cover_rows(w.q_len, w.n_q_heads,
                           sample_rows(w.q_len, w.n_q_heads,
                                       1200 if w.q_len * w.kv_len > 4e6 else 4000, seed=5))
    tpi = 21 * plan["variant"]
    assert unchecked_items(rows, w.q_len, tpi) == [], "items without a compared row"
    assert plan["n_items"] == 4 * -(-w.q_len // tpi)
    ref_o, ref_l = oracle.attention(q, k, v, w.scale, rows=rows)
    got_o, got_l = gather_rows(out, lse, rows)
    check_close(got_o, got_l, ref_o, ref_l, name)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_kv_head_bias_workload_every_element(cuda_device):
    """The 512 x 4096 shape with a per-KV-head key bias, checked on every row."""
    w = WORKLOADS["q512_kv4096_kbias"]
    q, k, v = make_workload(w)
    out, lse, _ = run_gpu(q, k, v, w.scale)
    ref_o, ref_l = oracle.attention(q, k, v, w.scale)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l, w.name)


def test_peaked_rows_with_large_scores(cuda_device):
    """Per-token key offsets make rows strongly peaked and push the running max up
    many times along the KV sweep, exercising the deferred O rescale."""
    q_len, kv_len = 64, 2000
    q, k, v = make_qkv(q_len, kv_len, seed=77)
    ramp = torch.linspace(0, 6, kv_len).reshape(kv_len, 1, 1)
    k = (k.float() + ramp * q.float().mean(dim=(0, 1)).sign()).to(torch.bfloat16)
    out, lse, _ = run_gpu(q, k, v, 0.2)
    ref_o, ref_l = oracle.attention(q, k, v, 0.2)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l, "peaked")


def test_lse_may_be_null(cuda_device):
    q, k, v = make_qkv(50, 300, seed=3)
    out_a, _, _ = run_gpu(q, k, v, SCALE, with_lse=False)
    out_b, _, _ = run_gpu(q, k, v, SCALE, with_lse=True)
    assert torch.equal(out_a, out_b)


@pytest.mark.parametrize("q_len", [1, 2, 3, 4])
@pytest.mark.parametrize("kv_len", [4096, 32768])
@pytest.mark.parametrize("splits,variant", [(0, 0), (32, 1), (24, 2), (5, 1), (-1, 1), (-1, 2)])
def test_decode_shapes_every_element(cuda_device, q_len, kv_len, splits, variant):
    """Decode-sized chunks (one to four new tokens, 6 to 24 live MMA rows) over a long
    prefix: the whole KV range is cut into many pieces and merged."""
    q, k, v = make_qkv(q_len, kv_len, seed=17 * q_len + kv_len)
    out, lse, plan = run_gpu(q, k, v, SCALE, force_splits=splits, force_variant=variant)
    if splits > 0:
        assert plan["tail_splits"] == splits and plan["kernels_per_call"] == 2
    if splits < 0:
        assert plan["tail_splits"] == 0 and plan["kernels_per_call"] == 2
    ref_o, ref_l = oracle.attention(q, k, v, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                f"decode {q_len}x{kv_len} S {splits}")
