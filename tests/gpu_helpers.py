"""Shared helpers for the GPU tests: run the CUDA path through the C ABI and
compare it with the FP64 oracle at the acceptance tolerance.

Acceptance (elementwise on O, mean on O, absolute on LSE):
    |out - ref| <= 1e-2 + 1e-2 * |ref|,  mean |out - ref| <= 2e-3,  |lse - ref| <= 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

ATOL, RTOL, MEAN_TOL, LSE_TOL = 1e-2, 1e-2, 2e-3, 1e-3


def run_gpu(q, k, v, scale, force_splits=0, force_grid=0, force_variant=0, with_lse=True,
            stream=None):
    """q, k, v: CPU or CUDA bf16. Returns (out bf16 CUDA, lse fp32 CUDA or None, plan)."""
    import gqa_chunked_prefill_gb300 as gqa
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev).contiguous() for t in (q, k, v))
    q_len, hq, d = qd.shape
    kv_len, hkv, _ = kd.shape
    out = torch.empty_like(qd)
    lse = torch.empty((q_len, hq), dtype=torch.float32, device=dev) if with_lse else None
    _, plan = gqa.gqa_prefill_attn_ex(qd, kd, vd, out, lse, q_len, kv_len, hq, hkv, d, scale,
                                      stream=stream, force_splits=force_splits,
                                      force_grid=force_grid, force_variant=force_variant)
    torch.cuda.synchronize()
    assert gqa.gqa_prefill_poll() == 0, "device-side wait timed out"
    return out, lse, plan


def check_close(out_rows: np.ndarray, lse_rows, ref_out: np.ndarray, ref_lse, what: str = ""):
    """out_rows/ref_out: [..., d] float64; lse: [...] or None."""
    err = np.abs(out_rows - ref_out)
    bound = ATOL + RTOL * np.abs(ref_out)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (
        f"{what}: elementwise tolerance exceeded at {worst}: got {out_rows[worst]}, "
        f"ref {ref_out[worst]}, max err {err.max():.3e}")
    assert err.mean() <= MEAN_TOL, f"{what}: mean |err| {err.mean():.3e} > {MEAN_TOL}"
    if lse_rows is not None:
        lerr = np.abs(lse_rows - ref_lse)
        assert np.all(lerr <= LSE_TOL), f"{what}: LSE max err {lerr.max():.3e}"


def gather_rows(out: torch.Tensor, lse, rows):
    """Rows t*Hq + h of out [q_len,Hq,d] / lse [q_len,Hq] as float64 numpy."""
    hq, d = out.shape[1], out.shape[2]
    r = torch.as_tensor(rows, dtype=torch.int64, device=out.device)
    o = out.reshape(-1, d).index_select(0, r).double().cpu().numpy()
    l = lse.reshape(-1).index_select(0, r).double().cpu().numpy() if lse is not None else None
    return o, l


TOK_PER_TILE = 21  # tokens of one 128-row MMA tile (21 tokens x 6 heads)
GROUP = 6          # query heads per KV head


def item_cover_rows(q_len: int, n_q_heads: int = 24, extra=None) -> np.ndarray:
    """Row ids t*Hq + h that touch every work item of a call, whatever its kernel variant.

    A work item is one query tile (21 tokens, or 42 for a CTA pair = two 21-token
    tiles) of one KV group (6 query heads). For every 21-token tile i and group g
    this takes the tile's first token and its last token (the last sees every KV
    tile of the item, so it depends on every KV piece of a split item), with the
    head inside the group rotating with i so all six heads of a group appear.
    ``extra`` (row ids) is merged in. Returns sorted unique int64 row ids."""
    rows = []
    n_tiles = -(-q_len // TOK_PER_TILE)
    for i in range(n_tiles):
        first = TOK_PER_TILE * i
        last = min(first + TOK_PER_TILE - 1, q_len - 1)
        for g in range(n_q_heads // GROUP):
            rows.append(first * n_q_heads + GROUP * g + i % GROUP)
            rows.append(last * n_q_heads + GROUP * g + (i + 3) % GROUP)
    if extra is not None:
        rows.extend(int(r) for r in np.asarray(extra).reshape(-1))
    return np.unique(np.asarray(rows, dtype=np.int64))


def unchecked_items(rows, q_len: int, tok_per_item: int, n_q_heads: int = 24):
    """Items (query tile of tok_per_item tokens, KV group) that the sampled rows do
    not check: no row at all, or no row of the item's last token (the one row
    that every KV piece of a split item contributes to). Returns a list of
    (tile, group); empty means every item and every piece is compared."""
    rows = np.asarray(rows, dtype=np.int64)
    tok, head = rows // n_q_heads, rows % n_q_heads
    n_tiles = -(-q_len // tok_per_item)
    seen = np.zeros((n_tiles, n_q_heads // GROUP), bool)
    seen_last = np.zeros_like(seen)
    seen[tok // tok_per_item, head // GROUP] = True
    last_tok = np.minimum((tok // tok_per_item + 1) * tok_per_item, q_len) - 1
    is_last = tok == last_tok
    seen_last[tok[is_last] // tok_per_item, head[is_last] // GROUP] = True
    bad = np.argwhere(~(seen & seen_last))
    return [tuple(int(x) for x in b) for b in bad]
