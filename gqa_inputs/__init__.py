"""Seeded synthetic inputs for chunked-prefill GQA attention.

This module only draws random numbers and shapes them; it holds none of the
attention arithmetic. Both the FP64 oracle (``oracle/``) and the CUDA path
(``gqa_chunked_prefill_gb300``) are fed from here, so the two sides see the
same bytes.

Workloads follow the shapes of the dedicated BF16 prefill kernel described in
"DCU使用技术报告（中篇）：gfx936 DCU上的Qwen3.5-27B Triton-ROCm Attention与GEMV深度优化实战",
§1 (24 query heads, 4 KV heads, head_dim 256, GQA ratio 6, BF16) and the
q_len x kv_len pairs measured in its §4 table (4096x8K, 4096x16K, 4096x32K,
3072x16K, 512x32K), plus the short-KV cases its §8 coverage rule asks for.

Recipe (one generator per shape, on the CPU so every machine gets the same
bytes): ``torch.Generator('cpu').manual_seed(seed)``; draw Q, then K, then V
as FP32 N(0, 1) and round each to BF16. The 512x4096 workload also draws, after
V, one bias vector per KV head with standard deviation 0.5, adds it to every
key of that head in FP32 and only then rounds K to BF16.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Optional

import torch

N_Q_HEADS = 24
N_KV_HEADS = 4
HEAD_DIM = 256
DEFAULT_SCALE = 1.0 / 16.0  # 1/sqrt(head_dim)


@dataclass(frozen=True)
class Workload:
    name: str
    q_len: int
    kv_len: int
    seed: int
    k_bias_std: Optional[float] = None  # per-KV-head key bias (N(0, std)), or None
    scale: float = DEFAULT_SCALE
    n_q_heads: int = N_Q_HEADS
    n_kv_heads: int = N_KV_HEADS
    head_dim: int = HEAD_DIM


# The seven shapes of the five workload families. Seeds are 1000 + 10*family + variant.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("q128_kv256", 128, 256, 1000),
        Workload("q512_kv4096_kbias", 512, 4096, 1010, k_bias_std=0.5),
        Workload("q4096_kv8192", 4096, 8192, 1020),
        Workload("q4096_kv16384", 4096, 16384, 1030),
        Workload("q3072_kv16384", 3072, 16384, 1031),
        Workload("q4096_kv32768", 4096, 32768, 1040),
        Workload("q512_kv32768", 512, 32768, 1041),
    )
}


def make_qkv(q_len: int, kv_len: int, seed: int, *, n_q_heads: int = N_Q_HEADS,
             n_kv_heads: int = N_KV_HEADS, head_dim: int = HEAD_DIM,
             k_bias_std: Optional[float] = None):
    """Return CPU BF16 tensors q [q_len,Hq,d], k [kv_len,Hkv,d], v [kv_len,Hkv,d]."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn((q_len, n_q_heads, head_dim), generator=g, dtype=torch.float32)
    k = torch.randn((kv_len, n_kv_heads, head_dim), generator=g, dtype=torch.float32)
    v = torch.randn((kv_len, n_kv_heads, head_dim), generator=g, dtype=torch.float32)
    if k_bias_std is not None:
        bias = torch.randn((n_kv_heads, head_dim), generator=g, dtype=torch.float32) * k_bias_std
        k = k + bias.unsqueeze(0)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def make_workload(w: Workload):
    return make_qkv(w.q_len, w.kv_len, w.seed, n_q_heads=w.n_q_heads,
                    n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, k_bias_std=w.k_bias_std)


# Page size of the serving engine's BF16 attention pages (DCU使用技术报告（中篇）, §8: 784).
SERVING_PAGE_SIZE = 784


def make_paged_cache(k: torch.Tensor, v: torch.Tensor, page_size: int, seed: int, *,
                     extra_pages: int = 3, fill: float = float("nan")):
    """Scatter one sequence's K/V [kv_len, Hkv, d] into paged caches.

    The cache has ceil(kv_len / page_size) + extra_pages pages; the sequence's
    logical pages go to distinct physical pages in a seeded random order, and
    every cache slot they do not fill (the other pages and the tail of the last
    one) holds ``fill`` (NaN by default: such slots must never reach a result).
    Returns (k_cache, v_cache [num_pages, page_size, Hkv, d] in k's dtype,
    block_table int32 [ceil(kv_len / page_size)]), all on the CPU.
    """
    kv_len = k.shape[0]
    n_log = -(-kv_len // page_size)
    num_pages = n_log + extra_pages
    g = torch.Generator("cpu").manual_seed(seed)
    table = torch.randperm(num_pages, generator=g)[:n_log].to(torch.int32)
    k_cache = torch.full((num_pages, page_size) + tuple(k.shape[1:]), fill, dtype=k.dtype)
    v_cache = torch.full((num_pages, page_size) + tuple(v.shape[1:]), fill, dtype=v.dtype)
    for i in range(n_log):
        lo, hi = i * page_size, min((i + 1) * page_size, kv_len)
        k_cache[int(table[i]), : hi - lo] = k[lo:hi]
        v_cache[int(table[i]), : hi - lo] = v[lo:hi]
    return k_cache, v_cache, table


def make_varlen(lens, seed: int):
    """A batch of sequences packed end to end. lens: [(q_len, kv_len), ...].
    Returns (q [sum q_len, 24, 256], k, v [sum kv_len, 4, 256] CPU BF16,
    cu_seqlens_q, cu_seqlens_k as lists of batch + 1 ints). Each sequence is drawn
    by make_qkv with seed + its index."""
    qs, ks, vs, cu_q, cu_k = [], [], [], [0], [0]
    for i, (ql, kl) in enumerate(lens):
        q, k, v = make_qkv(ql, kl, seed + i)
        qs.append(q), ks.append(k), vs.append(v)
        cu_q.append(cu_q[-1] + ql)
        cu_k.append(cu_k[-1] + kl)
    return torch.cat(qs), torch.cat(ks), torch.cat(vs), cu_q, cu_k


def make_paged_batch(k: torch.Tensor, v: torch.Tensor, cu_k, page_size: int, seed: int, *,
                     extra_pages: int = 5, fill: float = float("nan"), pad: int = 1 << 30):
    """Scatter every sequence of a packed batch into ONE shared paged cache.

    Pages go to distinct physical pages in a seeded random order across all
    sequences; unused slots hold ``fill``. Returns (k_cache, v_cache
    [num_pages, page_size, Hkv, d], block_table int32 [batch, bt_stride] whose
    unused entries hold ``pad``, kv_lens list)."""
    kv_lens = [cu_k[i + 1] - cu_k[i] for i in range(len(cu_k) - 1)]
    n_pages = [-(-kl // page_size) for kl in kv_lens]
    bt_stride = max(max(n_pages), 1)
    num_pages = sum(n_pages) + extra_pages
    g = torch.Generator("cpu").manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g).tolist()
    k_cache = torch.full((num_pages, page_size) + tuple(k.shape[1:]), fill, dtype=k.dtype)
    v_cache = torch.full((num_pages, page_size) + tuple(v.shape[1:]), fill, dtype=v.dtype)
    table = torch.full((len(kv_lens), bt_stride), pad, dtype=torch.int32)
    nxt = 0
    for b, kl in enumerate(kv_lens):
        for i in range(n_pages[b]):
            phys = perm[nxt]
            nxt += 1
            table[b, i] = phys
            lo, hi = cu_k[b] + i * page_size, min(cu_k[b] + (i + 1) * page_size, cu_k[b + 1])
            k_cache[phys, : hi - lo] = k[lo:hi]
            v_cache[phys, : hi - lo] = v[lo:hi]
    return k_cache, v_cache, table, kv_lens


def sample_rows(q_len: int, n_q_heads: int, n: int, seed: int) -> torch.Tensor:
    """A fixed, stratified set of (token, head) row ids ``t*n_q_heads + h``.

    Covers the first and last tokens, every head, and seeded random rows in
    between, so that both the diagonal region and long-prefix rows are checked.
    """
    total = q_len * n_q_heads
    if n >= total:
        return torch.arange(total, dtype=torch.int64)
    fixed = []
    for t in (0, 1, q_len // 2, q_len - 2, q_len - 1):
        if 0 <= t < q_len:
            fixed.extend(t * n_q_heads + h for h in range(n_q_heads))
    g = torch.Generator("cpu").manual_seed(seed)
    extra = torch.randint(0, total, (max(n - len(fixed), 0),), generator=g)
    return torch.unique(torch.cat([torch.tensor(fixed, dtype=torch.int64), extra]))
