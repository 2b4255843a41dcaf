"""Independent numpy FP64 restatement of chunked-prefill causal GQA attention.

TEST INFRASTRUCTURE ONLY (tiny shapes). It builds the whole score matrix of
each query head, applies the bottom-right causal mask as an explicit boolean
matrix, and takes a row softmax — the textbook form — so that it shares no
structure with the per-row loop of ``gqa_oracle.cpp``. It also offers the
"per-head MHA over replicated K/V heads" form of GQA, which needs no head
mapping at all: with K/V heads repeated n_q_heads/n_kv_heads times in order,
query head h simply meets K/V head h.

Sources: QK^T, causal mask, softmax and PV per the dedicated prefill kernel of
DCU使用技术报告（中篇）, §2; query heads 6g..6g+5 on KV head g per
gfx936 DCU上实现INT8 QK MMAC：分页访存、Fragment映射与GQA适配, §5.2.
"""
from __future__ import annotations

import numpy as np


def causal_mask(q_len: int, kv_len: int) -> np.ndarray:
    """Boolean [q_len, kv_len]: True where query token t may see key j.

    Token t of the chunk sits at absolute position kv_len - q_len + t.
    """
    pos = np.arange(q_len)[:, None] + (kv_len - q_len)
    keys = np.arange(kv_len)[None, :]
    return keys <= pos


def mha(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """Per-head attention with equal head counts: q [T,H,d], k/v [S,H,d]."""
    q_len, n_heads, _ = q.shape
    kv_len = k.shape[0]
    mask = causal_mask(q_len, kv_len)
    out = np.empty_like(q, dtype=np.float64)
    lse = np.empty((q_len, n_heads), np.float64)
    for h in range(n_heads):
        s = scale * (q[:, h, :] @ k[:, h, :].T)          # [T, S]
        s = np.where(mask, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        z = e.sum(axis=1, keepdims=True)
        out[:, h, :] = (e / z) @ v[:, h, :]
        lse[:, h] = (m + np.log(z))[:, 0]
    return out, lse


def gqa_by_replication(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """GQA as MHA over K/V heads repeated in order (head g -> copies 6g..6g+5)."""
    rep = q.shape[1] // k.shape[1]
    return mha(q, np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1), scale)
