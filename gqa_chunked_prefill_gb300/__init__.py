"""GB300 (sm_103a) chunked-prefill causal GQA attention.

A C-ABI CUDA library (libgqa_prefill.so, declared in include/gqa_prefill.h)
plus this thin binding. ``attention()`` is the convenience call on torch CUDA
tensors; the ``gqa_prefill_*`` functions mirror the C entry points one to one.
"""
from ._binding import (GqaError, GqaStatus, gqa_prefill_abi_version, gqa_prefill_attn,  # noqa: F401
                       gqa_prefill_attn_ex, gqa_prefill_attn_noalloc, gqa_prefill_attn_paged,
                       gqa_prefill_attn_paged_ex, gqa_prefill_attn_fp8qk, gqa_prefill_attn_fp8qk_ex,
                       gqa_prefill_attn_paged_varlen, gqa_prefill_attn_paged_varlen_ex,
                       gqa_prefill_attn_fp8qk_varlen_ex, gqa_prefill_attn_paged_fp8qk_varlen_ex,
                       gqa_prefill_attn_varlen, gqa_prefill_attn_varlen_ex, gqa_prefill_make_plan,
                       gqa_prefill_make_plan_varlen, gqa_prefill_poll, gqa_quantize_k_fp8,
                       gqa_quantize_k_fp8_varlen, gqa_quantize_q_fp8, gqa_status_string,
                       key_scale_columns, lib)

N_Q_HEADS, N_KV_HEADS, HEAD_DIM = 24, 4, 256


def attention(q, k, v, scale: float = HEAD_DIM ** -0.5, out=None, lse=None, stream=None,
              with_lse: bool = True):
    """out[t,h] = attention of chunk token t (at position kv_len - q_len + t) over keys
    0..kv_len - q_len + t of KV head h // 6. q: [q_len, 24, 256] bf16 CUDA; k, v:
    [kv_len, 4, 256] bf16 CUDA. Returns (out, lse) with lse FP32 [q_len, 24] or None."""
    import torch
    q_len, n_q_heads, head_dim = q.shape
    kv_len, n_kv_heads, _ = k.shape
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.bfloat16):
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((q_len, n_q_heads), dtype=torch.float32, device=q.device)
    gqa_prefill_attn(q, k, v, out, lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale,
                     stream)
    return out, lse
