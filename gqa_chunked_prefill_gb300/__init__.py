"""GB300 (sm_103a) chunked-prefill causal GQA attention.

A C-ABI CUDA library (libgqa_prefill.so, declared in include/gqa_prefill.h)
plus this thin binding. ``attention()`` is the convenience call on torch CUDA
tensors; the ``gqa_prefill_*`` functions mirror the C entry points one to one.
"""
from ._binding import (FORCE_BALANCED_TAIL, GqaError, GqaStatus, gqa_prefill_abi_version, gqa_prefill_attn,  # noqa: F401
                       gqa_prefill_attn_ex, gqa_prefill_attn_noalloc, gqa_prefill_attn_paged,
                       gqa_prefill_attn_paged_ex, gqa_prefill_attn_fp8qk, gqa_prefill_attn_fp8qk_ex,
                       gqa_prefill_attn_paged_varlen, gqa_prefill_attn_paged_varlen_ex,
                       gqa_prefill_attn_fp8qk_varlen_ex, gqa_prefill_attn_paged_fp8qk_varlen_ex,
                       gqa_prefill_attn_fp8qkpv, gqa_prefill_attn_fp8qkpv_ex, gqa_quantize_v_fp8,
                       gqa_prefill_attn_varlen, gqa_prefill_attn_varlen_ex, gqa_prefill_device_info,
                       gqa_prefill_make_plan, gqa_prefill_make_plan_paged_varlen,
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


def _check_bf16(*ts):
    import torch
    for t in ts:
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.bfloat16):
            raise ValueError("tensors must be contiguous bf16 CUDA tensors")


def _outputs(q, out, lse, with_lse):
    import torch
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    return out, lse


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float = HEAD_DIM ** -0.5,
                     out=None, lse=None, stream=None, with_lse: bool = True):
    """A batch packed end to end: sequence b is query rows cu_seqlens_q[b] ..
    cu_seqlens_q[b+1]-1 over key rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 (host
    int sequences). q [total_q, 24, 256], k/v [total_kv, 4, 256] bf16 CUDA."""
    _check_bf16(q, k, v)
    out, lse = _outputs(q, out, lse, with_lse)
    gqa_prefill_attn_varlen(q, k, v, out, lse, list(cu_seqlens_q), list(cu_seqlens_k), q.shape[1],
                            k.shape[1], q.shape[2], scale, stream)
    return out, lse


def attention_paged(q, k_cache, v_cache, block_table, kv_lens, cu_seqlens_q=None,
                    scale: float = HEAD_DIM ** -0.5, out=None, lse=None, stream=None,
                    with_lse: bool = True):
    """K/V from paged caches [num_pages, page_size, 4, 256] through block_table
    (int32 CUDA [batch, pages] or [pages] for one sequence). kv_lens: host ints per
    sequence (or one int); cu_seqlens_q: host [batch + 1] (default: one sequence)."""
    import torch
    _check_bf16(q, k_cache, v_cache)
    if block_table.dtype != torch.int32 or not block_table.is_cuda:
        raise ValueError("block_table must be an int32 CUDA tensor")
    table = block_table.reshape(1, -1) if block_table.dim() == 1 else block_table
    kv_lens = [int(kv_lens)] if isinstance(kv_lens, int) else [int(x) for x in kv_lens]
    cu_q = list(cu_seqlens_q) if cu_seqlens_q is not None else [0, q.shape[0]]
    out, lse = _outputs(q, out, lse, with_lse)
    gqa_prefill_attn_paged_varlen_ex(q, k_cache, v_cache, table.contiguous(), table.shape[1],
                                     k_cache.shape[0], k_cache.shape[1], out, lse, cu_q, kv_lens,
                                     q.shape[1], k_cache.shape[2], q.shape[2], scale,
                                     stream=stream)
    return out, lse


def quantize_fp8(x, cu_seqlens=None, stream=None):
    """E4M3 codes (uint8, same shape) and FP32 scales of every 256-value vector of x.
    Query tensors [rows, 24, 256] give scales [rows, 24]; key tensors [rows, 4, 256]
    give head-major scales [4, stride] in the layout the FP8 attention reads (with
    cu_seqlens, each sequence's columns start on a multiple of 4)."""
    import torch
    _check_bf16(x)
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if x.shape[1] == N_Q_HEADS:
        scales = torch.empty(x.shape[:2], dtype=torch.float32, device=x.device)
        gqa_quantize_q_fp8(x, codes, scales, x.shape[0], x.shape[1], x.shape[2], stream=stream)
        return codes, scales
    cu = list(cu_seqlens) if cu_seqlens is not None else [0, x.shape[0]]
    _, cols = key_scale_columns(cu)
    scales = torch.empty((x.shape[1], max(4, cols)), dtype=torch.float32, device=x.device)
    gqa_quantize_k_fp8_varlen(x, codes, scales, cu, x.shape[1], x.shape[2], scales.shape[1],
                              stream=stream)
    return codes, scales


def attention_fp8qk(q_codes, q_scale, k_codes, k_scale, v, cu_seqlens_q=None, cu_seqlens_k=None,
                    scale: float = HEAD_DIM ** -0.5, out=None, lse=None, stream=None,
                    with_lse: bool = True):
    """Attention with QK^T on E4M3 codes (from quantize_fp8) and BF16 V; one sequence
    unless cu_seqlens_q / cu_seqlens_k (host) describe a packed batch."""
    out, lse = _outputs(q_codes, out, lse, with_lse)
    cu_q = list(cu_seqlens_q) if cu_seqlens_q is not None else [0, q_codes.shape[0]]
    cu_k = list(cu_seqlens_k) if cu_seqlens_k is not None else [0, k_codes.shape[0]]
    gqa_prefill_attn_fp8qk_varlen_ex(q_codes, q_scale, k_codes, k_scale, k_scale.shape[1], v,
                                     out, lse, cu_q, cu_k, q_codes.shape[1], k_codes.shape[1],
                                     q_codes.shape[2], scale, stream=stream)
    return out, lse
