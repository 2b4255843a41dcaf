"""ctypes binding of libgqa_prefill.so (argument marshalling only).

Every entry point keeps the name and argument order of include/gqa_prefill.h.
Tensors may be passed as torch tensors (their data_ptr is used) or as raw
integer addresses; streams as torch.cuda.Stream, raw handles, or None for the
current torch stream. All computation happens in the CUDA library: if it is
missing this module raises at import time instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import enum
import os

# GQA_PREFILL_LIB selects another build of the same library, e.g. the bounds-checked
# libgqa_prefill_checked.so next to this file (the tests run the parity suite on it).
_LIB_PATH = os.environ.get("GQA_PREFILL_LIB") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libgqa_prefill.so")


class GqaStatus(enum.IntEnum):
    OK = 0
    ERR_NULL = 1
    ERR_SHAPE = 2
    ERR_UNSUPPORTED = 3
    ERR_ALIGN = 4
    ERR_CUDA = 5
    ERR_DEVICE_TIMEOUT = 6
    ERR_SCRATCH = 7
    ERR_PAGE_TABLE = 8
    ERR_BOUNDS = 9


class GqaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{GqaStatus(status).name}: {msg}")
        self.status = GqaStatus(status)


class PrefillOpts(ctypes.Structure):
    _fields_ = [("force_splits", ctypes.c_int), ("force_grid", ctypes.c_int),
                ("wait_timeout_us", ctypes.c_uint32),
                ("fwd_event_begin", ctypes.c_void_p), ("fwd_event_end", ctypes.c_void_p),
                ("test_withhold_q", ctypes.c_int), ("force_variant", ctypes.c_int),
                ("reserved", ctypes.c_int * 1)]


class PrefillPlan(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int), ("q_tiles", ctypes.c_int), ("n_items", ctypes.c_int),
                ("head_rounds", ctypes.c_int), ("tail_items", ctypes.c_int),
                ("tail_splits", ctypes.c_int), ("n_units", ctypes.c_int), ("grid", ctypes.c_int),
                ("kernels_per_call", ctypes.c_int), ("variant", ctypes.c_int),
                ("total_tiles", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("est_makespan_tiles", ctypes.c_int64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is not built; run gqa_chunked_prefill_gb300.build.build() "
                      "(there is no non-CUDA implementation to fall back to)")

lib = ctypes.CDLL(_LIB_PATH)
_vp, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_ATTN_ARGS = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]
lib.gqa_prefill_attn.argtypes = _ATTN_ARGS
lib.gqa_prefill_attn.restype = _i
lib.gqa_prefill_attn_ex.argtypes = _ATTN_ARGS + [ctypes.POINTER(PrefillOpts), ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_attn_ex.restype = _i
lib.gqa_prefill_attn_noalloc.argtypes = _ATTN_ARGS
lib.gqa_prefill_attn_noalloc.restype = _i
_PAGED_ARGS = [_vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]
lib.gqa_prefill_attn_paged.argtypes = _PAGED_ARGS
lib.gqa_prefill_attn_paged.restype = _i
lib.gqa_prefill_attn_paged_ex.argtypes = _PAGED_ARGS + [ctypes.POINTER(PrefillOpts),
                                                        ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_attn_paged_ex.restype = _i
lib.gqa_quantize_q_fp8.argtypes = [_vp, _vp, _vp, _i, _i, _i, _vp]
lib.gqa_quantize_q_fp8.restype = _i
lib.gqa_quantize_k_fp8.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp]
lib.gqa_quantize_k_fp8.restype = _i
_FP8_ARGS = [_vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]
lib.gqa_prefill_attn_fp8qk.argtypes = _FP8_ARGS
lib.gqa_prefill_attn_fp8qk.restype = _i
lib.gqa_prefill_attn_fp8qk_ex.argtypes = _FP8_ARGS + [ctypes.POINTER(PrefillOpts),
                                                      ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_attn_fp8qk_ex.restype = _i
_VARLEN_ARGS = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _vp]
lib.gqa_prefill_attn_varlen.argtypes = _VARLEN_ARGS
lib.gqa_prefill_attn_varlen.restype = _i
lib.gqa_prefill_attn_varlen_ex.argtypes = _VARLEN_ARGS + [ctypes.POINTER(PrefillOpts),
                                                          ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_attn_varlen_ex.restype = _i
_PVARLEN_ARGS = [_vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _vp]
lib.gqa_prefill_attn_paged_varlen.argtypes = _PVARLEN_ARGS
lib.gqa_prefill_attn_paged_varlen.restype = _i
lib.gqa_prefill_attn_paged_varlen_ex.argtypes = _PVARLEN_ARGS + [ctypes.POINTER(PrefillOpts),
                                                                 ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_attn_paged_varlen_ex.restype = _i
lib.gqa_prefill_make_plan_varlen.argtypes = [_vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                             ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_make_plan_varlen.restype = _i
lib.gqa_prefill_make_plan_paged_varlen.argtypes = [_vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                                   ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_make_plan_paged_varlen.restype = _i
lib.gqa_quantize_k_fp8_varlen.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]
lib.gqa_quantize_k_fp8_varlen.restype = _i
lib.gqa_prefill_attn_fp8qk_varlen_ex.argtypes = [_vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp,
                                                 _i, _i, _i, _i, _f, _vp,
                                                 ctypes.POINTER(PrefillOpts),
                                                 ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_attn_fp8qk_varlen_ex.restype = _i
lib.gqa_prefill_attn_paged_fp8qk_varlen_ex.argtypes = [
    _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _vp,
    ctypes.POINTER(PrefillOpts), ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_attn_paged_fp8qk_varlen_ex.restype = _i
lib.gqa_prefill_make_plan.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                      ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_make_plan.restype = _i
lib.gqa_prefill_device_info.argtypes = [ctypes.POINTER(_i), ctypes.POINTER(_i)]
lib.gqa_quantize_v_fp8.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp]
lib.gqa_quantize_v_fp8.restype = _i
_FP8PV_ARGS = [_vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]
lib.gqa_prefill_attn_fp8qkpv.argtypes = _FP8PV_ARGS
lib.gqa_prefill_attn_fp8qkpv.restype = _i
lib.gqa_prefill_attn_fp8qkpv_ex.argtypes = _FP8PV_ARGS + [ctypes.POINTER(PrefillOpts),
                                                          ctypes.POINTER(PrefillPlan)]
lib.gqa_prefill_attn_fp8qkpv_ex.restype = _i
lib.gqa_prefill_device_info.restype = _i
lib.gqa_prefill_poll.argtypes = [_vp, ctypes.POINTER(_i)]
lib.gqa_prefill_poll.restype = _i
lib.gqa_status_string.argtypes = [_i]
lib.gqa_status_string.restype = ctypes.c_char_p
lib.gqa_prefill_abi_version.argtypes = []
lib.gqa_prefill_abi_version.restype = _i


# force_splits value that asks for the balanced tail (GQA_FORCE_BALANCED_TAIL).
FORCE_BALANCED_TAIL = -1


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int) -> None:
    if rc != 0:
        raise GqaError(rc, lib.gqa_status_string(rc).decode())


def gqa_status_string(status: int) -> str:
    return lib.gqa_status_string(int(status)).decode()


def gqa_prefill_abi_version() -> int:
    return lib.gqa_prefill_abi_version()


def gqa_prefill_attn(q, k, v, out, lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale,
                     stream=None, check=True) -> int:
    rc = lib.gqa_prefill_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), q_len, kv_len,
                              n_q_heads, n_kv_heads, head_dim, scale, _stream(stream))
    if check:
        _check(rc)
    return rc


def gqa_prefill_attn_noalloc(q, k, v, out, lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim,
                             scale, stream=None, check=True) -> int:
    """The allocation-free entry point (split partials in the library's static scratch)."""
    rc = lib.gqa_prefill_attn_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), q_len,
                                      kv_len, n_q_heads, n_kv_heads, head_dim, scale,
                                      _stream(stream))
    if check:
        _check(rc)
    return rc


def gqa_prefill_attn_ex(q, k, v, out, lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale,
                        stream=None, force_splits=0, force_grid=0, force_variant=0,
                        wait_timeout_us=0, fwd_events=None, test_withhold_q=False, check=True):
    """fwd_events: optional (begin, end) torch.cuda.Event pair recorded around the
    attention kernel itself (not the split merge)."""
    opts = _opts(force_splits, force_grid, force_variant, wait_timeout_us, fwd_events,
                 test_withhold_q)
    plan = PrefillPlan()
    rc = lib.gqa_prefill_attn_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), q_len, kv_len,
                                 n_q_heads, n_kv_heads, head_dim, scale, _stream(stream),
                                 ctypes.byref(opts), ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def _opts(force_splits, force_grid, force_variant, wait_timeout_us, fwd_events, test_withhold_q):
    opts = PrefillOpts(force_splits=force_splits, force_grid=force_grid,
                       wait_timeout_us=wait_timeout_us, test_withhold_q=1 if test_withhold_q else 0,
                       force_variant=force_variant)
    if fwd_events is not None:
        opts.fwd_event_begin = fwd_events[0].cuda_event
        opts.fwd_event_end = fwd_events[1].cuda_event
    return opts


def gqa_prefill_attn_paged(q, k_cache, v_cache, block_table, num_pages, page_size, out, lse,
                           q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale, stream=None,
                           check=True) -> int:
    """K/V from paged caches [num_pages, page_size, 4, 256]; block_table: int32 device
    [ceil(kv_len / page_size)] (logical page -> physical page)."""
    rc = lib.gqa_prefill_attn_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                    num_pages, page_size, _ptr(out), _ptr(lse), q_len, kv_len,
                                    n_q_heads, n_kv_heads, head_dim, scale, _stream(stream))
    if check:
        _check(rc)
    return rc


def gqa_prefill_attn_paged_ex(q, k_cache, v_cache, block_table, num_pages, page_size, out, lse,
                              q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale, stream=None,
                              force_splits=0, force_grid=0, force_variant=0, wait_timeout_us=0,
                              fwd_events=None, test_withhold_q=False, check=True):
    opts = _opts(force_splits, force_grid, force_variant, wait_timeout_us, fwd_events,
                 test_withhold_q)
    plan = PrefillPlan()
    rc = lib.gqa_prefill_attn_paged_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                       num_pages, page_size, _ptr(out), _ptr(lse), q_len, kv_len,
                                       n_q_heads, n_kv_heads, head_dim, scale, _stream(stream),
                                       ctypes.byref(opts), ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def gqa_quantize_q_fp8(q, q_fp8, q_scale, q_len, n_q_heads, head_dim, stream=None,
                       check=True) -> int:
    """E4M3 codes [q_len, 24, 256] (uint8) and FP32 scales [q_len, 24] of BF16 q."""
    rc = lib.gqa_quantize_q_fp8(_ptr(q), _ptr(q_fp8), _ptr(q_scale), q_len, n_q_heads, head_dim,
                                _stream(stream))
    if check:
        _check(rc)
    return rc


def gqa_quantize_k_fp8(k, k_fp8, k_scale, kv_len, n_kv_heads, head_dim, k_scale_stride,
                       stream=None, check=True) -> int:
    """E4M3 codes [kv_len, 4, 256] (uint8) and FP32 scales [4, k_scale_stride] of BF16 k."""
    rc = lib.gqa_quantize_k_fp8(_ptr(k), _ptr(k_fp8), _ptr(k_scale), kv_len, n_kv_heads,
                                head_dim, k_scale_stride, _stream(stream))
    if check:
        _check(rc)
    return rc


def gqa_prefill_attn_fp8qk(q_fp8, q_scale, k_fp8, k_scale, k_scale_stride, v, out, lse, q_len,
                           kv_len, n_q_heads, n_kv_heads, head_dim, scale, stream=None,
                           check=True) -> int:
    rc = lib.gqa_prefill_attn_fp8qk(_ptr(q_fp8), _ptr(q_scale), _ptr(k_fp8), _ptr(k_scale),
                                    k_scale_stride, _ptr(v), _ptr(out), _ptr(lse), q_len, kv_len,
                                    n_q_heads, n_kv_heads, head_dim, scale, _stream(stream))
    if check:
        _check(rc)
    return rc


def gqa_prefill_attn_fp8qk_ex(q_fp8, q_scale, k_fp8, k_scale, k_scale_stride, v, out, lse, q_len,
                              kv_len, n_q_heads, n_kv_heads, head_dim, scale, stream=None,
                              force_splits=0, force_grid=0, force_variant=0, wait_timeout_us=0,
                              fwd_events=None, test_withhold_q=False, check=True):
    opts = _opts(force_splits, force_grid, force_variant, wait_timeout_us, fwd_events,
                 test_withhold_q)
    plan = PrefillPlan()
    rc = lib.gqa_prefill_attn_fp8qk_ex(_ptr(q_fp8), _ptr(q_scale), _ptr(k_fp8), _ptr(k_scale),
                                       k_scale_stride, _ptr(v), _ptr(out), _ptr(lse), q_len,
                                       kv_len, n_q_heads, n_kv_heads, head_dim, scale,
                                       _stream(stream), ctypes.byref(opts), ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def gqa_quantize_v_fp8(v, v_fp8t, v_scale, kv_len, n_kv_heads, head_dim, v_stride, stream=None,
                       check=True) -> int:
    """E4M3 codes of BF16 v [kv_len, 4, 256], transposed to [4, 256, v_stride] (uint8),
    and per-(KV head, channel) FP32 scales [4, 256]."""
    rc = lib.gqa_quantize_v_fp8(_ptr(v), _ptr(v_fp8t), _ptr(v_scale), kv_len, n_kv_heads,
                                head_dim, v_stride, _stream(stream))
    if check:
        _check(rc)
    return rc


def gqa_prefill_attn_fp8qkpv(q_fp8, q_scale, k_fp8, k_scale, k_scale_stride, v_fp8t, v_scale,
                             v_stride, out, lse, q_len, kv_len, n_q_heads, n_kv_heads, head_dim,
                             scale, stream=None, check=True) -> int:
    rc = lib.gqa_prefill_attn_fp8qkpv(_ptr(q_fp8), _ptr(q_scale), _ptr(k_fp8), _ptr(k_scale),
                                      k_scale_stride, _ptr(v_fp8t), _ptr(v_scale), v_stride,
                                      _ptr(out), _ptr(lse), q_len, kv_len, n_q_heads, n_kv_heads,
                                      head_dim, scale, _stream(stream))
    if check:
        _check(rc)
    return rc


def gqa_prefill_attn_fp8qkpv_ex(q_fp8, q_scale, k_fp8, k_scale, k_scale_stride, v_fp8t, v_scale,
                                v_stride, out, lse, q_len, kv_len, n_q_heads, n_kv_heads,
                                head_dim, scale, stream=None, force_splits=0, force_grid=0,
                                force_variant=0, wait_timeout_us=0, fwd_events=None,
                                test_withhold_q=False, check=True):
    opts = _opts(force_splits, force_grid, force_variant, wait_timeout_us, fwd_events,
                 test_withhold_q)
    plan = PrefillPlan()
    rc = lib.gqa_prefill_attn_fp8qkpv_ex(_ptr(q_fp8), _ptr(q_scale), _ptr(k_fp8), _ptr(k_scale),
                                         k_scale_stride, _ptr(v_fp8t), _ptr(v_scale), v_stride,
                                         _ptr(out), _ptr(lse), q_len, kv_len, n_q_heads,
                                         n_kv_heads, head_dim, scale, _stream(stream),
                                         ctypes.byref(opts), ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def _host_i32(xs):
    """A host int32 array (kept alive by the caller's reference) and its address."""
    arr = (ctypes.c_int32 * len(xs))(*[int(x) for x in xs])
    return arr, ctypes.addressof(arr)


def gqa_prefill_attn_varlen_ex(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, n_q_heads,
                               n_kv_heads, head_dim, scale, stream=None, force_splits=0,
                               force_grid=0, force_variant=0, wait_timeout_us=0, fwd_events=None,
                               test_withhold_q=False, check=True):
    """cu_seqlens_q / cu_seqlens_k: HOST sequences of batch + 1 ints (lists or arrays)."""
    cq, pq = _host_i32(cu_seqlens_q)
    ck, pk = _host_i32(cu_seqlens_k)
    opts = _opts(force_splits, force_grid, force_variant, wait_timeout_us, fwd_events,
                 test_withhold_q)
    plan = PrefillPlan()
    rc = lib.gqa_prefill_attn_varlen_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), pq, pk,
                                        len(cu_seqlens_q) - 1, n_q_heads, n_kv_heads, head_dim,
                                        scale, _stream(stream), ctypes.byref(opts),
                                        ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def gqa_prefill_attn_varlen(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, n_q_heads, n_kv_heads,
                            head_dim, scale, stream=None, check=True) -> int:
    cq, pq = _host_i32(cu_seqlens_q)
    ck, pk = _host_i32(cu_seqlens_k)
    rc = lib.gqa_prefill_attn_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), pq, pk,
                                     len(cu_seqlens_q) - 1, n_q_heads, n_kv_heads, head_dim,
                                     scale, _stream(stream))
    if check:
        _check(rc)
    return rc


def gqa_prefill_attn_paged_varlen_ex(q, k_cache, v_cache, block_table, bt_stride, num_pages,
                                     page_size, out, lse, cu_seqlens_q, kv_lens, n_q_heads,
                                     n_kv_heads, head_dim, scale, stream=None, force_splits=0,
                                     force_grid=0, force_variant=0, wait_timeout_us=0,
                                     fwd_events=None, test_withhold_q=False, check=True):
    """block_table: DEVICE int32 [batch, bt_stride]; cu_seqlens_q (batch + 1) and kv_lens
    (batch): HOST ints."""
    cq, pq = _host_i32(cu_seqlens_q)
    kl, pk = _host_i32(kv_lens)
    opts = _opts(force_splits, force_grid, force_variant, wait_timeout_us, fwd_events,
                 test_withhold_q)
    plan = PrefillPlan()
    rc = lib.gqa_prefill_attn_paged_varlen_ex(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), bt_stride, num_pages, page_size,
        _ptr(out), _ptr(lse), pq, pk, len(kv_lens), n_q_heads, n_kv_heads, head_dim, scale,
        _stream(stream), ctypes.byref(opts), ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def gqa_prefill_attn_paged_varlen(q, k_cache, v_cache, block_table, bt_stride, num_pages,
                                  page_size, out, lse, cu_seqlens_q, kv_lens, n_q_heads,
                                  n_kv_heads, head_dim, scale, stream=None, check=True) -> int:
    cq, pq = _host_i32(cu_seqlens_q)
    kl, pk = _host_i32(kv_lens)
    rc = lib.gqa_prefill_attn_paged_varlen(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), bt_stride, num_pages, page_size,
        _ptr(out), _ptr(lse), pq, pk, len(kv_lens), n_q_heads, n_kv_heads, head_dim, scale,
        _stream(stream))
    if check:
        _check(rc)
    return rc


def key_scale_columns(cu_seqlens_k):
    """Where gqa_quantize_k_fp8_varlen puts each sequence's key scales: column
    sum of the earlier kv_len rounded up to 4; returns (starts, columns used)."""
    starts, col = [], 0
    for b in range(len(cu_seqlens_k) - 1):
        starts.append(col)
        col += -(-(cu_seqlens_k[b + 1] - cu_seqlens_k[b]) // 4) * 4
    return starts, col


def gqa_quantize_k_fp8_varlen(k, k_fp8, k_scale, cu_seqlens_k, n_kv_heads, head_dim,
                              k_scale_stride, stream=None, check=True) -> int:
    ck, pk = _host_i32(cu_seqlens_k)
    rc = lib.gqa_quantize_k_fp8_varlen(_ptr(k), _ptr(k_fp8), _ptr(k_scale), pk,
                                       len(cu_seqlens_k) - 1, n_kv_heads, head_dim,
                                       k_scale_stride, _stream(stream))
    if check:
        _check(rc)
    return rc


def gqa_prefill_attn_fp8qk_varlen_ex(q_fp8, q_scale, k_fp8, k_scale, k_scale_stride, v, out, lse,
                                     cu_seqlens_q, cu_seqlens_k, n_q_heads, n_kv_heads, head_dim,
                                     scale, stream=None, force_splits=0, force_grid=0,
                                     force_variant=0, wait_timeout_us=0, fwd_events=None,
                                     test_withhold_q=False, check=True):
    cq, pq = _host_i32(cu_seqlens_q)
    ck, pk = _host_i32(cu_seqlens_k)
    opts = _opts(force_splits, force_grid, force_variant, wait_timeout_us, fwd_events,
                 test_withhold_q)
    plan = PrefillPlan()
    rc = lib.gqa_prefill_attn_fp8qk_varlen_ex(
        _ptr(q_fp8), _ptr(q_scale), _ptr(k_fp8), _ptr(k_scale), k_scale_stride, _ptr(v),
        _ptr(out), _ptr(lse), pq, pk, len(cu_seqlens_q) - 1, n_q_heads, n_kv_heads, head_dim,
        scale, _stream(stream), ctypes.byref(opts), ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def gqa_prefill_attn_paged_fp8qk_varlen_ex(q_fp8, q_scale, k_cache_fp8, k_scale, k_scale_stride,
                                           v_cache, block_table, bt_stride, num_pages, page_size,
                                           out, lse, cu_seqlens_q, kv_lens, n_q_heads, n_kv_heads,
                                           head_dim, scale, stream=None, force_splits=0,
                                           force_grid=0, force_variant=0, wait_timeout_us=0,
                                           fwd_events=None, test_withhold_q=False, check=True):
    cq, pq = _host_i32(cu_seqlens_q)
    kl, pk = _host_i32(kv_lens)
    opts = _opts(force_splits, force_grid, force_variant, wait_timeout_us, fwd_events,
                 test_withhold_q)
    plan = PrefillPlan()
    rc = lib.gqa_prefill_attn_paged_fp8qk_varlen_ex(
        _ptr(q_fp8), _ptr(q_scale), _ptr(k_cache_fp8), _ptr(k_scale), k_scale_stride,
        _ptr(v_cache), _ptr(block_table), bt_stride, num_pages, page_size, _ptr(out), _ptr(lse),
        pq, pk, len(kv_lens), n_q_heads, n_kv_heads, head_dim, scale, _stream(stream),
        ctypes.byref(opts), ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def gqa_prefill_make_plan_varlen(cu_seqlens_q, cu_seqlens_k, n_q_heads, n_kv_heads, head_dim,
                                 num_sms, max_pairs=-1, force_splits=0, force_grid=0,
                                 force_variant=0, check=True):
    cq, pq = _host_i32(cu_seqlens_q)
    ck, pk = _host_i32(cu_seqlens_k)
    plan = PrefillPlan()
    rc = lib.gqa_prefill_make_plan_varlen(pq, pk, len(cu_seqlens_q) - 1, n_q_heads, n_kv_heads,
                                          head_dim, num_sms, max_pairs, force_splits, force_grid,
                                          force_variant, ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def gqa_prefill_make_plan_paged_varlen(cu_seqlens_q, kv_lens, n_q_heads, n_kv_heads, head_dim,
                                       num_sms, max_pairs=-1, force_splits=0, force_grid=0,
                                       force_variant=0, check=True):
    """The plan of a paged call or paged batch (kv_lens: host ints per sequence)."""
    cq, pq = _host_i32(cu_seqlens_q)
    kl, pk = _host_i32(kv_lens)
    plan = PrefillPlan()
    rc = lib.gqa_prefill_make_plan_paged_varlen(pq, pk, len(cu_seqlens_q) - 1, n_q_heads,
                                                n_kv_heads, head_dim, num_sms, max_pairs,
                                                force_splits, force_grid, force_variant,
                                                ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def gqa_prefill_make_plan(q_len, kv_len, n_q_heads, n_kv_heads, head_dim, num_sms,
                          max_pairs=-1, force_splits=0, force_grid=0, force_variant=0,
                          check=True):
    """max_pairs < 0: num_sms / 2 co-resident CTA pairs (gqa_prefill_device_info gives
    the current device's number)."""
    plan = PrefillPlan()
    rc = lib.gqa_prefill_make_plan(q_len, kv_len, n_q_heads, n_kv_heads, head_dim, num_sms,
                                   max_pairs, force_splits, force_grid, force_variant,
                                   ctypes.byref(plan))
    if check:
        _check(rc)
    return rc, plan.as_dict()


def gqa_prefill_device_info():
    """(num_sms, max_pairs) the planner uses on the current device."""
    sms, pairs = _i(0), _i(0)
    _check(lib.gqa_prefill_device_info(ctypes.byref(sms), ctypes.byref(pairs)))
    return sms.value, pairs.value


def gqa_prefill_poll(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status word."""
    value = ctypes.c_int(0)
    _check(lib.gqa_prefill_poll(_stream(stream), ctypes.byref(value)))
    return value.value
