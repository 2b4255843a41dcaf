"""FP64 CPU oracle for chunked-prefill causal GQA attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product package never
imports this module, and this module never imports the product package; the
two share nothing but the seeded inputs of ``gqa_inputs``.

``paged_gather()`` reads one sequence's keys and values out of paged caches
through its block table; ``paged_attention()`` is attention on what it returns.
``varlen_attention()`` / ``paged_varlen_attention()`` apply the definition to
each sequence of a packed batch. ``quantize_e4m3()`` and ``fp8qk_attention()``
define the quantised-QK^T path; ``quantize_v_e4m3()``, ``fp8pv_attention()``
and ``fp8pv_p_bound()`` the quantised PV (per-channel V scales, P rounded to
E4M3, and the bound on what that rounding can change).

``attention()`` runs the plain C++ definition in ``gqa_oracle.cpp`` (explicit
full-row softmax in FP64, one std::thread per row at a time). ``restate_numpy``
holds an independent numpy restatement used to cross-check it on tiny shapes.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from typing import Optional, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.cpp")
_LIB = os.path.join(_HERE, "libgqa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (plain -O2, no fast-math,
    no FMA contraction, so x86 and Arm hosts give the same bits)."""
    stamp = _LIB + ".arch"
    try:
        same_arch = open(stamp).read().strip() == platform.machine()
    except OSError:
        same_arch = False
    if (force or not same_arch or not os.path.exists(_LIB)
            or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", _LIB + ".tmp"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
        with open(stamp, "w") as f:
            f.write(platform.machine())
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        f = lib.gqa_oracle_attn
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                      ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                      ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        _lib = lib
    return _lib


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def attention(q, k, v, scale: float, rows=None, n_threads: Optional[int] = None,
              with_prob_sum: bool = False):
    """FP64 attention of a q_len chunk at the end of a kv_len prefix.

    q: [q_len, Hq, d]; k, v: [kv_len, Hkv, d] (torch or numpy; BF16 is widened
    exactly). ``rows`` optionally lists row ids t*Hq + h to compute.
    Returns (out, lse[, prob_sum]) as numpy FP64: out [q_len, Hq, d] and
    lse [q_len, Hq] when ``rows`` is None, else out [n_rows, d], lse [n_rows].
    """
    lib = _load()
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    q_len, hq, d = q64.shape
    kv_len, hkv, d2 = k64.shape
    assert d2 == d and v64.shape == k64.shape
    if rows is not None:
        rows64 = np.ascontiguousarray(np.asarray(
            rows.numpy() if isinstance(rows, torch.Tensor) else rows, dtype=np.int64))
        n_rows = rows64.shape[0]
        out = np.empty((n_rows, d), np.float64)
        lse = np.empty((n_rows,), np.float64)
        psum = np.empty((n_rows,), np.float64) if with_prob_sum else None
        rows_ptr = rows64.ctypes.data
    else:
        n_rows = 0
        out = np.empty((q_len, hq, d), np.float64)
        lse = np.empty((q_len, hq), np.float64)
        psum = np.empty((q_len, hq), np.float64) if with_prob_sum else None
        rows_ptr = None
    rc = lib.gqa_oracle_attn(q64.ctypes.data, k64.ctypes.data, v64.ctypes.data,
                             q_len, kv_len, hq, hkv, d, float(scale), rows_ptr, n_rows,
                             out.ctypes.data, lse.ctypes.data,
                             psum.ctypes.data if psum is not None else None,
                             int(n_threads or host_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected arguments (rc={rc})")
    if with_prob_sum:
        return out, lse, psum
    return out, lse


def paged_gather(k_cache, v_cache, block_table, kv_len: int):
    """K and V of one sequence, read out of paged caches.

    Follows "gfx936 DCU上实现INT8 QK MMAC：分页访存、Fragment映射与GQA适配", §3: a
    logical key token is looked up in the block table, which names its physical
    block, and sits in that block at its slot. Here the slot of key j is
    j mod page_size and its block is block_table[j div page_size].
    k_cache, v_cache: [num_pages, page_size, Hkv, d]; block_table: integer
    [>= ceil(kv_len / page_size)]. Returns (k, v) [kv_len, Hkv, d] in the
    caches' dtype (torch in, torch out; numpy in, numpy out).
    """
    table = np.asarray(block_table.cpu().numpy() if isinstance(block_table, torch.Tensor)
                       else block_table, dtype=np.int64)
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    j = np.arange(kv_len, dtype=np.int64)
    block = table[j // page_size]
    slot = j % page_size
    if kv_len and (block.min() < 0 or block.max() >= num_pages):
        raise ValueError("block table entry outside the cache")
    if isinstance(k_cache, torch.Tensor):
        bi, si = torch.from_numpy(block), torch.from_numpy(slot)
        return k_cache[bi, si], v_cache[bi, si]
    return k_cache[block, slot], v_cache[block, slot]


def paged_attention(q, k_cache, v_cache, block_table, kv_len: int, scale: float, rows=None,
                    n_threads: Optional[int] = None):
    """``attention()`` of q over the sequence ``paged_gather()`` reads from the caches."""
    k, v = paged_gather(k_cache, v_cache, block_table, kv_len)
    return attention(q, k, v, scale, rows=rows, n_threads=n_threads)


# --- batches of sequences ------------------------------------------------------

def varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float,
                     n_threads: Optional[int] = None):
    """A batch packed end to end: sequence b is query rows cu_q[b] .. cu_q[b+1]-1
    and keys cu_k[b] .. cu_k[b+1]-1, each its own chunk-at-the-end attention
    (the single-sequence definition, applied per sequence; nothing crosses
    sequences). Returns (out [total_q, Hq, d], lse [total_q, Hq]) FP64."""
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    out = np.zeros(q64.shape, np.float64)
    lse = np.zeros(q64.shape[:2], np.float64)
    for b in range(len(cu_seqlens_q) - 1):
        q0, q1 = cu_seqlens_q[b], cu_seqlens_q[b + 1]
        k0, k1 = cu_seqlens_k[b], cu_seqlens_k[b + 1]
        if q1 == q0:
            continue
        o, l = attention(q64[q0:q1], k64[k0:k1], v64[k0:k1], scale, n_threads=n_threads)
        out[q0:q1], lse[q0:q1] = o, l
    return out, lse


def paged_varlen_attention(q, k_cache, v_cache, block_table, cu_seqlens_q, kv_lens, scale: float,
                           n_threads: Optional[int] = None):
    """Batch with K/V in one paged cache: sequence b reads its kv_lens[b] keys
    through block-table row b (``paged_gather``)."""
    q64 = _f64(q)
    out = np.zeros(q64.shape, np.float64)
    lse = np.zeros(q64.shape[:2], np.float64)
    table = np.asarray(block_table.cpu().numpy() if isinstance(block_table, torch.Tensor)
                       else block_table)
    for b in range(len(kv_lens)):
        q0, q1 = cu_seqlens_q[b], cu_seqlens_q[b + 1]
        if q1 == q0:
            continue
        k, v = paged_gather(k_cache, v_cache, table[b], kv_lens[b])
        o, l = attention(q64[q0:q1], k, v, scale, n_threads=n_threads)
        out[q0:q1], lse[q0:q1] = o, l
    return out, lse


# --- quantised QK^T -------------------------------------------------------------
#
# "gfx936 DCU上实现INT8 QK MMAC：分页访存、Fragment映射与GQA适配", §1 and §4: each query
# vector (token, query head) and each key vector (token, KV head) gets one
# symmetric dynamic scale s = max|x| / qmax and codes x / s; scores are restored
# as (code_q . code_k) * s_q * s_k * softmax_scale before the softmax. The codes
# here are FP8 E4M3 (qmax 448) instead of the report's INT8 (qmax 127).

def e4m3_values() -> np.ndarray:
    """Value of every non-negative E4M3 code 0x00 .. 0x7E (0x7F is NaN).

    E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits. Exponent
    field 0 is subnormal (m/8 * 2^-6); otherwise (1 + m/8) * 2^(e - 7). There is
    no infinity; 0x7E = 448 is the largest finite value.
    """
    vals = np.empty(127, np.float64)
    for code in range(127):
        e, m = code >> 3, code & 7
        vals[code] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def e4m3_encode(x) -> np.ndarray:
    """Codes of FP32 values: round to nearest, ties to the even code, saturating at
    +-448, sign kept (a negative value that rounds to zero gives 0x80)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    vals = e4m3_values()
    a = np.abs(x)
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, 126)  # first value >= a
    lo = np.clip(hi - 1, 0, 126)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= vals[126], 126, code)  # saturate
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    """FP64 value of E4M3 codes (0x7F / 0xFF, NaN, are not produced here)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag = e4m3_values()[np.minimum(c & 0x7F, 126)]
    return np.where(c & 0x80, -mag, mag)


def quantize_e4m3(x):
    """Per-vector quantisation of [..., d] values: s = max|x| / 448 and codes of
    x / s, both in FP32 with IEEE round-to-nearest division; a vector of zeros
    gets s = 0 and codes 0. Returns (codes uint8 [..., d], scales float32 [...])."""
    x32 = np.asarray(x.float().numpy() if isinstance(x, torch.Tensor) else x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    s = (amax / np.float32(448.0)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    codes = e4m3_encode((x32 / safe[..., None]).astype(np.float32))
    codes = np.where((s > 0)[..., None], codes, np.uint8(0)).astype(np.uint8)
    return codes, s


def dequantize_e4m3(codes, scales) -> np.ndarray:
    """code * s in FP64 (exact: a 4-bit-significand value times an FP32 scale)."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def fp8qk_attention(q_codes, q_scale, k_codes, k_scale, v, scale: float, rows=None,
                    n_threads: Optional[int] = None):
    """Attention of the dequantised query and keys (the quantised-QK^T result):
    q_codes [q_len, Hq, d] with q_scale [q_len, Hq]; k_codes [kv_len, Hkv, d] with
    k_scale [kv_len, Hkv] (token-major here); v as for ``attention``."""
    return attention(dequantize_e4m3(q_codes, q_scale), dequantize_e4m3(k_codes, k_scale), v,
                     scale, rows=rows, n_threads=n_threads)


# --- quantised PV ----------------------------------------------------------------
#
# The same report's final submission also multiplies P by V in 8 bits ("INT8 PV")
# without saying how V or P are scaled. The reading here, for GB300's FP8 tensor
# path: V gets one symmetric scale per (KV head, channel) over the call's keys,
# s_v = max_j |v[j,g,c]| / 448 with codes E4M3(v / s_v) (the rule of
# quantize_e4m3, applied along the key axis), so that the scale multiplies a
# column of P.V after the product; P is rounded to E4M3 as the MMA operand, while
# the softmax normaliser keeps the exact probabilities. The result below is the
# plain definition the method approximates: attention of the dequantised Q, K
# and V with exact probabilities; fp8pv_p_bound bounds what rounding P can change.

def quantize_v_e4m3(v):
    """Per (KV head, channel) quantisation of v [kv_len, Hkv, d]: the kv_len values of
    channel c of KV head g form one vector (quantize_e4m3's rule). Returns (codes
    uint8 [kv_len, Hkv, d], scales float32 [Hkv, d])."""
    v32 = np.asarray(v.float().numpy() if isinstance(v, torch.Tensor) else v, dtype=np.float32)
    codes_t, s = quantize_e4m3(np.ascontiguousarray(v32.transpose(1, 2, 0)))
    return np.ascontiguousarray(codes_t.transpose(2, 0, 1)), s


def dequantize_v_e4m3(codes, scales) -> np.ndarray:
    """codes [kv_len, Hkv, d] times the channel scales [Hkv, d], in FP64 (exact)."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[None, :, :]


def fp8pv_attention(q_codes, q_scale, k_codes, k_scale, v_codes, v_scale, scale: float,
                    rows=None, n_threads: Optional[int] = None):
    """The quantised QK^T and PV result: attention of the dequantised query, keys
    and values (FP64, exact probabilities). q: codes [q_len, Hq, d] + scales
    [q_len, Hq]; k: codes [kv_len, Hkv, d] + scales [kv_len, Hkv]; v: codes
    [kv_len, Hkv, d] + channel scales [Hkv, d]."""
    return attention(dequantize_e4m3(q_codes, q_scale), dequantize_e4m3(k_codes, k_scale),
                     dequantize_v_e4m3(v_codes, v_scale), scale, rows=rows, n_threads=n_threads)


E4M3_P_REL = 2.0 ** -4    # half a unit in the last place of a normal E4M3 value, relative
E4M3_P_FLOOR = 2.0 ** -16  # half the subnormal step 2^-10 of P stored as 2^6 * p, p <= 4


def fp8pv_p_bound(q, k, v, scale: float, rows=None, chunk: int = 256) -> np.ndarray:
    """Per-element bound on how far rounding the probabilities to E4M3 moves the
    output, for q [q_len, Hq, d], k, v [kv_len, Hkv, d] (FP64 values: the
    dequantised inputs), rows as in ``attention``:

        B[t, h, c] = sum_j (2^-4 p_j + 2^-16) |v[j, g, c]| / sum_j p_j,
        p_j = exp(s_j - max_i s_i)  over the visible keys j of row (t, h).

    Why: the kernel stores each probability as P = 2^6 * 2^(x_j - m), m a running
    maximum at most 2 (log2 units) below the row maximum seen so far, so P <= 256
    fits E4M3 unsaturated; rounding P moves it by at most 2^-4 P (normal range)
    or 2^-10 (subnormal). In the final normalisation the first term becomes
    2^-4 times the exact softmax weight and the second at most 2^-16 / sum_j p_j,
    since the normaliser taken against a maximum m <= max_i x_i is at least the
    one taken against the maximum itself."""
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    q_len, hq, d = q64.shape
    kv_len, hkv, _ = k64.shape
    group = hq // hkv
    p0 = kv_len - q_len
    ids = np.arange(q_len * hq) if rows is None else np.asarray(
        rows.numpy() if isinstance(rows, torch.Tensor) else rows, dtype=np.int64)
    out = np.empty((len(ids), d), np.float64)
    for a in range(0, len(ids), chunk):
        blk = ids[a:a + chunk]
        t, h = blk // hq, blk % hq
        for g in np.unique(h // group):
            sel = np.nonzero(h // group == g)[0]
            s = scale * q64[t[sel], h[sel]] @ k64[:, g].T            # [rows, kv_len]
            s[np.arange(kv_len)[None, :] > (p0 + t[sel])[:, None]] = -np.inf
            p = np.exp(s - s.max(axis=1, keepdims=True))
            w = E4M3_P_REL * p + np.where(np.isfinite(s), E4M3_P_FLOOR, 0.0)
            out[a + sel] = (w @ np.abs(v64[:, g])) / p.sum(axis=1, keepdims=True)
    return out if rows is not None else out.reshape(q_len, hq, d)
