"""FP64 CPU oracle for chunked-prefill causal GQA attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product package never
imports this module, and this module never imports the product package; the
two share nothing but the seeded inputs of ``gqa_inputs``.

``paged_gather()`` reads one sequence's keys and values out of paged caches
through its block table; ``paged_attention()`` is attention on what it returns.

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
