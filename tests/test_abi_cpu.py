"""CPU-only checks of the C ABI: the library loads without a GPU, exports every
function include/*.h declares, refuses bad calls before touching CUDA, and its
host planner behaves (no empty splits, deterministic, grid within SM count)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gqa():
    import __graft_entry__
    __graft_entry__.build()
    import gqa_chunked_prefill_gb300 as mod
    return mod


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(gqa):
    names = declared_functions()
    assert "gqa_prefill_attn" in names and len(names) >= 6
    lib = ctypes.CDLL(gqa._binding._LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_abi_version(gqa):
    assert gqa.gqa_prefill_abi_version() == 1


def test_refusals_before_any_cuda_call(gqa):
    S = gqa.GqaStatus
    f = lambda *a: gqa.gqa_prefill_attn(*a, stream=0, check=False)
    assert f(16, 16, 16, 16, None, 4, 3, 24, 4, 256, 0.0625) == S.ERR_SHAPE
    assert f(16, 16, 16, 16, None, -1, 3, 24, 4, 256, 0.0625) == S.ERR_SHAPE
    assert f(16, 16, 16, 16, None, 4, 8, 24, 4, 256, 0.0) == S.ERR_SHAPE
    assert f(16, 16, 16, 16, None, 4, 8, 24, 4, 256, float("nan")) == S.ERR_SHAPE
    assert f(16, 16, 16, 16, None, 4, 8, 32, 4, 256, 0.0625) == S.ERR_UNSUPPORTED
    assert f(16, 16, 16, 16, None, 4, 8, 24, 4, 64, 0.0625) == S.ERR_UNSUPPORTED
    assert f(None, 16, 16, 16, None, 4, 8, 24, 4, 256, 0.0625) == S.ERR_NULL
    assert f(16, 16, 16, None, None, 4, 8, 24, 4, 256, 0.0625) == S.ERR_NULL
    assert f(16, 16, 24, 16, None, 4, 8, 24, 4, 256, 0.0625) == S.ERR_ALIGN
    assert f(16, 16, 16, 16, 20, 4, 8, 24, 4, 256, 0.0625) == S.ERR_ALIGN
    assert f(None, None, None, None, None, 0, 0, 24, 4, 256, 0.0625) == S.OK  # empty chunk
    for s in S:
        assert isinstance(gqa.gqa_status_string(int(s)), str)


SHAPES = [(1, 1), (21, 21), (22, 5000), (128, 256), (512, 4096), (4096, 8192), (4096, 16384),
          (3072, 16384), (4096, 32768), (512, 32768)]


@pytest.mark.parametrize("q_len,kv_len", SHAPES)
@pytest.mark.parametrize("sms", [148, 152])
def test_planner_invariants(gqa, q_len, kv_len, sms):
    _, p = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, sms)
    q_tiles = -(-q_len // 21)
    assert p["q_tiles"] == q_tiles and p["n_items"] == 4 * q_tiles
    assert p["n_units"] == p["n_items"] * p["splits"]
    assert 1 <= p["grid"] <= sms and p["grid"] == min(p["n_units"], sms)
    # no split may be empty: splits <= KV tiles of the shortest item
    p0 = kv_len - q_len
    shortest = -(-(p0 + min(21, q_len)) // 128)
    assert 1 <= p["splits"] <= shortest
    assert p["kernels_per_call"] == (2 if p["splits"] > 1 else 1)
    expect_ws = p["splits"] * q_len * 24 * 257 * 4 if p["splits"] > 1 else 0
    assert p["workspace_bytes"] == expect_ws
    # the busiest CTA carries at least the average load
    total = 0
    for qt in range(q_tiles):
        nt = -(-(p0 + min(21 * (qt + 1), q_len)) // 128)
        total += 4 * nt
    assert p["est_makespan_tiles"] * p["grid"] >= total
    _, again = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, sms)
    assert again == p


def test_forced_splits_are_capped(gqa):
    _, p = gqa.gqa_prefill_make_plan(128, 256, 24, 4, 256, 148, force_splits=64)
    assert p["splits"] == 2  # shortest item covers keys 0..148 -> 2 KV tiles
    _, p = gqa.gqa_prefill_make_plan(512, 32768, 24, 4, 256, 148, force_splits=5)
    assert p["splits"] == 5 and p["kernels_per_call"] == 2


def test_make_plan_validates(gqa):
    S = gqa.GqaStatus
    assert gqa.gqa_prefill_make_plan(5, 4, 24, 4, 256, 148, check=False)[0] == S.ERR_SHAPE
    assert gqa.gqa_prefill_make_plan(5, 8, 24, 4, 256, 0, check=False)[0] == S.ERR_SHAPE
    assert gqa.gqa_prefill_make_plan(5, 8, 24, 2, 256, 148, check=False)[0] == S.ERR_UNSUPPORTED
