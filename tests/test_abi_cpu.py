"""CPU-only checks of the C ABI: the library loads without a GPU, exports every
function include/*.h declares, refuses bad calls before touching CUDA, and its
host planner behaves (deterministic, grid within SM count, tail split balances)."""
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


def test_bounds_checked_build_exports_the_same_abi(gqa):
    """build() also makes libgqa_prefill_checked.so (every epilogue store and merge
    access bounds-checked): same symbols, same ABI version, same status strings."""
    path = os.path.join(ROOT, "gqa_chunked_prefill_gb300", "libgqa_prefill_checked.so")
    lib = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} not exported by the bounds-checked build"
    lib.gqa_prefill_abi_version.restype = ctypes.c_int
    assert lib.gqa_prefill_abi_version() == gqa.gqa_prefill_abi_version()
    lib.gqa_status_string.restype = ctypes.c_char_p
    assert b"bounds" in lib.gqa_status_string(int(gqa.GqaStatus.ERR_BOUNDS))


def test_abi_version(gqa):
    assert gqa.gqa_prefill_abi_version() == 12


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


def test_paged_refusals_before_any_cuda_call(gqa):
    """Arguments: q, k_cache, v_cache, block_table, num_pages, page_size, out, lse,
    q_len, kv_len, heads..., scale."""
    S = gqa.GqaStatus
    f = lambda *a: gqa.gqa_prefill_attn_paged(*a, stream=0, check=False)
    ok = (16, 16, 16, 16, 4, 784, 16, None, 4, 8, 24, 4, 256, 0.0625)

    def call(**kw):
        names = ["q", "kc", "vc", "bt", "np", "ps", "out", "lse", "q_len", "kv_len", "hq", "hkv",
                 "d", "scale"]
        args = dict(zip(names, ok))
        args.update(kw)
        return f(*[args[n] for n in names])

    assert call(ps=0) == S.ERR_UNSUPPORTED
    assert call(ps=24) == S.ERR_UNSUPPORTED        # not a multiple of 16
    assert call(ps=-16) == S.ERR_UNSUPPORTED
    assert call(np=0) == S.ERR_SHAPE
    assert call(np=1 << 26, ps=16) == S.ERR_SHAPE   # 2^30 cache rows
    assert call(bt=None) == S.ERR_NULL
    assert call(bt=18) == S.ERR_ALIGN               # int32 table: 4-byte alignment
    assert call(kc=None) == S.ERR_NULL
    assert call(vc=24) == S.ERR_ALIGN
    assert call(kv_len=3) == S.ERR_SHAPE            # kv_len < q_len
    assert call(hkv=8) == S.ERR_UNSUPPORTED
    assert call(q=None, kc=None, vc=None, bt=None, out=None, q_len=0, kv_len=0) == S.OK
    assert call(q=None, kc=None, vc=None, bt=None, out=None, q_len=0, kv_len=0, ps=8) == \
        S.ERR_UNSUPPORTED


SHAPES = [(1, 1), (21, 21), (22, 5000), (128, 256), (512, 4096), (4096, 8192), (4096, 16384),
          (3072, 16384), (4096, 32768), (512, 32768)]


def _total_tiles(q_len, kv_len, tpi=21):
    p0, nq = kv_len - q_len, -(-q_len // tpi)
    return sum(4 * (-(-(p0 + min(tpi * (qt + 1), q_len)) // 128)) for qt in range(nq))


def _item_tiles(q_len, kv_len, tpi):
    """KV tiles of every item of one sequence in the call's order: query tiles
    from the last to the first, the 4 KV groups of each."""
    p0, nq = kv_len - q_len, -(-q_len // tpi)
    return [-(-(p0 + min(tpi * (qt + 1), q_len)) // 128) for qt in reversed(range(nq))
            for _ in range(4)]


def _balanced_cut(tail_tiles, G):
    """Pieces and split items when G workers take equal shares [x*W/G, (x+1)*W/G)
    of the tail's tiles laid end to end."""
    W = sum(tail_tiles)
    starts = [0]
    for t in tail_tiles:
        starts.append(starts[-1] + t)
    bounds = [x * W // G for x in range(G + 1)]
    pieces = sum(sum(1 for k in range(len(tail_tiles))
                     if starts[k] < bounds[x + 1] and starts[k + 1] > bounds[x]) for x in range(G))
    split = sum(1 for k in range(len(tail_tiles))
                if any(starts[k] < b < starts[k + 1] for b in bounds))
    return pieces, split


@pytest.mark.parametrize("q_len,kv_len", SHAPES)
@pytest.mark.parametrize("sms", [148, 152])
@pytest.mark.parametrize("force", [0, 1, 3, -1])
@pytest.mark.parametrize("variant", [0, 1, 2])
def test_planner_invariants(gqa, q_len, kv_len, sms, force, variant):
    _, p = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, sms, force_splits=force,
                                     force_variant=variant)
    assert p["variant"] in (1, 2) and (variant == 0 or p["variant"] == variant)
    cpi = p["variant"]  # CTAs per item
    tpi = 21 * cpi
    q_tiles = -(-q_len // tpi)
    n = 4 * q_tiles
    W = _total_tiles(q_len, kv_len, tpi)
    assert p["q_tiles"] == q_tiles and p["n_items"] == n and p["total_tiles"] == W
    shortest = -(-(kv_len - q_len + min(tpi, q_len)) // 128)
    assert p["grid"] % cpi == 0
    workers = p["grid"] // cpi
    head = min(p["head_rounds"] * workers, n)
    assert p["tail_items"] == n - head
    if p["tail_splits"] == 0:  # balanced tail
        assert force in (0, -1)
        tail = _item_tiles(q_len, kv_len, tpi)[head:]
        assert 1 <= len(tail) <= 512 and sum(tail) >= workers
        assert 1 <= workers <= sms // cpi
        pieces, split = _balanced_cut(tail, workers)
        assert p["n_units"] == head + pieces
        assert p["kernels_per_call"] == (2 if split else 1)
        assert p["workspace_bytes"] == (2 * workers * cpi * 128 * 257 * 4 if split else 0)
    else:
        assert 1 <= p["tail_splits"] <= max(shortest, 1)
        if force > 0:
            assert p["tail_splits"] == min(force, shortest)
        assert p["n_units"] == head + p["tail_items"] * p["tail_splits"]
        assert 1 <= workers <= min(sms // cpi, p["n_units"])
        split = p["tail_splits"] > 1 and p["tail_items"] > 0
        assert p["kernels_per_call"] == (2 if split else 1)
        assert p["workspace_bytes"] == (
            p["tail_items"] * p["tail_splits"] * cpi * 128 * 257 * 4 if split else 0)
    assert p["est_makespan_tiles"] * workers >= W  # the busiest worker carries at least the mean
    _, again = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, sms, force_splits=force,
                                         force_variant=variant)
    assert again == p


def test_split_tail_balances_long_chunks(gqa):
    """On the long workloads splitting the last round beats whole items."""
    for q_len, kv_len in ((4096, 16384), (4096, 32768)):
        for v in (1, 2):
            _, whole = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, 152, force_splits=1,
                                                 force_variant=v)
            _, auto = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, 152, force_variant=v)
            assert auto["tail_splits"] > 1 and auto["head_rounds"] >= 1
            assert auto["est_makespan_tiles"] < 0.95 * whole["est_makespan_tiles"]


def test_force_grid_caps_the_grid(gqa):
    _, p = gqa.gqa_prefill_make_plan(129, 1000, 24, 4, 256, 152, force_splits=3, force_grid=5,
                                     force_variant=1)
    assert p["grid"] == 5 and p["head_rounds"] == 5 and p["tail_items"] == 3
    _, p = gqa.gqa_prefill_make_plan(129, 1000, 24, 4, 256, 152, force_splits=1, force_grid=5,
                                     force_variant=1)
    assert p["grid"] == 5 and p["kernels_per_call"] == 1
    _, p = gqa.gqa_prefill_make_plan(129, 1000, 24, 4, 256, 152, force_splits=2, force_grid=6,
                                     force_variant=2)
    assert p["grid"] == 6 and p["variant"] == 2 and p["q_tiles"] == 4  # 3 pairs, 42-token items


def test_make_plan_validates(gqa):
    S = gqa.GqaStatus
    assert gqa.gqa_prefill_make_plan(5, 4, 24, 4, 256, 148, check=False)[0] == S.ERR_SHAPE
    assert gqa.gqa_prefill_make_plan(5, 8, 24, 4, 256, 0, check=False)[0] == S.ERR_SHAPE
    assert gqa.gqa_prefill_make_plan(5, 8, 24, 2, 256, 148, check=False)[0] == S.ERR_UNSUPPORTED


def test_fp8_refusals_before_any_cuda_call(gqa):
    S = gqa.GqaStatus
    qz = lambda *a: gqa.gqa_quantize_q_fp8(*a, stream=0, check=False)
    kz = lambda *a: gqa.gqa_quantize_k_fp8(*a, stream=0, check=False)
    assert qz(16, 16, 16, -1, 24, 256) == S.ERR_SHAPE
    assert qz(16, 16, 16, 4, 32, 256) == S.ERR_UNSUPPORTED
    assert qz(None, 16, 16, 4, 24, 256) == S.ERR_NULL
    assert qz(16, 24, 16, 4, 24, 256) == S.ERR_ALIGN
    assert qz(16, 16, 18, 4, 24, 256) == S.ERR_ALIGN   # q_scale: 4-byte alignment
    assert qz(None, None, None, 0, 24, 256) == S.OK     # nothing to do
    assert kz(16, 16, 16, 8, 4, 256, 6) == S.ERR_SHAPE  # stride not a multiple of 4
    assert kz(16, 16, 16, 8, 4, 256, 4) == S.ERR_SHAPE  # stride < kv_len
    assert kz(16, 16, 20, 8, 4, 256, 8) == S.ERR_ALIGN  # k_scale: 16-byte alignment
    assert kz(16, 16, 16, 8, 2, 256, 8) == S.ERR_UNSUPPORTED
    f = lambda *a: gqa.gqa_prefill_attn_fp8qk(*a, stream=0, check=False)
    ok = dict(q=16, qs=16, k=16, ks=16, st=8, v=16, out=16, lse=None, q_len=4, kv_len=8, hq=24,
              hkv=4, d=256, scale=0.0625)
    names = list(ok)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(*[a[n] for n in names])

    assert call(st=4) == S.ERR_SHAPE
    assert call(st=10) == S.ERR_SHAPE
    assert call(qs=None) == S.ERR_NULL
    assert call(ks=None) == S.ERR_NULL
    assert call(ks=20) == S.ERR_ALIGN
    assert call(qs=18) == S.ERR_ALIGN
    assert call(v=None) == S.ERR_NULL
    assert call(hq=16) == S.ERR_UNSUPPORTED
    assert call(q_len=9) == S.ERR_SHAPE
    assert call(q=None, qs=None, k=None, ks=None, v=None, out=None, q_len=0, kv_len=0, st=0) == S.OK


def test_varlen_refusals_before_any_cuda_call(gqa):
    S = gqa.GqaStatus
    f = lambda cq, ck, **kw: gqa.gqa_prefill_attn_varlen(
        kw.get("q", 16), 16, 16, kw.get("out", 16), None, cq, ck, 24, kw.get("hkv", 4), 256,
        0.0625, stream=0, check=False)
    assert f([1, 4], [0, 8]) == S.ERR_SHAPE          # must start at 0
    assert f([0, 4, 3], [0, 8, 16]) == S.ERR_SHAPE   # decreasing
    assert f([0, 9], [0, 8]) == S.ERR_SHAPE          # q_len > kv_len
    assert f([0, 4], [0, 8], hkv=2) == S.ERR_UNSUPPORTED
    assert f([0, 4], [0, 8], q=None) == S.ERR_NULL
    assert f([0, 4], [0, 8], out=24) == S.ERR_ALIGN
    assert f([0] * 130, [0] * 130) == S.ERR_UNSUPPORTED   # 129 sequences > GQA_MAX_SEQS
    assert f([0, 0, 0], [0, 5, 9], q=None, out=None) == S.OK  # no query rows: nothing to do
    pf = lambda bt_stride, kv_lens: gqa.gqa_prefill_attn_paged_varlen(
        16, 16, 16, 16, bt_stride, 10, 16, 16, None, [0, 2, 4], kv_lens, 24, 4, 256, 0.0625,
        stream=0, check=False)
    assert pf(2, [40, 20]) == S.ERR_SHAPE             # 40 keys need 3 pages per table row
    assert pf(3, [40, 1]) == S.ERR_SHAPE              # second sequence: q_len 2 > kv_len 1


def test_paged_plans_prefer_the_pair(gqa):
    """Paged calls weigh the one-CTA plan up: 512x32768 is planned one CTA per item
    on dense K/V and as CTA pairs on paged K/V; where the pair wins on dense K/V
    too (4096x32768) both plans are the same; with no pair resident both use one
    CTA; a forced variant is honoured by both."""
    def both(ql, kl, **kw):
        _, d = gqa.gqa_prefill_make_plan_varlen([0, ql], [0, kl], 24, 4, 256, 152, 76, **kw)
        _, p = gqa.gqa_prefill_make_plan_paged_varlen([0, ql], [kl], 24, 4, 256, 152, 76, **kw)
        return d, p
    d, p = both(512, 32768)
    assert d["variant"] == 1 and p["variant"] == 2
    d, p = both(4096, 32768)
    assert d == p and p["variant"] == 2
    for v in (1, 2):
        d, p = both(512, 32768, force_variant=v)
        assert d == p and p["variant"] == v
    _, p0 = gqa.gqa_prefill_make_plan_paged_varlen([0, 512], [32768], 24, 4, 256, 152, 0)
    assert p0["variant"] == 1
    # a batch: the same lengths as cu_seqlens_k or as kv_lens give the same dense plan
    lens = [(43, 300), (1, 4096), (129, 1000)]
    cu_q, cu_k, kv = [0], [0], []
    for ql, kl in lens:
        cu_q.append(cu_q[-1] + ql)
        cu_k.append(cu_k[-1] + kl)
        kv.append(kl)
    _, d = gqa.gqa_prefill_make_plan_varlen(cu_q, cu_k, 24, 4, 256, 152, 76, force_variant=1)
    _, p = gqa.gqa_prefill_make_plan_paged_varlen(cu_q, kv, 24, 4, 256, 152, 76, force_variant=1)
    assert d == p
    assert gqa.gqa_prefill_make_plan_paged_varlen([0, 5], [4], 24, 4, 256, 152, check=False)[0] \
        == gqa.GqaStatus.ERR_SHAPE  # q_len > kv_len


@pytest.mark.parametrize("lens", [[(4096, 32768)], [(43, 300), (1, 4096), (0, 50), (129, 1000)],
                                  [(1, 1000)] * 40, [(512, 4096), (300, 20000), (2000, 2000)],
                                  [(21, 21)] * 128])
@pytest.mark.parametrize("variant", [0, 1, 2])
def test_varlen_plan_invariants(gqa, lens, variant):
    cu_q, cu_k = [0], [0]
    for ql, kl in lens:
        cu_q.append(cu_q[-1] + ql)
        cu_k.append(cu_k[-1] + kl)
    rc, p = gqa.gqa_prefill_make_plan_varlen(cu_q, cu_k, 24, 4, 256, 152, force_variant=variant)
    assert rc == 0
    tpi = 42 if p["variant"] == 2 else 21
    n_items = sum(4 * -(-ql // tpi) for ql, _ in lens)
    tiles = 0
    for ql, kl in lens:
        for qt in range(-(-ql // tpi)):
            tok_end = min((qt + 1) * tpi, ql)
            tiles += 4 * ((kl - ql + tok_end + 127) // 128)
    assert p["n_items"] == n_items and p["total_tiles"] == tiles
    assert p["grid"] <= 152
    if p["tail_splits"] > 0:
        assert p["n_units"] == (p["n_items"] - p["tail_items"]) + p["tail_items"] * p["tail_splits"]
    else:  # balanced tail: every item at least once, at most two extra pieces per worker
        workers = p["grid"] // (2 if p["variant"] == 2 else 1)
        assert p["n_items"] <= p["n_units"] <= p["n_items"] + 2 * workers
    if len(lens) == 1:
        _, single = gqa.gqa_prefill_make_plan(lens[0][0], lens[0][1], 24, 4, 256, 152,
                                              force_variant=variant)
        assert single == p


def test_batched_key_quantisation_refusals(gqa):
    S = gqa.GqaStatus
    f = lambda cu_k, stride, **kw: gqa.gqa_quantize_k_fp8_varlen(
        kw.get("k", 16), 16, kw.get("ks", 16), cu_k, kw.get("hkv", 4), 256, stride, stream=0,
        check=False)
    assert gqa.key_scale_columns([0, 5, 12]) == ([0, 8], 16)
    assert f([0, 5, 12], 12) == S.ERR_SHAPE   # the two sequences need 8 + 8 columns
    assert f([0, 5, 12], 18) == S.ERR_SHAPE   # stride not a multiple of 4
    assert f([1, 5], 8) == S.ERR_SHAPE
    assert f([0, 5, 4], 16) == S.ERR_SHAPE    # decreasing
    assert f([0, 5], 8, hkv=2) == S.ERR_UNSUPPORTED
    assert f([0, 5], 8, ks=20) == S.ERR_ALIGN
    assert f([0, 5], 8, k=None) == S.ERR_NULL
    assert f([0, 0, 0], 0, k=None, ks=None) == S.OK


@pytest.mark.parametrize("q_len,kv_len,splits", [(1, 32768, 32), (4, 32768, 32), (2, 16384, 32),
                                                 (1, 131072, 32), (1, 4096, 16)])
def test_decode_plans_keep_the_measured_split_counts(gqa, q_len, kv_len, splits):
    """Decode-sized chunks: one CTA per 21-token item, each item's KV range cut into the
    split count that measured fastest on GB300 in sweeps of forced counts (16 to 38 and the
    balanced tail), one CTA per piece."""
    _, p = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, 152)
    assert p["variant"] == 1 and p["head_rounds"] == 0 and p["tail_items"] == 4
    assert p["tail_splits"] == splits and p["grid"] == 4 * splits and p["kernels_per_call"] == 2


@pytest.mark.parametrize("q_len,kv_len,plan", [
    (128, 256, (2, 0, 16, 1, 32)), (512, 4096, (2, 0, 52, 1, 104)),
    (4096, 8192, (2, 5, 12, 5, 152)), (4096, 16384, (2, 5, 12, 3, 152)),
    (3072, 16384, (2, 0, 296, 1, 152)), (512, 32768, (1, 0, 100, 3, 152)),
    (4096, 32768, (2, 5, 12, 5, 152))])
def test_workload_plans_are_the_measured_ones(gqa, q_len, kv_len, plan):
    """The seven workloads' plans (variant, whole rounds, tail items, splits, grid) on 152
    SMs: the ones the measured figures were taken with."""
    _, p = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, 152)
    assert (p["variant"], p["head_rounds"], p["tail_items"], p["tail_splits"], p["grid"]) == plan


def test_make_plan_respects_the_resident_pair_count(gqa):
    """max_pairs caps the CTA-pair grid; 0 plans without the pair kernel; a negative
    value assumes num_sms / 2 (the same plan as passing num_sms / 2)."""
    for q_len, kv_len in ((4096, 32768), (512, 4096), (3072, 16384), (1, 32768)):
        _, p_none = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, 152, max_pairs=0)
        assert p_none["variant"] == 1
        _, p_few = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, 152, max_pairs=10,
                                             force_variant=2)
        assert p_few["variant"] == 2 and p_few["grid"] <= 20
        _, p_def = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, 152)
        _, p_half = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, 152, max_pairs=76)
        _, p_big = gqa.gqa_prefill_make_plan(q_len, kv_len, 24, 4, 256, 152, max_pairs=1000)
        assert p_def == p_half == p_big
