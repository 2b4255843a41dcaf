"""The attention kernel's barrier protocol, checked on a model of its roles.

gqa_attn_fwd_sm103_kernel runs these roles per CTA (pair): the TMA producer
(two on paged K/V: Q/K and V), the softmax warps, the QK^T-issuing thread and
the PV-issuing thread, which hand work to one another through mbarriers. This
test restates, per work unit of nt KV tiles, the order in which each role waits
and arrives, and checks:

* no deadlock: a greedy run of all roles completes, with and without the
  data-dependent waits (the softmax's O rescale waits for the previous PV);
* phase safety: an mbarrier wait names a phase by its parity only, so a wait on
  the stage barrier of ring position p (stage p mod n) is correct only if the
  fill of position p - n has completed before the wait starts. TMA fills
  complete asynchronously and in any order, so this must follow from
  happens-before (program order plus arrive -> wait), not from timing.

The kernel splits its five K/V stages into a K ring read by the QK^T thread and
a V ring read by the PV thread. One producer fills both in the order K0, K1,
V0, K2, V1, ...; on paged K/V each ring has its own producer, filling it in
tile order. A negative control runs the same check on one shared ring filled by
one producer and read by both MMA threads (an earlier design): it must be
flagged.
"""
import collections
import itertools
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KERNEL = os.path.join(ROOT, "gqa_chunked_prefill_gb300", "csrc", "attn_fwd_sm103.cu")
STAGES = 5


def k_ring_stages(k_per_tile):
    """Stages of the K ring (the kernel's kStagesK); the V ring has the rest."""
    return 3 if k_per_tile == 2 else 2


def test_ring_split_matches_the_kernel():
    src = open(KERNEL).read()
    assert "constexpr int kStages = 5;" in src
    assert "kStagesK = kKStagesPerTile == 2 ? 3 : 2;" in src
    # one producer thread for both rings (dense), one per ring (paged)
    assert "if constexpr (!split) produce(BoolC<true>{}, BoolC<true>{});" in src
    assert "else if (warp == kTmaWarp) produce(BoolC<true>{}, BoolC<false>{});" in src
    assert "else produce(BoolC<false>{}, BoolC<true>{});" in src
    hdr = open(os.path.join(os.path.dirname(KERNEL), "gqa_internal.h")).read()
    assert "constexpr bool fwd_split_producer(int kv) { return kv == 1; }" in hdr


def roles_for(units, kk, kv, shared_ring=False, rescale=True, split_producer=False):
    """Event lists (("wait"|"arrive"|"fill", barrier-phase)) of the roles. units: tiles
    per work unit; kk / kv: stages per K / V tile (pair 1 / 1, one-CTA BF16 2 / 2,
    one-CTA FP8 QK^T 1 / 2). Ring barriers are named by (ring, position). One
    producer fills the rings in the order K0, K1, V0, K2, V1, ... (with shared_ring,
    one ring); with split_producer a second one fills the V ring."""
    assert not (shared_ring and split_producer)
    n_k = STAGES if shared_ring else k_ring_stages(kk)
    n_v = STAGES if shared_ring else STAGES - n_k
    prod, prod_v, sm, qk, pv = [], [], [], [], []
    pos = {"K": 0, "V": 0}
    ring = {"K": "K", "V": "K" if shared_ring else "V"}  # one ring: V positions in K's
    n_of = {"K": n_k, "V": n_v}
    t0 = 0
    for u, nt in enumerate(units):
        if u:
            prod.append(("wait", ("QEmpty", u - 1)))
        prod.append(("arrive", ("QFull", u)))
        if not split_producer:  # one producer: K0, K1, V0, K2, V1, ..., V_{nt-1}
            order = []
            for j in range(nt):
                order += [("K", t0 + j, h) for h in range(kk)]
                if j:
                    order += [("V", t0 + j - 1, h) for h in range(kv)]
            order += [("V", t0 + nt - 1, h) for h in range(kv)]
        else:  # each producer fills its ring in tile order
            order = [("K", t0 + j, h) for j in range(nt) for h in range(kk)]
            order += [("V", t0 + j, h) for j in range(nt) for h in range(kv)]
        where = {}
        for kind, t, h in order:
            r = ring[kind]
            p = pos[r]
            out = prod_v if (kind == "V" and split_producer) else prod
            if p >= n_of[kind]:
                out.append(("wait", (r + "Empty", p - n_of[kind])))
            out.append(("fill", (r + "Full", p)))
            where[(kind, t, h)] = (r, p)
            pos[r] += 1
        for j in range(nt):
            t = t0 + j
            sm += [("wait", ("SFull", t)), ("arrive", ("SFree", t))]
            if j and rescale:
                sm.append(("wait", ("PvDone", t - 1)))  # O rescale before P_t
            if t >= 2:
                sm.append(("wait", ("PvDone", t - 2)))  # P buffer t % 2 free
            sm.append(("arrive", ("PFull", t)))
        sm += [("wait", ("PvDone", t0 + nt - 1)), ("arrive", ("OFree", u))]
        qk.append(("wait", ("QFull", u)))
        for j in range(nt):
            t = t0 + j
            r, p = where[("K", t, 0)]
            qk.append(("wait", (r + "Full", p)))
            if t:
                qk.append(("wait", ("SFree", t - 1)))
            for h in range(kk):
                r, p = where[("K", t, h)]
                if h:
                    qk.append(("wait", (r + "Full", p)))
                qk.append(("arrive", (r + "Empty", p)))
            qk.append(("arrive", ("SFull", t)))
            if j == nt - 1:
                qk.append(("arrive", ("QEmpty", u)))
        for j in range(nt):
            t = t0 + j
            r, p = where[("V", t, 0)]
            pv += [("wait", (r + "Full", p)), ("wait", ("PFull", t))]
            if j == 0 and u:
                pv.append(("wait", ("OFree", u - 1)))
            for h in range(kv):
                r, p = where[("V", t, h)]
                if h:
                    pv.append(("wait", (r + "Full", p)))
                pv.append(("arrive", (r + "Empty", p)))
            pv.append(("arrive", ("PvDone", t)))
        t0 += nt
    roles = {"prod": prod, "softmax": sm, "qk": qk, "pv": pv}
    if split_producer:
        roles["prod_v"] = prod_v
    return roles, n_of


def completes(roles):
    done, idx = set(), dict.fromkeys(roles, 0)
    moved = True
    while moved:
        moved = False
        for r, evs in roles.items():
            while idx[r] < len(evs):
                kind, b = evs[idx[r]]
                if kind == "wait" and b not in done:
                    break
                if kind in ("arrive", "fill"):
                    done.add(b)
                idx[r] += 1
                moved = True
    return all(idx[r] == len(roles[r]) for r in roles)


def unsafe_ring_waits(roles, n_of):
    """Ring waits whose previous phase (position p - n) is not ordered before the wait."""
    succ = collections.defaultdict(list)
    source = {}
    for r, evs in roles.items():
        chain = []
        for i, (kind, b) in enumerate(evs):
            node = (r, i)
            chain.append(node)
            if kind == "fill":  # the copy completes some time after it is issued
                source[b] = (r, i, "done")
                succ[node].append(source[b])
            elif kind == "arrive":
                source[b] = node
        for a, b in zip(chain, chain[1:]):
            succ[a].append(b)
    for r, evs in roles.items():
        for i, (kind, b) in enumerate(evs):
            if kind == "wait":
                succ[source[b]].append((r, i))

    def reaches(a, b):
        seen, todo = {a}, [a]
        while todo:
            x = todo.pop()
            if x == b:
                return True
            for y in succ[x]:
                if y not in seen:
                    seen.add(y)
                    todo.append(y)
        return False

    bad = []
    for r, evs in roles.items():
        for i, (kind, b) in enumerate(evs):
            if kind == "wait" and b[0] in ("KFull", "VFull"):
                n = n_of["K"] if b[0] == "KFull" else n_of["V"]
                prev = (b[0], b[1] - n)
                if prev[1] >= 0 and (i == 0 or not reaches(source[prev], (r, i - 1))):
                    bad.append((r, b))
    return bad


LAYOUTS = [(1, 1), (2, 2), (1, 2)]  # stages per K / V tile: pair, one-CTA BF16, one-CTA FP8
UNITS = [u for n in (1, 2, 3) for u in itertools.product([1, 2, 3, 5], repeat=n)]


@pytest.mark.parametrize("split_producer", [False, True])
@pytest.mark.parametrize("kk,kv", LAYOUTS)
def test_no_deadlock(kk, kv, split_producer):
    for units in UNITS:
        for rescale in (True, False):
            roles, _ = roles_for(list(units), kk, kv, rescale=rescale, split_producer=split_producer)
            assert completes(roles), (units, kk, kv, rescale)


@pytest.mark.parametrize("split_producer", [False, True])
@pytest.mark.parametrize("kk,kv", LAYOUTS)
def test_every_ring_wait_is_phase_safe(kk, kv, split_producer):
    # Without the rescale waits there are fewest happens-before edges: the worst case.
    for units in UNITS[:20]:
        roles, n_of = roles_for(list(units), kk, kv, rescale=False, split_producer=split_producer)
        assert unsafe_ring_waits(roles, n_of) == [], (units, kk, kv)


def test_one_ring_read_by_both_threads_is_flagged():
    flagged = 0
    for units in itertools.product([1, 2, 3], repeat=2):
        roles, n_of = roles_for(list(units), 1, 1, shared_ring=True, rescale=False)
        assert completes(roles)
        flagged += bool(unsafe_ring_waits(roles, n_of))
    assert flagged > 0
