"""Policy of the HBM expert cache over the host tier (moe_cache_*), run without a
device (MOE_CACHE_POLICY_ONLY + moe_cache_plan).

The pages keep the hottest routed experts in an LFU cache (NeutronStar glm-local
README, "SSD streaming optimizations": the host expert cache with LFU eviction),
load a batch's union of experts once ("Long-prompt prefill": one union read
serves the chunk) and prefetch the next layer's picks (the cross-layer
router-lookahead prefetch).  The rule this library fixes (moe.h): one lookup per
distinct expert per ensure; a miss takes the lowest free slot, else evicts the
fewest-lookups expert, ties to the least recent use, then the lower
(layer, expert); the call's own experts are never evicted, nor (for a prefetch)
those of the latest ensure.  Pinned here by hand-worked traces, invariants, and
a separately written model of the rule on random traces."""
import random

import numpy as np
import pytest

from routed_expert_decode_gb300 import moe

FAKE = 1 << 20  # pointers are never dereferenced in policy-only mode


def _weights():
    w = moe.MoeWeights()
    for n in ("gate", "up", "down"):
        setattr(w, n, moe.MoeMat(FAKE, FAKE))
    return w


def make_cache(E=8, layers=1, slots=4):
    desc = moe.make_desc(E, 2, 256, 256, 0, 0, 1.0)
    return moe.ExpertCache(desc, [_weights() for _ in range(layers)], _weights(), slots, FAKE,
                           policy_only=True)


def test_fill_then_hit():
    c = make_cache()
    assert c.plan(0, [5, 2]) == [(2, 0, -1), (5, 1, -1)]  # ascending experts, lowest free slots
    assert c.plan(0, [2, 5]) == []
    st = c.stats()
    assert (st["lookups"], st["hits"], st["misses"]) == (4, 2, 2)
    assert c.slot(0, 5) == 1 and c.slot(0, 3) == -1


def test_union_load_counts_duplicates_once():
    c = make_cache()
    assert c.plan(0, [3, 3, 1, 3, 1]) == [(1, 0, -1), (3, 1, -1)]
    assert c.stats()["lookups"] == 2


def test_lfu_victim_with_lru_and_id_ties():
    """Hand-worked: slots 4.  Lookups 0:x3, 1:x1, 2:x2, 3:x1 (3 used after 1).
    Loading 4 evicts the fewest-lookups expert, tie 1 vs 3 -> the older use (1)."""
    c = make_cache(slots=4)
    for req in ([0, 1], [0, 2], [0, 2], [3]):
        c.plan(0, req)
    assert c.plan(0, [4]) == [(4, c.slot(0, 4), 1)]
    assert c.slot(0, 1) == -1
    # next miss: the candidates are 3 (1 lookup) and 4 (1 lookup, newer) -> 3
    assert c.plan(0, [5])[0][2] == 3
    # equal counts and equal stamps cannot both occur (stamps are unique); the id
    # tie-break is still part of the rule, exercised by the model test below


def test_counts_survive_eviction():
    """An evicted expert keeps its lookup count: when it returns it outranks a
    once-used newcomer."""
    c = make_cache(slots=2)
    for _ in range(3):
        c.plan(0, [0])  # 0: 3 lookups
    c.plan(0, [1])      # 1: 1
    c.plan(0, [2])      # evicts 1 (fewer lookups than 0)
    assert c.slot(0, 1) == -1
    c.plan(0, [1, 2])   # 1 returns: evicts 0? no: 0 has 3 lookups; 1 and 2 are the call's own
    assert c.slot(0, 0) == -1  # the only evictable expert was 0
    c.plan(0, [3])      # now 0 is gone; victims among 1 (2 lookups) and 2 (2 lookups): older -> 1
    assert c.slot(0, 1) == -1 and c.slot(0, 2) >= 0


def test_union_larger_than_capacity_fails_unchanged():
    c = make_cache(slots=2)
    c.plan(0, [0])
    before = c.stats()
    with pytest.raises(moe.MoeError) as ei:
        c.plan(0, [1, 2, 3])
    assert moe.STATUS_NAMES[ei.value.status] == "MOE_ERR_WORKSPACE"
    assert c.stats() == before and c.slot(0, 0) >= 0


def test_prefetch_protects_latest_ensure_and_is_not_a_lookup():
    c = make_cache(E=8, layers=2, slots=3)
    c.plan(0, [0, 1])                       # latest ensure: layer 0, experts 0, 1
    got = c.plan(1, [4, 5], prefetch=True)  # one free slot, then nothing evictable
    assert got == [(4, 2, -1)]
    st = c.stats()
    assert st["lookups"] == 2 and st["prefetch_loads"] == 1
    c.plan(1, [4])                          # the prefetched expert is used: a hit
    st = c.stats()
    assert st["hits"] == 1 and st["prefetch_hits"] == 1
    # the latest ensure is now (1, 4): a prefetch may evict layer 0's experts
    got = c.plan(0, [6], prefetch=True)
    assert got and got[0][2] in (0, 1)


def test_layers_are_separate_keys():
    c = make_cache(E=4, layers=2, slots=4)
    assert c.plan(0, [1]) == [(1, 0, -1)]
    assert c.plan(1, [1]) == [(1, 1, -1)]
    assert c.slot(0, 1) == 0 and c.slot(1, 1) == 1


def test_bad_arguments():
    c = make_cache(E=8, layers=1)
    with pytest.raises(moe.MoeError):
        c.plan(0, [8])
    with pytest.raises(moe.MoeError):
        c.plan(1, [0])
    with pytest.raises(moe.MoeError):
        c.ensure(0, [0], stream=0)  # policy-only: no device work


class _Model:
    """The rule as stated, written out separately: a dict of resident experts."""

    def __init__(self, E, L, S):
        self.E, self.S = E, S
        self.slot = {}
        self.count = {}
        self.last = {}
        self.stamp = 0
        self.busy = set()

    def step(self, layer, experts, prefetch):
        u = sorted(set(experts))
        keys = [layer * self.E + e for e in u]
        protect = set(keys) | (self.busy if prefetch else set())
        if not prefetch:
            missing = sum(1 for g in keys if g not in self.slot)
            free = self.S - len(self.slot)
            movable = free + sum(1 for g in self.slot if g not in protect)
            if missing > movable:
                return "fail"
        out = []
        for e, g in zip(u, keys):
            if not prefetch:
                self.count[g] = self.count.get(g, 0) + 1
                self.stamp += 1
                self.last[g] = self.stamp
            if g in self.slot:
                continue
            used = set(self.slot.values())
            free = [s for s in range(self.S) if s not in used]
            victim = -1
            if free:
                s = free[0]
            else:
                cands = [h for h in self.slot if h not in protect]
                if not cands:
                    break
                victim = min(cands, key=lambda h: (self.count.get(h, 0), self.last.get(h, 0), h))
                s = self.slot.pop(victim)
            self.slot[g] = s
            out.append((e, s, victim))
        if not prefetch:
            self.busy = set(keys)
        return out


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_traces_match_model(seed):
    rng = random.Random(seed)
    E, L, S = 12, 3, 7
    c = make_cache(E=E, layers=L, slots=S)
    m = _Model(E, L, S)
    # Zipf-like popularity, as in the synthetic router (a few experts dominate)
    weights = [1.0 / (i + 1) ** 1.1 for i in range(E)]
    for _ in range(400):
        layer = rng.randrange(L)
        prefetch = rng.random() < 0.3
        req = rng.choices(range(E), weights=weights, k=rng.randint(1, 6))
        want = m.step(layer, req, prefetch)
        if want == "fail":
            with pytest.raises(moe.MoeError):
                c.plan(layer, req, prefetch)
            continue
        assert c.plan(layer, req, prefetch) == want
        # invariants: after an ensure its union is resident; slots are distinct
        if not prefetch:
            assert all(c.slot(layer, e) >= 0 for e in req)
        resident = [c.slot(l, e) for l in range(L) for e in range(E) if c.slot(l, e) >= 0]
        assert len(resident) == len(set(resident)) <= S
