"""The expert cache's policy on the host (no GPU): the library's decisions, call by call,
against a model written here from the pages' rules (README of FareedKhan-dev/kimi-k3-in-c,
section 12 "An LRU cache for the experts": a slot is empty, in flight or holds an expert;
the victim is the first empty slot, else the least recently used slot that is neither
pinned nor in flight; README of Maknee/Kimi-K3.cpp, "The consumer-memory idea", item 4:
every selected hit is pinned before any victim is chosen)."""
import ctypes

import numpy as np
import pytest

import mxfp4_routed_expert_02_gb300 as k3
from mxfp4_routed_expert_02_gb300 import k3moe as B


class PageLRU:
    """The pages' cache, restated: per slot a key (or EMPTY), a last-use time, a pin."""
    EMPTY, INFLIGHT = "empty", "inflight"

    def __init__(self, n_slots, n_experts):
        self.key = [self.EMPTY] * n_slots
        self.used = [0] * n_slots
        self.E = n_experts
        self.clock = 0
        self.hits = self.misses = 0

    def victim(self, pinned):
        best, oldest = None, None
        for s, k in enumerate(self.key):
            if k == self.INFLIGHT:
                continue
            if k == self.EMPTY:
                return s
            if s in pinned:
                continue
            if oldest is None or self.used[s] < oldest:
                best, oldest = s, self.used[s]
        return best

    def call(self, layer, experts):
        keys = [layer * self.E + e for e in experts]
        resident = {k: s for s, k in enumerate(self.key) if k not in (self.EMPTY, self.INFLIGHT)}
        distinct = set(keys)
        nhit = sum(1 for k in distinct if k in resident)
        if len(distinct) - nhit > len(self.key) - nhit:
            return None                                   # refused, nothing changed
        self.clock += 1
        slots, load, pinned = [None] * len(keys), [0] * len(keys), set()
        for j, k in enumerate(keys):                      # pin the hits first
            if k in resident:
                s = resident[k]
                if s not in pinned:
                    self.hits += 1
                pinned.add(s)
                self.used[s] = self.clock
                slots[j] = s
        reserved = {}
        for j, k in enumerate(keys):                      # then reserve the misses
            if slots[j] is not None:
                continue
            if k in reserved:
                slots[j] = reserved[k]
                continue
            s = self.victim(pinned)
            self.key[s] = self.INFLIGHT
            pinned.add(s)
            self.used[s] = self.clock
            reserved[k] = s
            slots[j], load[j] = s, 1
            self.misses += 1
        for k, s in reserved.items():                     # publish
            self.key[s] = k
        return slots, load


def make_cache(n_slots, n_experts, n_layers=2):
    # host-only use: the addresses are never dereferenced by the lookup
    fake = [0x1000 * (l + 1) for l in range(n_layers)]
    return k3.ExpertCache(fake, n_experts, 4096, 4096, 0x7f0000000000, n_slots, 4096)


def test_policy_matches_the_pages_rules_call_by_call():
    rng = np.random.default_rng(0)
    for n_slots, E, K in [(4, 12, 2), (6, 20, 3), (16, 64, 4), (5, 5, 5)]:
        cache, model = make_cache(n_slots, E), PageLRU(n_slots, E)
        for step in range(400):
            layer = int(rng.integers(0, 2))
            T = int(rng.integers(1, 3))
            ex = np.concatenate([rng.choice(E, size=K, replace=False) for _ in range(T)])
            want = model.call(layer, ex.tolist())
            if want is None:
                with pytest.raises(k3.K3MoeError) as ei:
                    cache.lookup(layer, ex)
                assert ei.value.code == B.K3MOE_ERR_CACHE_FULL
                continue
            slots, load = cache.lookup(layer, ex)
            assert slots.tolist() == want[0], (n_slots, E, step)
            assert load.tolist() == want[1]
        st = cache.stats()
        assert (st["hits"], st["misses"]) == (model.hits, model.misses)
        assert st["bytes_loaded"] == model.misses * 4096


def test_hits_are_pinned_before_victims_are_chosen():
    cache = make_cache(3, 10)
    cache.lookup(0, [1])          # slot 0, least recently used
    cache.lookup(0, [2])          # slot 1
    cache.lookup(0, [3])          # slot 2
    # expert 1 is the LRU entry and is selected again with a miss: the miss must not evict
    # it (it is pinned first) but the next least recently used, expert 2
    slots, load = cache.lookup(0, [4, 1])
    assert slots.tolist() == [1, 0] and load.tolist() == [1, 0]


def test_empty_slots_first_duplicates_share_and_full_calls_change_nothing():
    cache = make_cache(4, 10)
    slots, load = cache.lookup(0, [7, 7, 3])
    assert slots.tolist() == [0, 0, 1] and load.tolist() == [1, 0, 1]
    slots, load = cache.lookup(1, [7])      # another layer's expert 7 is another record
    assert slots.tolist() == [2] and load.tolist() == [1]
    before = cache.stats()
    with pytest.raises(k3.K3MoeError):
        cache.lookup(0, [0, 1, 2, 4, 5])    # 5 distinct experts, 4 slots
    assert cache.stats() == before
    slots, load = cache.lookup(0, [3, 7])   # still resident, untouched by the refusal
    assert load.tolist() == [0, 0]
    # out-of-range experts are neither loaded nor given a slot
    slots, load = cache.lookup(0, [-1, 10])
    assert slots.tolist() == [-1, -1] and load.tolist() == [0, 0]


def test_create_checks_its_arguments():
    L = k3.lib()
    out = ctypes.c_void_p()
    ptrs = (ctypes.c_void_p * 1)(ctypes.c_void_p(0x1000))
    # slot stride below the record, misaligned slots, no layers
    assert L.k3moe_cache_create(1, ptrs, 4, 4096, 4096, ctypes.c_void_p(0x10000), 2, 2048,
                                ctypes.byref(out)) == 3
    assert L.k3moe_cache_create(1, ptrs, 4, 4096, 4096, ctypes.c_void_p(0x10008), 2, 4096,
                                ctypes.byref(out)) == 3
    assert L.k3moe_cache_create(0, ptrs, 4, 4096, 4096, ctypes.c_void_p(0x10000), 2, 4096,
                                ctypes.byref(out)) == 1
