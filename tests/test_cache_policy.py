"""The expert cache's replacement policy (include/moe_v41_cache.h) in
simulation mode, on the CPU: no CUDA call is made.

The model below restates the policy from its definition: the experts a fetch
needs become the most recently used (resident ones first, then the misses,
each in ascending id); a miss takes a free slot (lowest first) or else the
least recently used slot the fetch does not need.  Demand and prefetch
fetches are counted apart; a demanded expert that a prefetch brought in and
nothing demanded since is a prefetch hit."""
from collections import OrderedDict

import numpy as np
import pytest

import quantized_mixture_experts_router_gb300 as Q

SLOT = 4096


class ModelLRU:
    def __init__(self, n_slots, slot_bytes=SLOT):
        self.slot_bytes = slot_bytes
        self.od = OrderedDict()          # key -> slot, least recent first
        self.free = list(range(n_slots))
        self.pre = {}                     # slot -> brought in by a prefetch, not demanded since
        self.st = dict(hits=0, misses=0, evictions=0, bytes_copied=0, prefetched=0, prefetch_hits=0)

    def fetch(self, layer, experts, prefetch=False):
        ids = sorted(set(int(e) for e in experts))
        keys = [(layer, e) for e in ids]
        for k in keys:
            if k in self.od:
                self.od.move_to_end(k)
                if not prefetch:
                    self.st["hits"] += 1
                    if self.pre.get(self.od[k]):
                        self.st["prefetch_hits"] += 1
                        self.pre[self.od[k]] = False
        need = set(keys)
        for k in keys:
            if k in self.od:
                continue
            if self.free:
                s = self.free.pop(0)
            else:
                victim = next(v for v in self.od if v not in need)
                s = self.od.pop(victim)
                self.st["evictions"] += 1
            self.od[k] = s
            self.pre[s] = bool(prefetch)
            self.st["prefetched" if prefetch else "misses"] += 1
            self.st["bytes_copied"] += self.slot_bytes

    def slot_of(self, layer, e):
        return self.od.get((layer, e), -1)


def _sim(n_layers, n_routed, n_slots):
    return Q.ExpertCache(n_layers, n_routed, n_slots, SLOT, 0, 1024, 2048)


def test_first_fetch_fills_slots_in_order_and_hits_after():
    c = _sim(2, 16, 8)
    c.fetch(0, [5, 3, 3, 9])
    assert [c.slot_of(0, e) for e in (3, 5, 9)] == [0, 1, 2]
    c.fetch(0, [9, 3])
    st = c.stats()
    assert st["misses"] == 3 and st["hits"] == 2 and st["evictions"] == 0 and st["bytes_copied"] == 3 * SLOT
    assert c.slot_of(1, 3) == -1 and c.slot_of(0, 4) == -1


def test_eviction_takes_the_least_recently_used_not_needed():
    c = _sim(1, 16, 3)
    c.fetch(0, [0, 1, 2])      # slots 0, 1, 2; recency 0 < 1 < 2
    c.fetch(0, [0])            # recency 1 < 2 < 0
    c.fetch(0, [1, 7])         # 1 is needed: the victim is 2, its slot goes to 7
    assert c.slot_of(0, 2) == -1 and c.slot_of(0, 7) == 2 and c.slot_of(0, 1) == 1
    assert c.stats()["evictions"] == 1


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_policy_matches_the_model_on_random_traces(seed):
    rng = np.random.default_rng(seed)
    n_layers, n_routed, n_slots = 5, 24, 11
    c = _sim(n_layers, n_routed, n_slots)
    ref = ModelLRU(n_slots)
    for step in range(600):
        layer = int(rng.integers(n_layers))
        k = int(rng.integers(1, 7))
        # a skewed draw, so that hits and misses both happen
        experts = rng.choice(n_routed, size=k, p=np.linspace(2, 1, n_routed) / np.linspace(2, 1, n_routed).sum())
        pre = bool(rng.random() < 0.3)
        c.fetch(layer, experts, prefetch=pre)
        ref.fetch(layer, experts, prefetch=pre)
        if step % 50 == 0:
            for l in range(n_layers):
                assert [c.slot_of(l, e) for e in range(n_routed)] == [ref.slot_of(l, e) for e in range(n_routed)]
    assert c.stats() == ref.st
    assert ref.st["prefetch_hits"] > 0 and ref.st["evictions"] > 0 and ref.st["hits"] > 0


def test_prefetch_then_demand_counts_a_prefetch_hit_once():
    c = _sim(2, 8, 4)
    c.fetch(1, [2, 6], prefetch=True)
    c.fetch(1, [2, 6])
    c.fetch(1, [2])
    st = c.stats()
    assert st["prefetched"] == 2 and st["misses"] == 0 and st["hits"] == 3 and st["prefetch_hits"] == 2


def test_argument_errors():
    with pytest.raises(Q.MoeError):
        Q.ExpertCache(1, 8, 4, 1000, 0, 256, 512)          # slot size not a multiple of 256
    with pytest.raises(Q.MoeError):
        Q.ExpertCache(1, 8, 4, SLOT, 0, 256, SLOT)         # an offset past the slot
    c = _sim(2, 8, 3)
    with pytest.raises(Q.MoeError):
        c.fetch(0, [0, 1, 2, 3])                           # more distinct experts than slots
    with pytest.raises(Q.MoeError):
        c.fetch(2, [0])                                    # layer out of range
    with pytest.raises(Q.MoeError):
        c.fetch(0, [8])                                    # expert out of range
    c.fetch(0, [1, 1, 1, 2, 2])                            # repeats count once
    assert c.stats()["misses"] == 2
