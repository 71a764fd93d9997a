"""Pins of the oracle LRU expert cache."""

import numpy as np
import pytest

from oracle.cache import ExpertCache


class ListLRU:
    """Independent twin: an explicit least- to most-recently-used slot list.

    Within one layer-call every touched slot becomes most recent; slots
    touched in the same call are ordered by slot id.  Victims are taken from
    the least-recent end, skipping the call's own hits.
    """

    def __init__(self, C):
        self.order = list(range(C))
        self.slot_key = [-1] * C
        self.key_slot = {}

    def preload(self, keys):
        for s, k in enumerate(keys):
            self.slot_key[s] = k
            self.key_slot[k] = s

    def step(self, picks):
        U = sorted(set(int(k) for k in np.asarray(picks).ravel()))
        hits = [k for k in U if k in self.key_slot]
        misses = [k for k in U if k not in self.key_slot]
        hit_slots = {self.key_slot[k] for k in hits}
        victims = [s for s in self.order if s not in hit_slots][:len(misses)]
        assert len(victims) == len(misses)
        for k, v in zip(misses, victims):
            old = self.slot_key[v]
            if old >= 0:
                del self.key_slot[old]
            self.slot_key[v] = k
            self.key_slot[k] = v
        touched = sorted(hit_slots | set(victims))
        tset = set(touched)
        self.order = [s for s in self.order if s not in tset] + touched
        th = sum(1 for k in np.asarray(picks).ravel() if int(k) in set(hits))
        return misses, victims, th


@pytest.mark.parametrize("seed", range(6))
def test_matches_list_twin_on_random_streams(seed):
    rng = np.random.default_rng(seed)
    C = int(rng.integers(4, 20))
    n_keys = int(rng.integers(C + 1, 3 * C + 5))
    T, k = int(rng.integers(1, 4)), int(rng.integers(1, 3))
    if T * k > C:
        T = 1
    zipf = 1.0 / np.arange(1, n_keys + 1) ** rng.uniform(0, 1.5)
    zipf /= zipf.sum()
    cache, twin = ExpertCache(C, n_keys), ListLRU(C)
    if seed % 2:
        pre = np.sort(rng.choice(n_keys, C // 2, replace=False))
        cache.preload(pre)
        twin.preload(pre.tolist())
    for t in range(300):
        picks = np.array([rng.choice(n_keys, k, replace=False, p=zipf) for _ in range(T)])
        r = cache.step(picks, t)
        misses, victims, th = twin.step(picks)
        assert r.miss_keys.tolist() == misses
        assert r.miss_slots.tolist() == victims
        assert r.token_hits == th
        assert r.token_hits + r.token_misses == T * k
        for key, slot in zip(r.keys, r.slots):
            assert twin.key_slot[int(key)] == slot
        cache.check_invariants()


def test_cyclic_scan_of_c_plus_one_keys_never_hits():
    C = 7
    cache = ExpertCache(C, 100)
    hits = 0
    for t in range(10 * (C + 1)):
        r = cache.step(np.array([[t % (C + 1)]]), t)
        hits += r.token_hits
    assert hits == 0


def test_cache_holding_every_key_misses_once_per_key():
    n_keys = 12
    cache = ExpertCache(n_keys, n_keys)
    rng = np.random.default_rng(0)
    misses = 0
    seen = set()
    for t in range(200):
        picks = rng.choice(n_keys, (3, 2))
        picks = np.array([rng.choice(n_keys, 2, replace=False) for _ in range(3)])
        r = cache.step(picks, t)
        misses += r.miss_keys.size
        seen |= set(picks.ravel().tolist())
        assert np.all(r.evicted == -1)
    assert misses == len(seen)


def test_empty_slots_fill_in_slot_order_then_lru_evicts_oldest():
    cache = ExpertCache(3, 10)
    assert cache.step(np.array([[5, 2]]), 0).miss_slots.tolist() == [0, 1]   # key 2 -> 0, key 5 -> 1
    assert cache.step(np.array([[7]]), 1).miss_slots.tolist() == [2]
    r = cache.step(np.array([[2, 9]]), 2)      # 2 hits; 9 evicts the LRU slot (slot 1, key 5)
    assert r.hit.tolist() == [True, False] and r.miss_slots.tolist() == [1]
    assert r.evicted.tolist() == [5]
    r = cache.step(np.array([[4, 8]]), 3)      # slots by (stamp, id): 2 (t=1), then 0 and 1 (t=2)
    assert r.miss_slots.tolist() == [2, 0] and sorted(r.evicted.tolist()) == [2, 7]


def test_call_never_evicts_its_own_hits():
    cache = ExpertCache(2, 10)
    cache.step(np.array([[1, 2]]), 0)
    with pytest.raises(AssertionError):
        cache.step(np.array([[1, 2, 3]]), 1)     # 3 distinct keys cannot fit 2 slots
    cache = ExpertCache(3, 10)
    cache.step(np.array([[1], [2], [3]]), 0)
    r = cache.step(np.array([[1, 4]]), 1)       # hit 1 (slot 0) is stamped before the miss picks
    assert r.miss_slots.tolist() == [1]
