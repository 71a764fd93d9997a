"""Fixed-capacity expert cache keyed by (layer, expert), LRU replacement.

From the pages: a VRAM hot cache of a fixed number of slots (8,445 on one
RTX 4090, P1 §先看结果) holds (layer, expert) identities; hits compute in
place, misses are fetched over PCIe from pinned host RAM that holds every
expert (P1 §如何做到：三层存储; P2 §2.1); the engine reports
"hits / lookups" per token pick (P2 §7.2).  The pages do not state the
replacement policy; the workload definition fixes LRU by (layer, expert)
with ties broken by the lower slot id.

One layer-call, at logical clock t (strictly increasing):
  1. U = the distinct (layer, expert) keys over the call's T*k picks.
  2. Every resident key of U is stamped t (hits first, so a call never
     evicts its own experts).
  3. The misses, in ascending key, each take the slot with the smallest
     (stamp, slot id); empty slots have stamp -1.  The victim's old key is
     dropped, the new key installed, and the slot stamped t.
A token pick counts as a hit iff its key was resident when the layer-call
began.  Shared experts live outside the cache and are not counted.

Pins: an independent ordered-list LRU twin on random small caches; cyclic
access of C+1 keys hits never; a cache that holds every key misses only
once per key; invariants (<= C resident, no duplicate keys,
hits + misses = k per token).
"""

from dataclasses import dataclass

import numpy as np


@dataclass
class LayerCallResult:
    keys: np.ndarray          # U, ascending
    slots: np.ndarray         # slot of each key of U after the call
    hit: np.ndarray           # bool per key of U: resident at the start
    miss_keys: np.ndarray     # ascending
    miss_slots: np.ndarray    # victim slot of each miss
    evicted: np.ndarray       # key previously held by each victim (-1: empty)
    token_hits: int
    token_misses: int


class ExpertCache:
    def __init__(self, capacity, n_keys):
        self.C = int(capacity)
        self.n_keys = int(n_keys)
        self.table = np.full(self.n_keys, -1, dtype=np.int64)   # key -> slot
        self.owner = np.full(self.C, -1, dtype=np.int64)        # slot -> key
        self.stamp = np.full(self.C, -1, dtype=np.int64)

    def preload(self, keys):
        """Install ``keys`` (ascending) into slots 0, 1, ... with stamp -1."""
        keys = np.asarray(keys, dtype=np.int64)
        assert keys.size <= self.C and np.all(np.diff(keys) > 0)
        for s, key in enumerate(keys):
            self.table[key] = s
            self.owner[s] = key
            self.stamp[s] = -1

    def step(self, pick_keys, t):
        """Apply one layer-call whose token picks are ``pick_keys`` [T, k]."""
        pick_keys = np.asarray(pick_keys, dtype=np.int64)
        U = np.unique(pick_keys)
        assert U.size <= self.C, "a call touches more experts than the cache holds"
        resident = self.table[U] >= 0
        for key in U[resident]:
            self.stamp[self.table[key]] = t
        misses = U[~resident]
        m = misses.size
        victims = np.empty(m, dtype=np.int64)
        evicted = np.empty(m, dtype=np.int64)
        if m:
            # the m smallest (stamp, slot) over all slots, ordered; this call's
            # hits now carry stamp t, larger than every other stamp.  The pair
            # is encoded as one integer (stamp + 1) * C + slot, whose integer
            # order is the lexicographic order of (stamp, slot).
            code = (self.stamp + 1) * self.C + np.arange(self.C)
            if m < self.C:
                part = np.argpartition(code, m - 1)[:m]
            else:
                part = np.arange(self.C)
            victims[:] = part[np.argsort(code[part])]
            assert np.all(self.stamp[victims] < t)
            for j in range(m):
                v = victims[j]
                old = self.owner[v]
                evicted[j] = old
                if old >= 0:
                    self.table[old] = -1
                self.owner[v] = misses[j]
                self.table[misses[j]] = v
                self.stamp[v] = t
        token_hits = int(np.count_nonzero(np.isin(pick_keys, U[resident])))
        return LayerCallResult(
            keys=U, slots=self.table[U].copy(), hit=resident,
            miss_keys=misses, miss_slots=victims, evicted=evicted,
            token_hits=token_hits, token_misses=int(pick_keys.size - token_hits))

    def check_invariants(self):
        res = self.owner[self.owner >= 0]
        assert np.unique(res).size == res.size, "duplicate key in two slots"
        for s in range(self.C):
            key = self.owner[s]
            if key >= 0:
                assert self.table[key] == s
        assert np.count_nonzero(self.table >= 0) == res.size <= self.C
