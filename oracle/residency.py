"""Plain reference of the expert-residency replacement policies, and Belady's
offline optimum for the hit-rate ceiling.

TEST INFRASTRUCTURE ONLY (the test suite and the benchmark's replay leg call it).
It shares nothing with the library: each policy is restated from the pages in
slow, direct Python (lists and dicts, a full scan per decision):

  LRU -- kairos-engine README, "Decode, 2026-09-28/29": a layer's experts are
      resolved before any is computed, and resolving stamps each of them most
      recently used, so the layer never evicts its own experts.
  decayed frequency -- kairos-engine README, "2026-09-29: which experts to keep":
      frequency with a 32-token half-life and a 2-token recency guard.
  LFU with swaps -- Strata article, "The cache's replacement rule": a float
      counter per (layer, expert) bumped by every routed id; every fourth round,
      per layer, the hottest missing experts (counter >= 2) are paired with the
      coldest resident ones and swapped while the newcomer beats the resident by
      1.5; the 96 largest gains over all layers are kept; after each round every
      counter is multiplied by 0.7.
  Belady -- evict the resident entry whose next use is farthest away (the replay
      ceiling the kairos README compares LRU against).

Readings of what the pages leave open (the library follows the same ones):
  - a routing event is the ids one token routes to in one layer; duplicates count
    once; resident ids are touched first in event order, then the misses are
    loaded in event order;
  - decayed scores: s <- s * 2^(-(t - tau) / half_life) + 1 at each access (t the
    token index); the victim has the lowest decayed score among entries outside
    the event and not accessed in the last `guard` tokens (all guarded: outside
    the event only); equal scores go to the least recently accessed, then the
    lower (layer, expert) index (a never-accessed entry is older than any other);
  - LFU counters and their arithmetic are fp32 (the Strata code's float counters);
    a round is one token: accesses, then (every fourth token) the swaps, then the
    decay; swapped-in experts count from the next token; misses do not load;
  - the pool starts empty or seeded from a profile (hottest first; seeded LRU
    entries are older than any access, the first listed the most recent of them).
"""
from __future__ import annotations

import math

import numpy as np

LRU, DECAYED_FREQ, LFU_SWAP = 0, 1, 2


class Policy:
    def __init__(self, kind: int, capacity: int, n_layers: int, n_experts: int, half_life: float = 32.0,
                 guard: int = 2, decay: float = 0.7, margin: float = 1.5, min_count: float = 2.0,
                 swap_every: int = 4, max_swaps: int = 96):
        self.kind, self.cap, self.L, self.E = kind, capacity, n_layers, n_experts
        self.half_life, self.guard = half_life, guard
        self.decay, self.margin, self.min_count = np.float32(decay), np.float32(margin), np.float32(min_count)
        self.swap_every, self.max_swaps = swap_every, max_swaps
        self.resident = set()
        self.order = []          # LRU: resident pairs, least recent first
        self.score = {}          # decayed frequency: pair -> (score, tau)
        self.last = {}           # pair -> token of last access
        self.stamp = {}          # pair -> access order
        self.clock = 0
        self.cnt = {}            # LFU: pair -> np.float32
        self.token = 0

    # -- helpers
    def _decayed(self, k):
        s, tau = self.score.get(k, (0.0, 0))
        return s * math.pow(math.pow(2.0, -1.0 / self.half_life), self.token - tau)

    def seed(self, pairs):
        placed = 0
        for k in pairs:
            if len(self.resident) >= self.cap:
                break
            k = tuple(k)
            if k in self.resident:
                continue
            self.resident.add(k)
            if self.kind == LRU:
                self.order.insert(0, k)  # older than anything seeded before it
            placed += 1
        return placed

    def _victim(self, event):
        if self.kind == LRU:
            for k in self.order:
                if k not in event:
                    return k
            return None
        for guarded in (True, False):
            best = None
            for k in sorted(self.resident):
                if k in event:
                    continue
                if guarded and k in self.last and self.token - self.last[k] < self.guard:
                    continue
                key = (self._decayed(k), self.stamp.get(k, 0), k)
                if best is None or key < best[0]:
                    best = (key, k)
            if best is not None:
                return best[1]
        return None

    def route(self, layer, ids):
        """Returns (hits [n] bool, loads [(expert, evicted pair or None)])."""
        hits = [(layer, int(e)) in self.resident for e in ids]
        event = []
        for e in ids:
            k = (layer, int(e))
            if k not in event:
                event.append(k)
        loads = []
        if self.kind == LFU_SWAP:
            for k in event:
                self.cnt[k] = np.float32(self.cnt.get(k, np.float32(0.0)) + np.float32(1.0))
            return hits, loads
        for k in event:
            if self.kind == LRU:
                if k in self.resident:
                    self.order.remove(k)
                    self.order.append(k)
            else:
                f = math.pow(2.0, -1.0 / self.half_life)
                s, tau = self.score.get(k, (0.0, 0))
                self.score[k] = (s * math.pow(f, self.token - tau) + 1.0, self.token)
                self.last[k] = self.token
                self.clock += 1
                self.stamp[k] = self.clock
        for k in event:
            if k in self.resident:
                continue
            victim = None
            if len(self.resident) >= self.cap:
                victim = self._victim(set(event))
                if victim is None:
                    continue
                self.resident.remove(victim)
                if self.kind == LRU:
                    self.order.remove(victim)
            self.resident.add(k)
            if self.kind == LRU:
                self.order.append(k)
            loads.append((k[1], victim))
        return hits, loads

    def end_token(self):
        """Returns the swaps made [(layer, in, out)]."""
        self.token += 1
        swaps = []
        if self.kind != LFU_SWAP:
            return swaps
        if self.token % self.swap_every == 0:
            gains = []
            for l in range(self.L):
                cand, vict = [], []
                for e in range(self.E):
                    c = self.cnt.get((l, e), np.float32(0.0))
                    if (l, e) in self.resident:
                        vict.append((c, e))
                    elif c >= self.min_count:
                        cand.append((c, e))
                cand.sort(key=lambda v: (-v[0], v[1]))
                vict.sort(key=lambda v: (v[0], v[1]))
                for i in range(min(len(cand), len(vict))):
                    if cand[i][0] < np.float32(vict[i][0] + self.margin):
                        break
                    gains.append((np.float32(cand[i][0] - vict[i][0]), l, i, cand[i][1], vict[i][1]))
            gains.sort(key=lambda g: (-g[0], g[1], g[2]))
            for g, l, _, e_in, e_out in gains[:self.max_swaps]:
                self.resident.remove((l, e_out))
                self.resident.add((l, e_in))
                swaps.append((l, e_in, e_out))
        for k in list(self.cnt):
            self.cnt[k] = np.float32(self.cnt[k] * self.decay)
        return swaps


def belady_hits(events, capacity, seed_pairs=()):
    """Hits of Belady's optimal demand cache over `events` (one list of (layer, ids)
    per token), the pool seeded like the policies: a miss evicts the resident entry
    (outside the current event) whose next use is farthest away."""
    import heapq
    seq = []
    for tok in events:
        for layer, ids in tok:
            ev = []
            for e in ids:
                k = (layer, int(e))
                if k not in ev:
                    ev.append(k)
            seq.append(ev)
    flat = [k for ev in seq for k in ev]
    nxt = [math.inf] * len(flat)
    seen = {}
    for i in range(len(flat) - 1, -1, -1):
        nxt[i] = seen.get(flat[i], math.inf)
        seen[flat[i]] = i
    first = {}
    for i, k in enumerate(flat):
        first.setdefault(k, i)
    resident, next_use, heap = set(), {}, []

    def push(k):
        heapq.heappush(heap, (-next_use[k], k))

    for k in seed_pairs:
        k = tuple(int(v) for v in k)
        if len(resident) >= capacity:
            break
        if k in resident:
            continue
        resident.add(k)
        next_use[k] = first.get(k, math.inf)
        push(k)
    hits, i = 0, 0
    for ev in seq:
        evs = set(ev)
        for k in ev:
            if k in resident:
                hits += 1
                next_use[k] = nxt[i]
                push(k)
            i += 1
        base = i - len(ev)
        for j, k in enumerate(ev):
            if k in resident:
                continue
            if len(resident) >= capacity:
                skipped, victim = [], None
                while heap:
                    nu, r = heapq.heappop(heap)
                    if r not in resident or next_use[r] != -nu:
                        continue  # stale entry
                    if r in evs:
                        skipped.append((nu, r))
                        continue
                    victim = r
                    break
                for item in skipped:
                    heapq.heappush(heap, item)
                if victim is None:
                    continue
                resident.remove(victim)
            resident.add(k)
            next_use[k] = nxt[base + j]
            push(k)
    return hits
