"""Global cross-layer LRU expert-slot cache: the state the device tables must match.

TEST INFRASTRUCTURE: see the package docstring for who may import this.

Sources:
  [EXPLAINER §3]      one slot holds one whole (layer, expert) pair; every layer
                      competes for one pool; the host pool stays the source of truth.
  [EXPLAINER §6.1]    per decode step: H = resident, M = unique missing, m = |M|;
                      routes are deduplicated across the batch; replacement is LRU
                      over all layers.
  [EXPLAINER §6.2]    M = F (filled, stays resident) disjoint-union C (computed on the
                      host, residency unchanged); q = |F|.
  [EXPLAINER §6.7]    choose at most q victims from the global LRU, copy the chosen
                      misses into them; the rest become CPU tasks.
  [EXPLAINER §8.2]    one pass picks K LRU candidates; the first q <= K are used.
  [JUHE "生成阶段：专家缓存到底怎么工作"]  slot_for_id[l][e] -> slot,
                      id_of_slot[slot] -> l*E + e, usage[slot] = current step.
  [JUHE "为什么 LRU 专家缓存会有效"]  hit: refresh usage; miss: take the least
                      recently used slot, update forward and reverse tables.
  [EXPLAINER §4.2-4.3] prefill borrows two whole-layer buffers from the same pool;
                      what they hold afterwards is decode's initial cache.
  [JUHE "Prefill 为什么不能也按需加载"]  the double buffer needs cache_size >= 2 * E.
  [EXPLAINER §7.2]    resize at a safe point: rebuild the GPU cache, keep the host
                      pool, let misses re-warm it.
  [EXPLAINER §4.3], [JUHE "Prefill 为什么不能也按需加载"]  when the free memory cannot
                      hold two whole layers the system does not over-allocate: it
                      falls back to loading on demand.

Readings where the pages are silent (each is listed in the design notes):
  * usage is stamped with a tick that advances once per call (per decode layer
    call and per prefill layer call), not once per token; within one call the
    touched slots are ordered by ascending slot index.
  * the first q misses in ascending flat id are filled; victim i takes fill i.
  * LRU order: never-used (free) slots first in ascending index, then occupied
    slots by ascending (usage, slot) -- which is the OrderedDict order below.
  * a route whose expert id is outside [0, E) is masked: neither hit, miss nor
    deferred, and the call reports an argument error.
  * a prefill load that finds an expert resident in another slot moves it: the
    old slot becomes free.
  * on-demand prefill (the fallback) loads the layer's routed union -- every expert
    some token of the chunk routes to -- through the LRU exactly like decode misses
    with every miss filled, in groups of at most C experts taken in ascending flat
    id; each group is one call (one tick; the first group ticks even when the union
    is empty) and is computed before the next group may evict it.
"""
from __future__ import annotations

import bisect
from collections import OrderedDict
from dataclasses import dataclass, field

import numpy as np

from .qrule import q_for_call


class CapacityError(ValueError):
    pass


@dataclass
class DecodeResult:
    route_slot: np.ndarray          # int32 [B, k]: slot, or -1 (deferred or masked)
    deferred: np.ndarray            # int32 [B, k]: flat id of a CPU-set route, else -1
    n_hit: int
    m: int
    q: int
    n_def_routes: int
    fills: list = field(default_factory=list)      # [(flat_id, slot)] in fill order
    hits: list = field(default_factory=list)       # hit flat ids, ascending
    arg_error: bool = False


class SlotCache:
    """OrderedDict model of the global LRU slot cache."""

    def __init__(self, L: int, E: int, capacity: int, full_offload: bool = True,
                 f_q16: int = 1 << 16):
        self.L, self.E = L, E
        self.full_offload = full_offload
        self.f_q16 = f_q16
        self.tick = 0
        self._empty(capacity)

    # -- state -------------------------------------------------------------
    def _empty(self, capacity: int):
        self.C = capacity
        self.slot_for_id: dict[int, int] = {}
        self.id_of_slot = [-1] * capacity
        self.usage = [-1] * capacity
        self.order: OrderedDict[int, None] = OrderedDict()   # occupied slots, LRU first
        self.free: list[int] = list(range(capacity))          # ascending

    def set_split(self, full_offload: bool, f_q16: int = 1 << 16):
        self.full_offload, self.f_q16 = full_offload, f_q16

    def resize(self, capacity: int):
        """Safe-point rebuild: every slot becomes free; the tick keeps counting."""
        self._empty(capacity)

    def snapshot(self):
        sfi = np.full(self.L * self.E, -1, np.int32)
        for f, s in self.slot_for_id.items():
            sfi[f] = s
        return (sfi, np.array(self.id_of_slot, np.int32),
                np.array(self.usage, np.int64), self.tick)

    def _stamp(self, slots):
        for s in sorted(slots):
            i = bisect.bisect_left(self.free, s)
            if i < len(self.free) and self.free[i] == s:
                self.free.pop(i)
            self.order.pop(s, None)
            self.order[s] = None
            self.usage[s] = self.tick

    def _map(self, flat: int, slot: int):
        old = self.id_of_slot[slot]
        if old >= 0:
            del self.slot_for_id[old]
        self.slot_for_id[flat] = slot
        self.id_of_slot[slot] = flat

    # -- decode ------------------------------------------------------------
    def decode(self, layer: int, ids) -> DecodeResult:
        ids = np.asarray(ids, np.int64)
        B, k = ids.shape
        E = self.E
        self.tick += 1
        valid = (ids >= 0) & (ids < E)
        U = sorted({layer * E + int(e) for e in ids[valid]})
        H = [u for u in U if u in self.slot_for_id]
        M = [u for u in U if u not in self.slot_for_id]
        q = q_for_call(len(M), len(H), self.C, self.full_offload, self.f_q16)
        hit_slots = {self.slot_for_id[u] for u in H}
        # LRU order of the slots this call did not touch: free ones, then occupied.
        candidates = list(self.free) + [s for s in self.order if s not in hit_slots]
        victims = candidates[:q]
        fills = list(zip(M[:q], victims))
        for flat, slot in fills:
            self._map(flat, slot)
        self._stamp(hit_slots | set(victims))

        route_slot = np.full((B, k), -1, np.int32)
        deferred = np.full((B, k), -1, np.int32)
        for b in range(B):
            for j in range(k):
                if not valid[b, j]:
                    continue
                flat = layer * E + int(ids[b, j])
                s = self.slot_for_id.get(flat, -1)
                route_slot[b, j] = s
                if s < 0:
                    deferred[b, j] = flat
        return DecodeResult(route_slot, deferred, len(H), len(M), q,
                            int((deferred >= 0).sum()), fills, H,
                            bool((~valid).any()))

    # -- prefill -----------------------------------------------------------
    def prefill(self, layer: int, double_buffer: bool) -> None:
        E = self.E
        if double_buffer and self.C < 2 * E:
            raise CapacityError("double buffering needs capacity >= 2 * num_experts")
        if self.C < E:
            raise CapacityError("prefill needs capacity >= num_experts")
        self.tick += 1
        touched = set(self._load_layer(layer, layer % 2 if double_buffer else 0))
        if double_buffer and layer + 1 < self.L:
            touched |= set(self._load_layer(layer + 1, (layer + 1) % 2))
        self._stamp(touched)

    def prefill_on_demand(self, layer: int, ids) -> list:
        """On-demand prefill of one layer: the routed union U (ascending flat id) in
        groups of at most C experts; per group, hits are touched and every miss takes
        the next least recently used slot that no hit of the group holds.  Returns
        the groups as lists of (flat id, slot, was_hit) in ascending flat id."""
        ids = np.asarray(ids, np.int64)
        E = self.E
        valid = (ids >= 0) & (ids < E)
        U = sorted({layer * E + int(e) for e in ids[valid]})
        groups = [U[i:i + self.C] for i in range(0, len(U), self.C)] or [[]]
        out = []
        for grp in groups:
            self.tick += 1
            H = [u for u in grp if u in self.slot_for_id]
            M = [u for u in grp if u not in self.slot_for_id]
            hit_slots = {self.slot_for_id[u] for u in H}
            candidates = list(self.free) + [s for s in self.order if s not in hit_slots]
            victims = candidates[:len(M)]
            for flat, slot in zip(M, victims):
                self._map(flat, slot)
            self._stamp(hit_slots | set(victims))
            out.append([(u, self.slot_for_id[u], u in H) for u in grp])
        return out

    def _load_layer(self, layer: int, buf: int):
        E = self.E
        slots = range(buf * E, buf * E + E)
        for e, s in zip(range(E), slots):
            flat = layer * E + e
            cur = self.slot_for_id.get(flat)
            if cur == s:
                continue
            if cur is not None:            # resident elsewhere: that slot becomes free
                del self.slot_for_id[flat]
                self.id_of_slot[cur] = -1
                self.usage[cur] = -1
                self.order.pop(cur, None)
                bisect.insort(self.free, cur)
            self._map(flat, s)
        return slots


class SlotCacheBruteForce:
    """Twin of SlotCache that keeps the whole touch history and re-derives the LRU
    order from it on every call (no OrderedDict, no usage array)."""

    def __init__(self, L, E, capacity, full_offload=True, f_q16=1 << 16):
        self.L, self.E = L, E
        self.full_offload, self.f_q16 = full_offload, f_q16
        self.tick = 0
        self.resize(capacity)

    def resize(self, capacity):
        self.C = capacity
        self.owner = [-1] * capacity           # slot -> flat id
        self.history: list[tuple[int, int]] = []   # (tick, slot), append-only

    def _last_touch(self, slot):
        last = None
        for t, s in self.history:
            if s == slot:
                last = t
        return last

    def _lru_order(self, exclude):
        free = [s for s in range(self.C) if self.owner[s] < 0 and s not in exclude]
        occ = [s for s in range(self.C) if self.owner[s] >= 0 and s not in exclude]
        occ.sort(key=lambda s: (self._last_touch(s), s))
        return free + occ

    def decode(self, layer, ids):
        ids = np.asarray(ids, np.int64)
        E = self.E
        self.tick += 1
        wanted = sorted({layer * E + int(e) for e in ids.reshape(-1) if 0 <= e < E})
        where = {f: s for s, f in enumerate(self.owner) if f >= 0}
        hits = [f for f in wanted if f in where]
        misses = [f for f in wanted if f not in where]
        q = q_for_call(len(misses), len(hits), self.C, self.full_offload, self.f_q16)
        hit_slots = {where[f] for f in hits}
        victims = self._lru_order(hit_slots)[:q]
        for f, s in zip(misses, victims):
            self.owner[s] = f
        for s in sorted(hit_slots | set(victims)):
            self.history.append((self.tick, s))
        return len(hits), len(misses), q

    def prefill_on_demand(self, layer, ids):
        """The routed union in groups of at most C, each group a call that fills
        every miss (re-derived from the touch history, like decode above)."""
        ids = np.asarray(ids, np.int64)
        E = self.E
        wanted = sorted({layer * E + int(e) for e in ids.reshape(-1) if 0 <= e < E})
        for g0 in range(0, max(len(wanted), 1), self.C):
            grp = wanted[g0:g0 + self.C]
            self.tick += 1
            where = {f: s for s, f in enumerate(self.owner) if f >= 0}
            hit_slots = {where[f] for f in grp if f in where}
            misses = [f for f in grp if f not in where]
            victims = self._lru_order(hit_slots)[:len(misses)]
            for f, s in zip(misses, victims):
                self.owner[s] = f
            for s in sorted(hit_slots | set(victims)):
                self.history.append((self.tick, s))

    def snapshot(self):
        sfi = np.full(self.L * self.E, -1, np.int32)
        usage = np.full(self.C, -1, np.int64)
        for s, f in enumerate(self.owner):
            if f >= 0:
                sfi[f] = s
                usage[s] = self._last_touch(s)
        return sfi, np.array(self.owner, np.int32), usage, self.tick
