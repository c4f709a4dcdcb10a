"""Pins for oracle.lru (global LRU slot cache) and oracle.static_placement."""
import numpy as np
import pytest

from conftest import read_golden
from oracle.lru import CapacityError, SlotCache, SlotCacheBruteForce
from oracle.static_placement import lru_miss_rate, static_miss_rate
from synth import locality_trace


def test_hand_worked_sequence():
    # C = 4 slots, one layer of 8 experts, full offload (q = m).
    c = SlotCache(1, 8, 4)
    r = c.decode(0, [[1, 0]])            # tick 1: misses 0,1 -> free slots 0,1
    assert (r.m, r.q, r.fills) == (2, 2, [(0, 0), (1, 1)])
    assert r.route_slot.tolist() == [[1, 0]]
    c.decode(0, [[2]])                   # tick 2: 2 -> slot 2
    r = c.decode(0, [[0, 3]])            # tick 3: hit 0 (slot 0); 3 -> free slot 3
    assert (r.n_hit, r.m, r.fills) == (1, 1, [(3, 3)])
    r = c.decode(0, [[4]])               # tick 4: LRU is slot 1 (tick 1) -> evict id 1
    assert r.fills == [(4, 1)]
    r = c.decode(0, [[5, 6]])            # tick 5: LRU order slot 2 (t2), then 0, 3 (t3)
    assert r.fills == [(5, 2), (6, 0)]
    sfi, ios, usage, tick = c.snapshot()
    assert ios.tolist() == [6, 4, 5, 3] and usage.tolist() == [5, 4, 5, 3] and tick == 5
    assert sfi.tolist() == [-1, -1, -1, 3, 1, 2, 0, -1]


def test_split_defers_the_tail_of_the_misses():
    c = SlotCache(1, 16, 8, full_offload=False, f_q16=16384)   # f = 1/4
    r = c.decode(0, [[9, 2, 7, 4]])      # m = 4 -> q = 1: fill the lowest id only
    assert (r.m, r.q, r.fills) == (4, 1, [(2, 0)])
    assert r.route_slot.tolist() == [[-1, 0, -1, -1]]
    assert r.deferred.tolist() == [[9, -1, 7, 4]] and r.n_def_routes == 3


def test_masked_routes():
    c = SlotCache(2, 8, 4)
    r = c.decode(1, [[3, 8], [-1, 3]])
    assert r.arg_error and r.m == 1 and r.n_hit == 0
    assert r.route_slot.tolist() == [[0, -1], [-1, 0]] and r.deferred.tolist() == [[-1, -1], [-1, -1]]


@pytest.mark.parametrize("seed", range(12))
def test_ordered_dict_matches_brute_force_history(seed):
    rng = np.random.default_rng(seed)
    L, E, B, k = 3, 8, 2, 3
    C = int(rng.integers(2, 10))
    full = bool(rng.integers(0, 2))
    f = int(rng.choice([16384, 32768, 43691, 65536]))
    a = SlotCache(L, E, C, full, f)
    b = SlotCacheBruteForce(L, E, C, full, f)
    for step in range(60):
        for l in range(L):
            ids = rng.integers(0, E, (B, k))
            r = a.decode(l, ids)
            assert (r.n_hit, r.m, r.q) == b.decode(l, ids)
            for x, y in zip(a.snapshot(), b.snapshot()):
                assert np.array_equal(x, y)
        if step == 30:
            a.resize(C + 1)
            b.resize(C + 1)


def test_capacity_covering_every_expert_only_misses_first_touches():
    L, E, B, k = 4, 16, 2, 3
    trace = locality_trace(5, L, E, k, B, 40, 0.5)
    c = SlotCache(L, E, L * E)
    seen, misses = set(), 0
    for t in range(trace.shape[0]):
        for l in range(L):
            r = c.decode(l, trace[t, l])
            misses += r.m
            seen |= {l * E + int(e) for e in trace[t, l].reshape(-1)}
    assert misses == len(seen)
    for l in range(L):                    # warm cache: zero misses from now on
        assert c.decode(l, trace[-1, l]).m == 0


def test_lru_beats_static_with_locality_not_without():
    rows = {r[0]: (float(r[1]), float(r[2])) for r in read_golden("lru_vs_static.txt")}
    E, k, steps = 256, 8, 4000
    loc = locality_trace(0, 1, E, k, 1, steps, 0.8)[:, 0, 0]
    lru, sta = lru_miss_rate(loc, E, 64), static_miss_rate(loc, E, 64)
    assert lru < sta / 3                                  # 3.8 % vs 72.7 % on the page
    hi = locality_trace(2, 1, E, k, 1, steps, 0.95)[:, 0, 0]
    assert lru_miss_rate(hi, E, 64) < static_miss_rate(hi, E, 64) / 10
    assert rows["locality"][0] < rows["locality"][1] / 10
    none = locality_trace(1, 1, E, k, 1, steps, 0.0)[:, 0, 0]
    lru0, sta0 = lru_miss_rate(none, E, 16), static_miss_rate(none, E, 16)
    assert lru0 >= sta0 - 0.01                            # 94.8 % vs 93.6 %: no gain
    assert rows["no_locality"][0] >= rows["no_locality"][1]


def test_prefill_double_buffer_state():
    L, E = 5, 4
    c = SlotCache(L, E, 10)
    c.decode(0, [[1, 2]])                 # something resident before the chunk
    for l in range(L):
        c.prefill(l, True)
    sfi, ios, usage, tick = c.snapshot()
    for l in range(L):
        for e in range(E):
            want = (l % 2) * E + e if l >= L - 2 else -1
            assert sfi[l * E + e] == want
    assert tick == 1 + L
    assert usage[: 2 * E].tolist() == [L + 1] * E + [L] * E    # layer L-1 stamped last


def test_prefill_single_buffer_and_capacity():
    c = SlotCache(3, 4, 6)
    with pytest.raises(CapacityError):
        c.prefill(0, True)
    for l in range(3):
        c.prefill(l, False)
    sfi = c.snapshot()[0]
    assert sfi[8:12].tolist() == [0, 1, 2, 3] and (sfi[:8] == -1).all()


def test_prefill_moves_an_expert_resident_elsewhere():
    c = SlotCache(2, 4, 10)
    c.decode(1, [[0]])                    # flat id 4 -> slot 0
    c.prefill(0, True)                    # layer 0 -> slots 0..3 (evicts id 4), layer 1 -> 4..7
    sfi, ios, usage, _ = c.snapshot()
    assert sfi.tolist() == [0, 1, 2, 3, 4, 5, 6, 7]
    assert ios.tolist() == [0, 1, 2, 3, 4, 5, 6, 7, -1, -1]


def test_resize_empties_and_keeps_counting():
    c = SlotCache(1, 8, 4)
    c.decode(0, [[1, 2, 3]])
    c.resize(2)
    sfi, ios, usage, tick = c.snapshot()
    assert (sfi == -1).all() and ios.tolist() == [-1, -1] and tick == 1
    r = c.decode(0, [[1, 2, 3]])          # cold again; only two slots
    assert (r.m, r.q, r.n_def_routes) == (3, 2, 1) and c.tick == 2


# ---------------------------------------------------------------- on-demand prefill

def test_on_demand_prefill_hand_worked():
    # L = 2, E = 8, C = 3.  Layer 0 decodes experts 0, 1 (slots 0, 1, tick 1); then
    # layer 1 prefills on demand with the routed union {1, 3, 4, 6, 7} = flats
    # {9, 11, 12, 14, 15} in groups of three: [9, 11, 12] then [14, 15].
    c = SlotCache(2, 8, 3)
    c.decode(0, [[0, 1]])
    ids = np.array([[1, 3], [4, 1], [6, 7], [3, 6]])
    groups = c.prefill_on_demand(1, ids)
    # group 1 (tick 2): no hits; victims in LRU order: free slot 2, then slots 0, 1
    # (tick 1, by slot) -> 9 -> 2, 11 -> 0 (evicts 0), 12 -> 1 (evicts 1)
    # group 2 (tick 3): LRU order 0, 1, 2 (all tick 2) -> 14 -> 0, 15 -> 1
    assert groups == [[(9, 2, False), (11, 0, False), (12, 1, False)],
                      [(14, 0, False), (15, 1, False)]]
    sfi, ios, usage, tick = c.snapshot()
    assert ios.tolist() == [14, 15, 9] and usage.tolist() == [3, 3, 2] and tick == 3
    assert [int(v) for v in np.nonzero(sfi >= 0)[0]] == [9, 14, 15]
    # hand-off: decode of layer 1 finds what the prefill left behind
    r = c.decode(1, [[1, 6]])
    assert (r.n_hit, r.m, r.q) == (2, 0, 0)


def test_on_demand_prefill_hits_stay_and_empty_union_ticks_once():
    c = SlotCache(1, 8, 4)
    c.decode(0, [[2, 5]])                                  # 2 -> 0, 5 -> 1 (tick 1)
    g = c.prefill_on_demand(0, np.array([[5, 7], [2, 7]]))
    assert g == [[(2, 0, True), (5, 1, True), (7, 2, False)]]       # one group, hits kept
    assert c.snapshot()[2].tolist() == [2, 2, 2, -1] and c.tick == 2
    before = c.snapshot()
    assert c.prefill_on_demand(0, np.array([[-1, 9]])) == [[]]       # masked routes only
    after = c.snapshot()
    assert after[3] == before[3] + 1
    for x, y in zip(after[:3], before[:3]):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("seed", range(8))
def test_on_demand_prefill_matches_brute_force_history(seed):
    """Decode calls and on-demand prefill layers interleaved (capacities below, at and
    above the union size): the OrderedDict model and the history twin agree."""
    rng = np.random.default_rng(100 + seed)
    L, E = 3, 16
    C = int(rng.integers(3, 20))
    a = SlotCache(L, E, C)
    b = SlotCacheBruteForce(L, E, C)
    for it in range(25):
        l = int(rng.integers(0, L))
        if it % 3 == 0:
            T, k = int(rng.integers(1, 12)), 4
            ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
            groups = a.prefill_on_demand(l, ids)
            b.prefill_on_demand(l, ids)
            union = sorted({l * E + int(e) for e in ids.reshape(-1)})
            assert [f for g in groups for (f, _, _) in g] == union
            assert all(len(g) <= C for g in groups)
            # the last group is resident after the call
            sfi = a.snapshot()[0]
            assert all(sfi[f] == s for (f, s, _) in groups[-1])
        else:
            ids = rng.integers(0, E, (2, 3))
            r = a.decode(l, ids)
            assert (r.n_hit, r.m, r.q) == b.decode(l, ids)
        for x, y in zip(a.snapshot(), b.snapshot()):
            assert np.array_equal(x, y)
