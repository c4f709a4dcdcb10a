"""Failure path without a fault: every kind of bounded wait the decode kernel uses gives
up after its bound when nothing will satisfy it (no hang, no trap), and the context
stays usable: decode calls afterwards run with state bit-exact and a clean status."""
import numpy as np
import pytest

from oracle.lru import SlotCache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ft():
    import __graft_entry__ as entry
    entry.build()
    import expert_cache_gb300
    return expert_cache_gb300


def test_bounded_waits_expire_and_context_stays_usable(ft):
    from expert_cache_gb300 import workloads as wl_mod
    assert ft.ft_check_bounded_waits() == 0xF      # counter, acquire, batch, mbarrier

    s = wl_mod.SHAPES["tiny"]
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr)
    wl = wl_mod.DecodeWorkload(s, seed=0, steps=4)
    ref = SlotCache(s.L, s.E, s.C)
    for t in range(wl.steps):
        for l in range(s.L):
            wl.run_layer(cache, t, l)
            r = ref.decode(l, wl.trace[t, l])
            assert wl.route_slot[t, l].cpu().numpy().tolist() == r.route_slot.tolist()
            assert wl.counters[t, l].cpu().numpy().tolist() == [r.n_hit, r.m, r.q, r.n_def_routes]
    for a, b in zip(ft.ft_cache_snapshot(cache.handle, s.L, s.E), ref.snapshot()):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
    pool.free()
