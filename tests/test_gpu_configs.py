"""Full-size parity of the DeepSeek-V4-Flash-shaped workloads through the C ABI.

State (route slots, deferred list, counters) is checked on every call and the
tables after each phase; outputs on sampled (step, layer, token) triples -- tokens
are independent, so the oracle computes only the sampled rows (each DSV4-shaped
expert costs the fp64 oracle seconds).
"""
import numpy as np
import pytest
import torch

from oracle.lru import SlotCache
from oracle.moe import decode_layer
from parity import assert_close, oracle_experts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ft():
    import __graft_entry__ as entry
    entry.build()
    import expert_cache_gb300
    return expert_cache_gb300


@pytest.fixture(scope="module")
def dsv4_pool(ft):
    from expert_cache_gb300.workloads import SHAPES, build_pool
    s = SHAPES["dsv4_decode"]
    pool = build_pool(0, s.L, s.E, s.H, s.I)
    yield pool
    pool.free()


def _check_calls(wl, ref, t0, t1, samples, experts):
    s = wl.shape
    for t in range(t0, t1):
        for l in range(s.L):
            r = ref.decode(l, wl.trace[t, l])
            assert wl.route_slot[t, l].cpu().numpy().tolist() == r.route_slot.tolist(), (t, l)
            assert wl.deferred[t, l].cpu().numpy().tolist() == r.deferred.tolist(), (t, l)
            assert wl.counters[t, l].cpu().numpy().tolist() == [r.n_hit, r.m, r.q, r.n_def_routes], (t, l)
            for (ts, ls, b) in samples:
                if (ts, ls) != (t, l):
                    continue
                x = wl.x[t, l, b:b + 1].float().cpu().numpy()
                ids = wl.trace[t, l, b:b + 1]
                g = wl.gates[t, l, b:b + 1]
                y_ref = decode_layer(x, ids, g, l, s.E, experts)
                y_cpu = decode_layer(x, ids, g, l, s.E, experts, include=r.deferred[b:b + 1] >= 0)
                y = wl.y[t, l, b:b + 1].cpu().numpy().astype(np.float64)
                assert_close(y + y_cpu, y_ref, f"step {t} layer {l} token {b}")


@pytest.mark.parametrize("B", [1, 4])
@pytest.mark.parametrize("f", [2 / 3, 0.5, 0.25])
def test_dsv4_shaped_decode(ft, dsv4_pool, f, B):
    """16 layers x 256 experts (H 4096, I 2048), 1024 slots, locality 0.8, q* split
    with f = B_P / B_H for B_H / B_P in {1.5, 2, 4}, batch 1 and 4."""
    from dataclasses import replace
    from expert_cache_gb300.workloads import SHAPES, DecodeWorkload, split_tuple
    s = replace(SHAPES["dsv4_decode"], B=B)
    steps = 24
    f_q16 = ft.ft_split_from_bandwidth(f, 1.0)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, dsv4_pool.ptr,
                           split=split_tuple("qstar", f_q16))
    wl = DecodeWorkload(s, seed=1, steps=steps)
    for t in range(steps):
        wl.run_step(cache, t)
    torch.cuda.synchronize()
    ref = SlotCache(s.L, s.E, s.C, full_offload=False, f_q16=f_q16)
    samples = [(0, 0, 0), (steps - 1, s.L - 1, B - 1)]
    _check_calls(wl, ref, 0, steps, samples, oracle_experts(0, s.H, s.I))
    for a, b in zip(ft.ft_cache_snapshot(cache.handle, s.L, s.E), ref.snapshot()):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    cache.close()


def test_stress_elastic_resize_overlap_split(ft, dsv4_pool):
    """Batch 16, locality 0.3, the slot cache resized 1024 -> 256 -> 768 mid-run
    without touching the host pool; split f = p_ov / (p_ov + c_ov) with 48 / 40 GB/s;
    deferred routes merged with the oracle's host partial."""
    from expert_cache_gb300.workloads import SHAPES, DecodeWorkload, split_tuple
    s = SHAPES["stress"]
    f_q16 = ft.ft_split_from_overlap(48.0, 40.0)
    assert f_q16 == 35747
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, dsv4_pool.ptr,
                           split=split_tuple("qstar", f_q16), capacity_max=1024)
    wl = DecodeWorkload(s, seed=0)
    ref = SlotCache(s.L, s.E, s.C, full_offload=False, f_q16=f_q16)
    experts = oracle_experts(0, s.H, s.I)
    samples = [(0, 0, 0), (170, 15, 3), (171, 0, 7), (342, 5, 15), (s.steps - 1, 9, 11)]
    bounds = [0] + sorted(s.resize) + [s.steps]
    for i in range(len(bounds) - 1):
        t0, t1 = bounds[i], bounds[i + 1]
        if t0 in s.resize:
            ft.ft_cache_resize(cache.handle, s.resize[t0], cache.slot_buf)
            ref.resize(s.resize[t0])
            assert ft.ft_cache_capacity(cache.handle) == s.resize[t0]
        for t in range(t0, t1):
            wl.run_step(cache, t)
        torch.cuda.synchronize()
        _check_calls(wl, ref, t0, t1, samples, experts)
        for a, b in zip(ft.ft_cache_snapshot(cache.handle, s.L, s.E), ref.snapshot()):
            assert np.array_equal(np.asarray(a), np.asarray(b))
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
