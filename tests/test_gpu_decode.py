"""GPU parity of the decode path through the C ABI against the CPU oracle.

Cache state (route slots, deferred list, counters, slot tables) must be bit-exact
per call; outputs y_gpu + y_cpu(oracle) must match the fp64 oracle within
rel-L2 5e-3 and max-abs 2e-2 * rms(y_ref).
"""
import numpy as np
import pytest
import torch

import synth
from oracle.formats import encode_record
from oracle.lru import SlotCache
from oracle.moe import decode_layer
from parity import assert_close, oracle_experts, oracle_shared

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ft():
    import __graft_entry__ as entry
    entry.build()
    import expert_cache_gb300
    return expert_cache_gb300


@pytest.fixture(scope="module")
def wl_mod(ft):
    from expert_cache_gb300 import workloads
    return workloads


def _check_call(ft, wl, ref, t, l, cache=None, check_tables=False):
    s = wl.shape
    r = ref.decode(l, wl.trace[t, l])
    got_rs = wl.route_slot[t, l].cpu().numpy()
    got_df = wl.deferred[t, l].cpu().numpy()
    got_ct = wl.counters[t, l].cpu().numpy().tolist()
    assert got_rs.tolist() == r.route_slot.tolist(), (t, l)
    assert got_df.tolist() == r.deferred.tolist(), (t, l)
    assert got_ct == [r.n_hit, r.m, r.q, r.n_def_routes], (t, l)
    if check_tables:
        for a, b in zip(ft.ft_cache_snapshot(cache.handle, s.L, s.E), ref.snapshot()):
            assert np.array_equal(np.asarray(a), np.asarray(b)), (t, l)
    return r


def _check_output(wl, r, t, l, experts, shared=None):
    s = wl.shape
    x = wl.x[t, l].float().cpu().numpy()
    y_ref = decode_layer(x, wl.trace[t, l], wl.gates[t, l], l, s.E, experts, shared)
    y_cpu = decode_layer(x, wl.trace[t, l], wl.gates[t, l], l, s.E, experts,
                         include=r.deferred >= 0)
    y = wl.y[t, l].cpu().numpy().astype(np.float64)
    assert_close(y + y_cpu, y_ref, f"step {t} layer {l}")


def test_quantiser_is_bit_exact(ft, wl_mod):
    for H, I, flats in ((64, 32, range(8)), (2048, 512, (0, 7777)), (4096, 2048, (123,))):
        rb = ft.ft_record_bytes(H, I)
        n = len(flats)
        w_gu = torch.stack([synth.expert_weights(1, f, H, I, "cuda")[0] for f in flats])
        w_d = torch.stack([synth.expert_weights(1, f, H, I, "cuda")[1] for f in flats])
        out = torch.empty(n * rb, dtype=torch.uint8, device="cuda")
        ft.ft_quantize_experts(w_gu, w_d, n, H, I, out)
        got = out.cpu().numpy().reshape(n, rb)
        for j, f in enumerate(flats):
            want = encode_record(*[w.numpy() for w in synth.expert_weights(1, f, H, I, "cpu")])
            assert np.array_equal(got[j], want), (H, I, f)


def test_quantiser_edge_blocks(ft):
    # zero matrix, a block of exact midpoints, huge and tiny blocks
    H, I = 64, 32
    g = torch.zeros((1, 2 * I, H), dtype=torch.float32)
    d = torch.zeros((1, H, I), dtype=torch.float32)
    g[0, 0, :16] = torch.tensor([6, 2.5, 3.5, 5, 0.25, 0.75, 1.25, 1.75, -2.5, -5, 0, 1, 2, 3, 4, -6.])
    g[0, 1, :16] = 1e-30
    g[0, 2, 16:32] = torch.linspace(-3000, 3000, 16)
    rb = ft.ft_record_bytes(H, I)
    out = torch.empty(2 * rb, dtype=torch.uint8, device="cuda")
    ft.ft_quantize_experts(torch.cat([g, g]).cuda(), torch.cat([d, torch.randn(1, H, I)]).cuda(),
                           2, H, I, out)
    got = out.cpu().numpy().reshape(2, rb)
    assert np.array_equal(got[0], encode_record(g[0].numpy(), d[0].numpy()))


@pytest.mark.parametrize("mode", ["full", "qstar"])
def test_tiny_decode_every_call(ft, wl_mod, mode):
    s = wl_mod.SHAPES["tiny"]
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I)
    f_q16 = ft.ft_split_from_bandwidth(50.0, 100.0)
    split = wl_mod.split_tuple(mode, f_q16)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr, split=split)
    wl = wl_mod.DecodeWorkload(s, seed=0)
    ref = SlotCache(s.L, s.E, s.C, full_offload=(mode == "full"), f_q16=f_q16)
    experts = oracle_experts(0, s.H, s.I)
    misses = 0
    for t in range(wl.steps):
        for l in range(s.L):
            wl.run_layer(cache, t, l)
            r = _check_call(ft, wl, ref, t, l, cache, check_tables=True)
            misses += r.m
            _check_output(wl, r, t, l, experts)
    assert misses > 0
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
    pool.free()


def test_decode_batch_duplicates_invalid_ids_shared_and_capacity(ft, wl_mod):
    L, E, H, I, k, B, C = 3, 16, 128, 64, 4, 3, 5
    pool = wl_mod.build_pool(2, L, E, H, I)
    shared = wl_mod.build_shared(2, L, H, I)
    cache = ft.ExpertCache(L, E, H, I, k, B, C, pool.ptr, shared=shared,
                           split=(ft.FT_SPLIT_QSTAR, 43691))
    ref = SlotCache(L, E, C, full_offload=False, f_q16=43691)
    experts = oracle_experts(2, H, I)
    rng = np.random.default_rng(7)
    x = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((B, H), dtype=torch.float32, device="cuda")
    dfr = torch.empty((B, k), dtype=torch.int32, device="cuda")
    rs = torch.empty_like(dfr)
    ct = torch.empty(4, dtype=torch.int32, device="cuda")
    for call in range(40):
        l = call % L
        ids = rng.integers(0, E, (B, k)).astype(np.int32)
        ids[0, 1] = ids[0, 0]                       # duplicate inside a row
        ids[1, :2] = ids[2, :2]                     # same experts on two tokens
        if call % 7 == 3:
            ids[2, 3] = 99 if call % 2 else -1      # invalid id: masked route
        gates = rng.random((B, k)).astype(np.float32)
        x.copy_(synth.decode_x(2, call, l, L, B, H, "cuda"))
        ft.ft_moe_decode(cache.handle, l, x, torch.from_numpy(ids).cuda(),
                         torch.from_numpy(gates).cuda(), B, k, y, dfr, rs, ct)
        r = ref.decode(l, ids)
        assert rs.cpu().numpy().tolist() == r.route_slot.tolist()
        assert dfr.cpu().numpy().tolist() == r.deferred.tolist()
        assert ct.cpu().numpy().tolist() == [r.n_hit, r.m, r.q, r.n_def_routes]
        for a, b in zip(ft.ft_cache_snapshot(cache.handle, L, E), ref.snapshot()):
            assert np.array_equal(np.asarray(a), np.asarray(b))
        st = ft.ft_cache_status(cache.handle)
        assert st == (ft.FT_DEV_BAD_ID if r.arg_error else 0)
        xx = x.float().cpu().numpy()
        sh = oracle_shared(2, l, H, I)
        y_ref = decode_layer(xx, ids, gates, l, E, experts, sh)
        y_cpu = decode_layer(xx, ids, gates, l, E, experts, include=r.deferred >= 0)
        assert_close(y.cpu().numpy() + y_cpu, y_ref, f"call {call}")
    cache.close()
    pool.free()


def test_all_routes_masked_gives_zero(ft, wl_mod):
    L, E, H, I = 1, 16, 64, 32
    pool = wl_mod.build_pool(3, L, E, H, I)
    cache = ft.ExpertCache(L, E, H, I, 2, 2, 4, pool.ptr)
    ids = torch.tensor([[-1, 16], [20, -5]], dtype=torch.int32, device="cuda")
    w = torch.ones((2, 2), dtype=torch.float32, device="cuda")
    x = torch.ones((2, H), dtype=torch.bfloat16, device="cuda")
    y = torch.full((2, H), 7.0, dtype=torch.float32, device="cuda")
    d = torch.empty((2, 2), dtype=torch.int32, device="cuda")
    ct = torch.empty(4, dtype=torch.int32, device="cuda")
    ft.ft_moe_decode(cache.handle, 0, x, ids, w, 2, 2, y, d, None, ct)
    assert torch.all(y == 0) and d.cpu().tolist() == [[-1, -1], [-1, -1]]
    assert ct.cpu().tolist() == [0, 0, 0, 0]
    assert ft.ft_cache_status(cache.handle) == ft.FT_DEV_BAD_ID
    cache.close()
    pool.free()


def test_resize_matches_oracle(ft, wl_mod):
    s = wl_mod.SHAPES["tiny"]
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr, capacity_max=12)
    wl = wl_mod.DecodeWorkload(s, seed=4)
    ref = SlotCache(s.L, s.E, s.C)
    experts = oracle_experts(0, s.H, s.I)
    plan = {10: 3, 20: 12}
    for t in range(wl.steps):
        if t in plan:
            ft.ft_cache_resize(cache.handle, plan[t], cache.slot_buf)
            ref.resize(plan[t])
        for l in range(s.L):
            wl.run_layer(cache, t, l)
            r = _check_call(ft, wl, ref, t, l, cache, check_tables=True)
            _check_output(wl, r, t, l, experts)
    with pytest.raises(ft.FtError):
        ft.ft_cache_resize(cache.handle, 13, cache.slot_buf)
    cache.close()
    pool.free()


@pytest.fixture(scope="module")
def qwen_pool(wl_mod):
    s = wl_mod.SHAPES["qwen_decode"]
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I)
    shared = wl_mod.build_shared(0, s.L, s.H, s.I)
    yield pool, shared
    pool.free()


@pytest.mark.parametrize("mode", ["full", "qstar"])
@pytest.mark.parametrize("p", [0.5, 0.8, 0.95])
def test_qwen_shaped_decode_full_size(ft, wl_mod, qwen_pool, p, mode):
    """Config at full size (40 x 256 experts, H 2048, I 512, 600 slots, shared expert)
    at locality p in {0.5, 0.8, 0.95}, full offload (q = m) and q* with B_H = 2 B_P
    (f = 1/2), in the launch configuration the benchmark times: state on every call,
    tables at the end, outputs on sampled (step, layer) pairs."""
    from dataclasses import replace
    s = replace(wl_mod.SHAPES["qwen_decode"], p=p)
    pool, shared = qwen_pool
    steps = 48
    split = wl_mod.split_tuple(mode, 32768)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr, shared=shared, split=split)
    wl = wl_mod.DecodeWorkload(s, seed=0, steps=steps)
    ref = SlotCache(s.L, s.E, s.C, full_offload=(mode == "full"), f_q16=32768)
    for t in range(steps):
        wl.run_step(cache, t)
    torch.cuda.synchronize()
    assert ft.ft_cache_status(cache.handle) == 0
    experts = oracle_experts(0, s.H, s.I)
    sample = {(0, 0), (1, 17), (5, 39), (31, 3), (steps - 1, 20)}
    shared_cache = {}
    misses = deferred = 0
    for t in range(steps):
        for l in range(s.L):
            r = _check_call(ft, wl, ref, t, l)
            misses += r.m
            deferred += r.n_def_routes
            if (t, l) in sample:
                if l not in shared_cache:
                    shared_cache[l] = oracle_shared(0, l, s.H, s.I)
                _check_output(wl, r, t, l, experts, shared_cache[l])
    assert misses > 0 and (deferred > 0) == (mode == "qstar")
    for a, b in zip(ft.ft_cache_snapshot(cache.handle, s.L, s.E), ref.snapshot()):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    cache.close()


def _abs_sum_of_terms(x, ids, gates, layer, E, experts, shared, include):
    """Per output element, the sum of |term| over the terms the GPU adds into y:
    |w_j o_j| of its routes and |shared|.  Bounds the reordering error of the sum."""
    from oracle.moe import swiglu
    x = np.asarray(x, np.float64)
    S = np.zeros_like(x)
    for b in range(ids.shape[0]):
        for j in range(ids.shape[1]):
            if include[b, j]:
                w_gu, w_d = experts(layer * E + int(ids[b, j]))
                S[b] += np.abs(float(gates[b, j]) * swiglu(w_gu, w_d, x[b:b + 1])[0])
        if shared is not None:
            S[b] += np.abs(swiglu(shared[0], shared[1], x[b:b + 1])[0])
    return S


def test_decode_repeat_differs_only_by_summation_order(ft, wl_mod, qwen_pool):
    """Race check: two caches with the same history make the same calls; the cache
    state must be identical and y may differ only by the order of its fp32 adds.
    For n terms summed in two orders the results differ by at most
    2 (n - 1) u sum|term| (u = 2^-24; checked with 2 n u); a lost, doubled or misplaced term is far larger.
    Checked on every element of sampled calls against that bound, and on every call
    against max |y1 - y2| <= 1e-5 rms(y), far below the 5e-3 parity tolerance."""
    s = wl_mod.SHAPES["qwen_decode"]
    pool, shared = qwen_pool
    steps = 8
    wls, caches = [], []
    for _ in range(2):
        caches.append(ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr, shared=shared))
        wls.append(wl_mod.DecodeWorkload(s, seed=3, steps=steps))
    for t in range(steps):
        for i in range(2):
            wls[i].run_step(caches[i], t)
    torch.cuda.synchronize()
    for name in ("route_slot", "deferred", "counters"):
        assert torch.equal(getattr(wls[0], name), getattr(wls[1], name)), name
    y1 = wls[0].y.double().cpu().numpy()
    y2 = wls[1].y.double().cpu().numpy()
    d = np.abs(y1 - y2)
    rms = np.sqrt(np.mean(y1 ** 2, axis=-1, keepdims=True))
    assert np.all(d <= 1e-5 * rms), f"largest |y1 - y2| / rms {np.max(d / rms):.2e}"
    experts = oracle_experts(0, s.H, s.I)
    n_terms = s.k + 1
    u = 2.0 ** -24
    for (t, l) in ((0, 0), (3, 21), (steps - 1, s.L - 1)):
        x = wls[0].x[t, l].float().cpu().numpy()
        sh = oracle_shared(0, l, s.H, s.I)
        inc = wls[0].route_slot[t, l].cpu().numpy() >= 0
        S = _abs_sum_of_terms(x, wls[0].trace[t, l], wls[0].gates[t, l], l, s.E, experts, sh, inc)
        assert np.all(d[t, l] <= 2 * n_terms * u * S), (t, l)
    for a, b in zip(ft.ft_cache_snapshot(caches[0].handle, s.L, s.E),
                    ft.ft_cache_snapshot(caches[1].handle, s.L, s.E)):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    print("calls with any differing element: %d of %d; largest |y1 - y2| / rms %.2e"
          % (int(np.any(d > 0, axis=(-1, -2)).sum()), steps * s.L, float(np.max(d / rms))))
    for c in caches:
        c.close()
