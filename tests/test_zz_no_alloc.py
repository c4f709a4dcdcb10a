"""ft_moe_decode_static: the decode call whose per-call scratch is a static device
array, for callers that cannot allocate device memory (a framework that owns every
device allocation through its own pool, or a serving loop that must never enter the
CUDA allocator).  Checked through the C ABI against ft_moe_decode on two calls in
a row: two caches with the same history, one driven by each entry point."""
import numpy as np
import pytest
import torch

from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ft():
    import __graft_entry__ as entry
    entry.build()
    import expert_cache_gb300
    return expert_cache_gb300


def test_static_scratch_decode_matches_workspace_decode(ft):
    from expert_cache_gb300.workloads import SHAPES, DecodeWorkload, build_pool, build_shared
    s = SHAPES["tiny"]
    L, E, H, I, k, B, C = s.L, s.E, 128, 64, 3, 2, 5
    pool = build_pool(11, L, E, H, I)
    shared = build_shared(11, L, H, I)
    split = (ft.FT_SPLIT_QSTAR, 43691)
    ref = ft.ExpertCache(L, E, H, I, k, B, C, pool.ptr, shared=shared, split=split)
    new = ft.ExpertCache(L, E, H, I, k, B, C, pool.ptr, shared=shared, split=split)
    rng = np.random.default_rng(5)
    x = torch.randn((B, H), device="cuda").to(torch.bfloat16)
    outs = {}
    for name, cache, fn in (("ref", ref, ft.ft_moe_decode), ("static", new, ft.ft_moe_decode_static)):
        rng = np.random.default_rng(5)
        res = []
        for call in range(2):                       # two calls in a row
            ids = torch.from_numpy(rng.integers(0, E, (B, k)).astype(np.int32)).cuda()
            w = torch.from_numpy(rng.random((B, k)).astype(np.float32)).cuda()
            y = torch.full((B, H), float("nan"), device="cuda")
            d = torch.empty((B, k), dtype=torch.int32, device="cuda")
            rs = torch.empty_like(d)
            ct = torch.empty(4, dtype=torch.int32, device="cuda")
            fn(cache.handle, call % L, x, ids, w, B, k, y, d, rs, ct)
            torch.cuda.synchronize()
            res.append((y.cpu().numpy(), d.cpu().numpy(), rs.cpu().numpy(), ct.cpu().numpy()))
        outs[name] = res
    for (y0, d0, r0, c0), (y1, d1, r1, c1) in zip(outs["ref"], outs["static"]):
        assert np.array_equal(d0, d1) and np.array_equal(r0, r1) and np.array_equal(c0, c1)
        assert np.all(np.isfinite(y1))
        assert_close(y1, y0, "static vs workspace decode")
    for a, b in zip(ft.ft_cache_snapshot(ref.handle, L, E), ft.ft_cache_snapshot(new.handle, L, E)):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    ref.close()
    new.close()
    pool.free()


def test_static_scratch_two_caches_benchmark_shape(ft):
    """Two caches of different shapes take turns on the shared static array: the
    Qwen3.6-shaped layer of the benchmark (H 2048, I 512, top-8 + shared expert,
    600 slots) and a small one (H 256, I 128, batch 3, top-4).  Each is paired
    with a twin driven through ft_moe_decode; state must be bit-exact and y may
    differ only by the order of its fp32 adds (far inside the parity tolerance)."""
    from expert_cache_gb300.workloads import (SHAPES, DecodeWorkload, Shape, build_pool,
                                              build_shared)
    q = SHAPES["qwen_decode"]
    small = Shape("small", L=3, E=16, k=4, H=256, I=128, C=12, B=3, steps=8, p=0.5, shared=True)
    steps = 3
    setups = []
    for s_ in (q, small):
        pool = build_pool(13, s_.L, s_.E, s_.H, s_.I)
        shared = build_shared(13, s_.L, s_.H, s_.I)
        pair = [ft.ExpertCache(s_.L, s_.E, s_.H, s_.I, s_.k, s_.B, s_.C, pool.ptr, shared=shared)
                for _ in range(2)]
        wls = [DecodeWorkload(s_, seed=2, steps=steps) for _ in range(2)]
        setups.append((s_, pool, shared, pair, wls))
    for t in range(steps):
        for l in range(max(q.L, small.L)):
            for s_, _, _, pair, wls in setups:      # the two shapes alternate on the array
                if l >= s_.L:
                    continue
                x, ids, w, y, d, rs, ct = wls[1].addresses(t, l)
                ft.ft_moe_decode_static(pair[1].handle, l, x, ids, w, s_.B, s_.k, y, d, rs, ct)
                wls[0].run_layer(pair[0], t, l)
    torch.cuda.synchronize()
    for s_, pool, _, pair, wls in setups:
        for name in ("route_slot", "deferred", "counters"):
            assert torch.equal(getattr(wls[0], name), getattr(wls[1], name)), (s_.name, name)
        y0 = wls[0].y.double().cpu().numpy()
        y1 = wls[1].y.double().cpu().numpy()
        assert np.all(np.isfinite(y1))
        rms = np.sqrt(np.mean(y0 ** 2, axis=-1, keepdims=True))
        assert np.all(np.abs(y1 - y0) <= 1e-5 * rms), s_.name
        assert_close(y1, y0, s_.name)
        for a, b in zip(ft.ft_cache_snapshot(pair[0].handle, s_.L, s_.E),
                        ft.ft_cache_snapshot(pair[1].handle, s_.L, s_.E)):
            assert np.array_equal(np.asarray(a), np.asarray(b)), s_.name
        assert ft.ft_cache_status(pair[1].handle) == 0
        for c in pair:
            c.close()
        pool.free()


def test_static_scratch_rejects_oversized_calls(ft):
    from expert_cache_gb300.workloads import build_pool
    # (B*k + B) * I * 8 bytes of tagged h: 1024 pairs x 2048 x 8 B = 16 MiB > 8 MiB
    L, E, H, I, k, B = 1, 4, 4096, 2048, 31, 32
    pool = build_pool(12, L, E, H, I)
    cache = ft.ExpertCache(L, E, H, I, k, B, 4, pool.ptr)
    ids = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    w = torch.ones((B, k), device="cuda")
    x = torch.zeros((B, H), device="cuda").to(torch.bfloat16)
    y = torch.empty((B, H), device="cuda")
    d = torch.empty((B, k), dtype=torch.int32, device="cuda")
    with pytest.raises(ft.FtError) as ei:
        ft.ft_moe_decode_static(cache.handle, 0, x, ids, w, B, k, y, d)
    assert ei.value.status == ft.FT_ERR_ARG
    ft.ft_moe_decode_static(cache.handle, 0, x, ids[:1, :1], w[:1, :1], 1, 1, y, d)
    torch.cuda.synchronize()
    cache.close()
    pool.free()
