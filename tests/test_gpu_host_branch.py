"""The host branch on the GPU machine.  With a branch attached, every decode call hands its
deferred routes to the host workers through the mailbox and the join kernel adds their
partial: y must be the whole layer output, so it is checked against the oracle's full
sum with no CPU partial added by the test.  Also: the branch's NEON GEMV against the
oracle, the hand-off under CUDA-graph replay at the benchmark shape, the static entry
point, and the bandwidth profile (sane rates, the backend rule, an empty cache after)."""
import numpy as np
import pytest
import torch

import synth
from oracle.lru import SlotCache
from oracle.moe import decode_layer
from oracle.qrule import recommend_backend, split_from_overlap
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


def test_neon_host_share_matches_oracle(ft):
    """The branch's GEMV on this host (NEON on aarch64) against the oracle."""
    import test_host_branch as hbt
    for fmt in ("nvfp4", "mxfp4"):
        hbt.test_host_share_matches_oracle_tiny(ft, fmt)
    hbt.test_host_share_deterministic_over_thread_counts(ft)
    hbt.test_host_share_qwen_shape(ft)


@pytest.mark.parametrize("static,fmt", [(False, "nvfp4"), (True, "nvfp4"), (False, "mxfp4")])
def test_hybrid_decode_is_whole_layer(ft, wl_mod, static, fmt):
    """q* split at f = 1/2 with a branch attached: tables bit-exact with the oracle,
    y = y_gpu + y_host against the oracle's full sum (shared expert included)."""
    L, E, H, I, k, B, C = 3, 16, 128, 64, 4, 2, 6
    pool = wl_mod.build_pool(2, L, E, H, I, fmt=fmt)
    shared = wl_mod.build_shared(2, L, H, I, fmt=fmt)
    cache = ft.ExpertCache(L, E, H, I, k, B, C, pool.ptr, shared=shared, split=(ft.FT_SPLIT_QSTAR, 32768),
                           fmt=fmt)
    hb = ft.HostBranch(L, E, H, I, k, B, pool.ptr, 4, fmt=fmt)
    ft.ft_cache_set_host_branch(cache.handle, hb.handle)
    ref = SlotCache(L, E, C, full_offload=False, f_q16=32768)
    experts = oracle_experts(2, H, I, fmt)
    rng = np.random.default_rng(11)
    x = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((B, H), dtype=torch.float32, device="cuda")
    dfr = torch.empty((B, k), dtype=torch.int32, device="cuda")
    ct = torch.empty(4, dtype=torch.int32, device="cuda")
    call_fn = ft.ft_moe_decode_static if static else ft.ft_moe_decode
    n_host_calls = 0
    for call in range(30):
        l = call % L
        ids = rng.integers(0, E, (B, k)).astype(np.int32)
        gates = rng.random((B, k)).astype(np.float32)
        x.copy_(synth.decode_x(2, call, l, L, B, H, "cuda"))
        call_fn(cache.handle, l, x, torch.from_numpy(ids).cuda(), torch.from_numpy(gates).cuda(), B, k, y,
                dfr, None, ct)
        r = ref.decode(l, ids)
        assert dfr.cpu().numpy().tolist() == r.deferred.tolist()
        assert ct.cpu().numpy().tolist() == [r.n_hit, r.m, r.q, r.n_def_routes]
        n_host_calls += r.n_def_routes > 0
        xx = x.float().cpu().numpy()
        y_ref = decode_layer(xx, ids, gates, l, E, experts, oracle_shared(2, l, H, I, fmt))
        assert_close(y.cpu().numpy(), y_ref, f"call {call}")
    assert n_host_calls > 5
    jobs, mailbox_jobs = ft.ft_host_branch_stats(hb.handle)
    assert mailbox_jobs == n_host_calls
    assert ft.ft_cache_status(cache.handle) == 0
    ft.ft_cache_set_host_branch(cache.handle, None)
    cache.close()
    hb.close()
    pool.free()


def test_hybrid_decode_graph_replay_qwen_shape(ft, wl_mod):
    """The benchmark's layer shape at p = 0.5, f = 1/2, whole steps as graph replays:
    sampled (step, layer) outputs against the oracle's full sum."""
    from dataclasses import replace
    s = replace(wl_mod.SHAPES["qwen_decode"], L=4, E=64, C=96, p=0.5)
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I)
    shared = wl_mod.build_shared(0, s.L, s.H, s.I)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr, shared=shared,
                           split=(ft.FT_SPLIT_QSTAR, 32768))
    hb = ft.HostBranch(s.L, s.E, s.H, s.I, s.k, s.B, pool.ptr, 8)
    ft.ft_cache_set_host_branch(cache.handle, hb.handle)
    wl = wl_mod.DecodeWorkload(s, seed=5, steps=24)
    for t in range(4):
        wl.run_step(cache, t)
    g = wl_mod.StepGraph(wl, cache)
    g.capture()
    for t in range(4, 24):
        g.replay(t)
    torch.cuda.synchronize()
    experts = oracle_experts(0, s.H, s.I)
    ct = wl.counters.cpu().numpy()
    assert ct[4:, :, 3].sum() > 0                          # some routes went to the host
    checked = 0
    for t in (5, 11, 17, 23):
        for l in range(s.L):
            x = wl.x[t, l].float().cpu().numpy()
            y_ref = decode_layer(x, wl.trace[t, l], wl.gates[t, l], l, s.E, experts, oracle_shared(0, l, s.H, s.I))
            assert_close(wl.y[t, l].cpu().numpy(), y_ref, f"step {t} layer {l}")
            checked += 1
    assert checked == 16
    assert ft.ft_cache_status(cache.handle) == 0
    ft.ft_cache_set_host_branch(cache.handle, None)
    cache.close()
    hb.close()
    pool.free()


def test_host_branch_attach_errors(ft, wl_mod):
    L, E, H, I = 1, 8, 64, 32
    pool = wl_mod.build_pool(1, L, E, H, I)
    other = wl_mod.build_pool(1, L, E, H, I)
    cache = ft.ExpertCache(L, E, H, I, 2, 2, 4, pool.ptr)
    for hb in (ft.HostBranch(L, E, H, I, 2, 2, other.ptr, 1),          # another pool
               ft.HostBranch(L, E, H, I, 1, 2, pool.ptr, 1),           # k_max below the cache's
               ft.HostBranch(L, E, H, I, 2, 2, pool.ptr, 1, mailbox=False)):
        with pytest.raises(ft.FtError):
            ft.ft_cache_set_host_branch(cache.handle, hb.handle)
        hb.close()
    cache.close()
    pool.free()
    other.free()


def test_bandwidth_profile(ft, wl_mod):
    """Both paths over 48 records of the benchmark's record size; the recommendation
    and the overlap split follow the oracle's rules; the cache is empty afterwards."""
    L, E, H, I = 1, 64, 2048, 512
    pool = wl_mod.build_pool(0, L, E, H, I)
    cache = ft.ExpertCache(L, E, H, I, 8, 1, 64, pool.ptr)
    hb = ft.HostBranch(L, E, H, I, 8, 1, pool.ptr, 8, mailbox=False)
    for t in range(2):                                     # some residency before
        ids = torch.arange(8 * t, 8 * t + 8, dtype=torch.int32, device="cuda")[None]
        ft.ft_moe_decode(cache.handle, 0, torch.ones((1, H), dtype=torch.bfloat16, device="cuda"), ids,
                         torch.ones((1, 8), device="cuda"), 1, 8, torch.empty((1, H), device="cuda"),
                         torch.empty((1, 8), dtype=torch.int32, device="cuda"))
    prof = ft.ft_profile_bandwidth(cache.handle, hb.handle, 48)
    assert prof["n_records"] == 48
    for key in ("pcie_gbs", "cpu_gbs", "pcie_ov_gbs", "cpu_ov_gbs"):
        assert 0.1 < prof[key] < 5000, (key, prof)
    want = ft.FT_BACKEND_HYBRID if recommend_backend(prof["cpu_gbs"], prof["pcie_gbs"]) == "hybrid" \
        else ft.FT_BACKEND_OFFLOAD
    assert prof["recommend"] == want
    assert prof["f_q16"] == split_from_overlap(prof["pcie_ov_gbs"], prof["cpu_ov_gbs"])
    sfi, ios, usage, tick = ft.ft_cache_snapshot(cache.handle, L, E)
    assert np.all(np.asarray(sfi) == -1) and np.all(np.asarray(ios) == -1)
    with pytest.raises(ft.FtError):
        ft.ft_profile_bandwidth(cache.handle, hb.handle, 65)  # more records than slots
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
    hb.close()
    pool.free()
