"""Host-driven failure cases and the state subsystems of the cache, through the C ABI:
a pageable pool is refused, a resize or restore while the stream is captured is
refused, snapshot + restore replays a run from a saved point, and the per-call
stats ring records every decode call.  Nothing here faults or hangs a GPU: every
failure is an argument or state the host checks before launching anything."""
import numpy as np
import pytest
import torch

from oracle.lru import SlotCache

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


def test_pageable_pool_is_refused(ft):
    L, E, H, I = 2, 16, 64, 32
    rb = ft.ft_record_bytes(H, I)
    pageable = np.zeros(L * E * rb + 256, np.uint8)       # ordinary (pageable) host memory
    addr = (pageable.ctypes.data + 255) // 256 * 256
    desc = ft.FtCacheDesc(L, E, H, I, 2, 1, 8, 0, 0, None, None, None, None,
                          ft.FtSplit(ft.FT_SPLIT_FULL_OFFLOAD, 65536))
    _, ws = ft.ft_cache_required_sizes(desc)
    slots = torch.empty(8 * rb, dtype=torch.uint8, device="cuda")
    work = torch.empty(ws, dtype=torch.uint8, device="cuda")
    desc.host_pool, desc.slot_buf, desc.workspace = addr, slots.data_ptr(), work.data_ptr()
    with pytest.raises(ft.FtError) as ei:
        ft.ft_cache_create(desc)
    assert ei.value.status == ft.FT_ERR_UNPINNED


def _capture_and_call(fn):
    """Run fn(stream) while `stream` is being captured into a CUDA graph; return the
    exception it raised (None if it returned)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    err = None
    with torch.cuda.graph(g, stream=side):
        try:
            fn(torch.cuda.current_stream().cuda_stream)
        except Exception as e:       # noqa: BLE001 - the status is checked by the caller
            err = e
    torch.cuda.current_stream().wait_stream(side)
    return err


def test_resize_and_restore_during_capture_are_refused(ft, wl_mod):
    s = wl_mod.SHAPES["tiny"]
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr)
    err = _capture_and_call(lambda st: ft.ft_cache_resize(cache.handle, s.C, cache.slot_buf, st))
    assert isinstance(err, ft.FtError) and err.status == ft.FT_ERR_STATE
    sfi, ios, usage, tick = ft.ft_cache_snapshot(cache.handle, s.L, s.E)
    err = _capture_and_call(lambda st: ft.ft_cache_restore(cache.handle, sfi, ios, usage, tick, st))
    assert isinstance(err, ft.FtError) and err.status == ft.FT_ERR_STATE
    # the cache is still usable afterwards
    wl = wl_mod.DecodeWorkload(s, seed=0, steps=2)
    wl.run_step(cache, 0)
    torch.cuda.synchronize()
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
    pool.free()


def test_restore_replays_a_run_from_a_saved_point(ft, wl_mod):
    """Snapshot the tables (and the slot bytes they describe) after step 10, run on,
    then restore and replay steps 10..: route slots, deferred lists, counters and
    tables repeat bit for bit, y within the reordering bound of its fp32 adds."""
    s = wl_mod.SHAPES["tiny"]
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I)
    f_q16 = ft.ft_split_from_bandwidth(50.0, 100.0)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr,
                           split=wl_mod.split_tuple("qstar", f_q16))
    wl = wl_mod.DecodeWorkload(s, seed=0)
    ref = SlotCache(s.L, s.E, s.C, full_offload=False, f_q16=f_q16)
    t0 = 10
    for t in range(t0):
        wl.run_step(cache, t)
        for l in range(s.L):
            ref.decode(l, wl.trace[t, l])
    torch.cuda.synchronize()
    saved = ft.ft_cache_snapshot(cache.handle, s.L, s.E)
    saved_slots = cache.slot_buf.clone()
    for a, b in zip(saved, ref.snapshot()):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    for t in range(t0, wl.steps):
        wl.run_step(cache, t)
    torch.cuda.synchronize()
    first = [getattr(wl, n)[t0:].clone() for n in ("route_slot", "deferred", "counters", "y")]
    end_state = ft.ft_cache_snapshot(cache.handle, s.L, s.E)
    # back to the saved point: slot bytes first (the caller's buffer), then the tables
    cache.slot_buf.copy_(saved_slots)
    ft.ft_cache_restore(cache.handle, *saved)
    for a, b in zip(ft.ft_cache_snapshot(cache.handle, s.L, s.E), saved):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    for t in range(t0, wl.steps):
        wl.run_step(cache, t)
    torch.cuda.synchronize()
    second = [getattr(wl, n)[t0:] for n in ("route_slot", "deferred", "counters", "y")]
    for a, b in zip(first[:3], second[:3]):
        assert torch.equal(a, b)
    y1, y2 = first[3].double().cpu().numpy(), second[3].double().cpu().numpy()
    rms = np.sqrt(np.mean(y1 ** 2, axis=-1, keepdims=True))
    assert np.all(np.abs(y1 - y2) <= 1e-5 * rms)
    for a, b in zip(ft.ft_cache_snapshot(cache.handle, s.L, s.E), end_state):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
    pool.free()


def test_restore_rejects_inconsistent_tables(ft, wl_mod):
    s = wl_mod.SHAPES["tiny"]
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr)
    wl = wl_mod.DecodeWorkload(s, seed=0, steps=4)
    for t in range(4):
        wl.run_step(cache, t)
    sfi, ios, usage, tick = ft.ft_cache_snapshot(cache.handle, s.L, s.E)
    occ = int(np.nonzero(ios >= 0)[0][0])
    bad = []
    b = ios.copy(); b[occ] = (ios[occ] + 1) % (s.L * s.E); bad.append((sfi, b, usage, tick))
    b = usage.copy(); b[occ] = tick + 1; bad.append((sfi, ios, b, tick))
    b = usage.copy(); b[occ] = -1; bad.append((sfi, ios, b, tick))
    b = sfi.copy(); b[int(ios[occ])] = -1; bad.append((b, ios, usage, tick))
    b = sfi.copy(); b[0 if ios[occ] != 0 else 1] = s.C; bad.append((b, ios, usage, tick))
    for args in bad:
        with pytest.raises(ft.FtError) as ei:
            ft.ft_cache_restore(cache.handle, *args)
        assert ei.value.status == ft.FT_ERR_ARG
    # nothing was written by the refused calls
    for a, b_ in zip(ft.ft_cache_snapshot(cache.handle, s.L, s.E), (sfi, ios, usage, tick)):
        assert np.array_equal(np.asarray(a), np.asarray(b_))
    cache.close()
    pool.free()


def test_stats_ring_records_every_decode_call(ft, wl_mod):
    s = wl_mod.SHAPES["tiny"]
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I)
    f_q16 = ft.ft_split_from_bandwidth(50.0, 100.0)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr,
                           split=wl_mod.split_tuple("qstar", f_q16))
    cap = 16
    ring = torch.zeros(ft.TRACE_HEADER_BYTES + cap * ft.TRACE_DTYPE.itemsize, dtype=torch.uint8,
                       device="cuda")
    ft.ft_cache_set_trace(cache.handle, ring, cap)
    wl = wl_mod.DecodeWorkload(s, seed=0, steps=20)
    ref = SlotCache(s.L, s.E, s.C, full_offload=False, f_q16=f_q16)
    want = []
    for t in range(20):
        wl.run_step(cache, t)
        for l in range(s.L):
            r = ref.decode(l, wl.trace[t, l])
            want.append((t * s.L + l + 1, l, r.n_hit, r.m, r.q, r.n_def_routes))
    torch.cuda.synchronize()
    count, recs = ft.trace_records(ring.cpu().numpy(), cap)
    assert count == 20 * s.L
    got = [(int(r["tick"]), int(r["layer"]), int(r["n_hit"]), int(r["m"]), int(r["q"]),
            int(r["n_def_routes"])) for r in recs]
    assert got == want[-cap:]
    assert all(int(r["n_units"]) == int(r["n_hit"]) + int(r["q"]) for r in recs)
    assert np.all(np.diff(recs["t_commit_ns"]) >= 0)
    ft.ft_cache_set_trace(cache.handle, None, 0)             # off: later calls leave it alone
    wl.run_step(cache, 0)
    torch.cuda.synchronize()
    assert ft.trace_records(ring.cpu().numpy(), cap)[0] == count
    cache.close()
    pool.free()
