"""MXFP4 expert records (E2M1 codes, E8M0 scale per 32) on the GPU path, against the
oracle: the record quantiser bit for bit; decode (the GEMV reads E8M0 scales natively,
any exponent) with the cache state bit-exact and outputs in tolerance; prefill (the
tcgen05 GEMM takes each E8M0 scale as the equal UE4M3 pair, exact for 2^-9..2^8;
outside that range the call flags FT_DEV_SCALE_RANGE)."""
import numpy as np
import pytest
import torch

import synth
from oracle.formats import encode_record
from oracle.lru import SlotCache
from oracle.moe import decode_layer, prefill_from_h, prefill_layer
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


def test_mx_quantiser_is_bit_exact(ft):
    for H, I, flats, scale in ((64, 32, range(6), 1.0), (2048, 512, (0, 7777), 1.0),
                               (4096, 2048, (123,), 1.0), (256, 256, (5, 6), 2.0 ** 20),
                               (256, 256, (7,), 2.0 ** -40)):
        rb = ft.ft_record_bytes(H, I, "mxfp4")
        n = len(flats)
        w_gu = torch.stack([synth.expert_weights(1, f, H, I, "cuda")[0] for f in flats]) * scale
        w_d = torch.stack([synth.expert_weights(1, f, H, I, "cuda")[1] for f in flats]) * scale
        out = torch.empty(n * rb, dtype=torch.uint8, device="cuda")
        ft.ft_quantize_experts(w_gu, w_d, n, H, I, out, fmt="mxfp4")
        got = out.cpu().numpy().reshape(n, rb)
        for j, f in enumerate(flats):
            want = encode_record(*[w.numpy() * np.float32(scale)
                                   for w in synth.expert_weights(1, f, H, I, "cpu")], "mxfp4")
            assert np.array_equal(got[j], want), (H, I, f, scale)


def test_mx_quantiser_edge_blocks(ft):
    H, I = 64, 32
    g = torch.zeros((1, 2 * I, H), dtype=torch.float32)
    d = torch.zeros((1, H, I), dtype=torch.float32)
    g[0, 0, :32] = torch.tensor([6, 2.5, 3.5, 5, 0.25, 0.75, 1.25, 1.75, -2.5, -5, 0, 1, 2, 3, 4, -6.] * 2)
    g[0, 1, :32] = 1e-42                                  # subnormal amax: the clamp at -127
    g[0, 2, 32:64] = torch.linspace(-3e30, 3e30, 32)      # large exponents
    g[0, 3, :32] = 7.0                                    # saturation after the shared exponent
    d[0, 5, :] = torch.linspace(-1e-3, 1e-3, 32)
    rb = ft.ft_record_bytes(H, I, "mxfp4")
    out = torch.empty(rb, dtype=torch.uint8, device="cuda")
    ft.ft_quantize_experts(g.cuda(), d.cuda(), 1, H, I, out, fmt="mxfp4")
    assert np.array_equal(out.cpu().numpy(), encode_record(g[0].numpy(), d[0].numpy(), "mxfp4"))


def _check_call(wl, ref, t, l):
    r = ref.decode(l, wl.trace[t, l])
    assert wl.route_slot[t, l].cpu().numpy().tolist() == r.route_slot.tolist(), (t, l)
    assert wl.deferred[t, l].cpu().numpy().tolist() == r.deferred.tolist(), (t, l)
    assert wl.counters[t, l].cpu().numpy().tolist() == [r.n_hit, r.m, r.q, r.n_def_routes], (t, l)
    return r


@pytest.mark.parametrize("mode", ["full", "qstar"])
def test_mx_decode_tiny_every_call(ft, wl_mod, mode):
    from dataclasses import replace
    s = replace(wl_mod.SHAPES["tiny"], shared=True)
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I, fmt="mxfp4")
    shared = wl_mod.build_shared(0, s.L, s.H, s.I, fmt="mxfp4")
    split = wl_mod.split_tuple(mode, 32768)
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr, shared=shared, split=split,
                           fmt="mxfp4")
    wl = wl_mod.DecodeWorkload(s, seed=0)
    ref = SlotCache(s.L, s.E, s.C, full_offload=(mode == "full"), f_q16=32768)
    experts = oracle_experts(0, s.H, s.I, "mxfp4")
    for t in range(wl.steps):
        for l in range(s.L):
            wl.run_layer(cache, t, l)
            r = _check_call(wl, ref, t, l)
            x = wl.x[t, l].float().cpu().numpy()
            sh = oracle_shared(0, l, s.H, s.I, "mxfp4")
            y_ref = decode_layer(x, wl.trace[t, l], wl.gates[t, l], l, s.E, experts, sh)
            y_cpu = decode_layer(x, wl.trace[t, l], wl.gates[t, l], l, s.E, experts,
                                 include=r.deferred >= 0)
            assert_close(wl.y[t, l].cpu().numpy() + y_cpu, y_ref, f"step {t} layer {l}")
    for a, b in zip(ft.ft_cache_snapshot(cache.handle, s.L, s.E), ref.snapshot()):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
    pool.free()


def test_mx_decode_dsv4_shaped(ft, wl_mod):
    """DeepSeek-V4-Flash-shaped layers (256 experts, H 4096, I 2048, top-6; 4 of the 16
    layers) from an MXFP4 pool, 1024 slots, batch 4, q* with f = 1/2: state on every
    call, outputs on sampled tokens."""
    from dataclasses import replace
    s = replace(wl_mod.SHAPES["dsv4_decode"], L=4, B=4)
    steps = 12
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I, fmt="mxfp4")
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr,
                           split=wl_mod.split_tuple("qstar", 32768), fmt="mxfp4")
    wl = wl_mod.DecodeWorkload(s, seed=2, steps=steps)
    for t in range(steps):
        wl.run_step(cache, t)
    torch.cuda.synchronize()
    ref = SlotCache(s.L, s.E, s.C, full_offload=False, f_q16=32768)
    experts = oracle_experts(0, s.H, s.I, "mxfp4")
    for t in range(steps):
        for l in range(s.L):
            r = _check_call(wl, ref, t, l)
            if (t, l) in ((0, 0), (steps - 1, s.L - 1)):
                b = 3 if t else 0
                x = wl.x[t, l, b:b + 1].float().cpu().numpy()
                ids, g = wl.trace[t, l, b:b + 1], wl.gates[t, l, b:b + 1]
                y_ref = decode_layer(x, ids, g, l, s.E, experts)
                y_cpu = decode_layer(x, ids, g, l, s.E, experts, include=r.deferred[b:b + 1] >= 0)
                assert_close(wl.y[t, l, b:b + 1].cpu().numpy() + y_cpu, y_ref, f"step {t} layer {l}")
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
    pool.free()


def _prefill_mx(ft, wl_mod, scale, db, C):
    L, E, H, I, k, T = 2, 8, 256, 256, 4, 160
    seed = 9
    pool = wl_mod.build_pool(seed, L, E, H, I, fmt="mxfp4")
    if scale != 1.0:                                    # re-quantise with scaled weights
        rb = ft.ft_record_bytes(H, I, "mxfp4")
        host = pool.tensor()
        for f in range(L * E):
            a, b = synth.expert_weights(seed, f, H, I, "cuda")
            out = torch.empty(rb, dtype=torch.uint8, device="cuda")
            ft.ft_quantize_experts((a * scale).contiguous(), (b * scale).contiguous(), 1, H, I, out, fmt="mxfp4")
            host[f * rb:(f + 1) * rb].copy_(out.cpu())
    cache = ft.ExpertCache(L, E, H, I, k, 1, C, pool.ptr, T_max=T, fmt="mxfp4")
    ref = SlotCache(L, E, C)
    experts = oracle_experts(seed, H, I, "mxfp4", scale)
    R = T * k
    dbg = torch.empty(R * (I // 2 + I // 16), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, H), device="cuda")
    statuses = []
    for l in range(L):
        x = synth.prefill_x(seed, l, T, H, "cuda")
        ids, gates = synth.prefill_routes(seed, l, T, E, k, "cuda")
        ft.ft_moe_prefill_layer(cache.handle, l, x, ids, gates, T, k, y,
                                ft.FT_PREFILL_DOUBLE_BUFFER if db else 0, dbg)
        torch.cuda.synchronize()
        statuses.append(ft.ft_cache_status(cache.handle))
        ref.prefill(l, db) if C >= (2 if db else 1) * E else ref.prefill_on_demand(l, ids.cpu().numpy())
        for a_, b_ in zip(ft.ft_cache_snapshot(cache.handle, L, E), ref.snapshot()):
            assert np.array_equal(np.asarray(a_), np.asarray(b_)), f"layer {l}"
        xn, idn, gn = x.float().cpu().numpy(), ids.cpu().numpy(), gates.cpu().numpy()
        y_or, oc, os_ = prefill_layer(xn, idn, gn, l, E, experts)
        d = dbg.cpu().numpy()
        codes = d[: R * I // 2].reshape(R, I // 2)
        gc = np.empty((R, I), np.uint8)
        gc[:, 0::2] = codes & 0xF
        gc[:, 1::2] = codes >> 4
        gs = d[R * I // 2:].reshape(R, I // 16)
        assert (gc != oc).mean() <= 1e-4 and (gs != os_).mean() <= 1e-4, f"h flips, layer {l}"
        assert_close(y.cpu().numpy(), prefill_from_h(gc, gs, idn, gn, l, E, experts), f"stage 2, layer {l}")
        assert_close(y.cpu().numpy(), y_or, f"end to end, layer {l}")
    cache.close()
    pool.free()
    return statuses


@pytest.mark.parametrize("db,C", [(True, 16), (False, 8), (True, 5)])
def test_mx_prefill(ft, wl_mod, db, C):
    """Double-buffered, single-buffered and on-demand (5 slots) prefill of MXFP4
    experts whose E8M0 scales all have exact UE4M3 twins: no range flag."""
    assert _prefill_mx(ft, wl_mod, 1.0, db, C) == [0, 0]


def test_mx_prefill_flags_scales_outside_the_ue4m3_range(ft, wl_mod):
    """Weights scaled by 2^20 give E8M0 exponents above 2^8: the prefill GEMM cannot
    take them exactly and says so in the status word (decode reads them exactly)."""
    L, E, H, I, k, T, C = 1, 8, 256, 256, 2, 32, 16
    pool = wl_mod.build_pool(10, L, E, H, I, fmt="mxfp4")
    rb = ft.ft_record_bytes(H, I, "mxfp4")
    host = pool.tensor()
    for f in range(L * E):
        a, b = synth.expert_weights(10, f, H, I, "cuda")
        out = torch.empty(rb, dtype=torch.uint8, device="cuda")
        ft.ft_quantize_experts((a * 2.0 ** 20).contiguous(), (b * 2.0 ** 20).contiguous(), 1, H, I, out,
                               fmt="mxfp4")
        host[f * rb:(f + 1) * rb].copy_(out.cpu())
    cache = ft.ExpertCache(L, E, H, I, k, 1, C, pool.ptr, T_max=T, fmt="mxfp4")
    x = synth.prefill_x(10, 0, T, H, "cuda")
    ids, gates = synth.prefill_routes(10, 0, T, E, k, "cuda")
    y = torch.empty((T, H), device="cuda")
    ft.ft_moe_prefill_layer(cache.handle, 0, x, ids, gates, T, k, y, 0)
    assert ft.ft_cache_status(cache.handle) & ft.FT_DEV_SCALE_RANGE
    # decode of the same records is exact consumption: in tolerance of the oracle
    experts = oracle_experts(10, H, I, "mxfp4", 2.0 ** 20)
    ids_d = torch.tensor([[1, 6]], dtype=torch.int32, device="cuda")
    w = torch.tensor([[0.25, 0.75]], device="cuda")
    xd = synth.decode_x(10, 0, 0, L, 1, H, "cuda")
    yd = torch.empty((1, H), device="cuda")
    dd = torch.empty((1, 2), dtype=torch.int32, device="cuda")
    ft.ft_moe_decode(cache.handle, 0, xd, ids_d, w, 1, 2, yd, dd)
    y_ref = decode_layer(xd.float().cpu().numpy(), ids_d.cpu().numpy(), w.cpu().numpy(), 0, E, experts)
    assert_close(yd.cpu().numpy(), y_ref, "decode of out-of-range MXFP4 scales")
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
    pool.free()
