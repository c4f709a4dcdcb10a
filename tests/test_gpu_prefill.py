"""GPU parity of prefill (full-layer double buffering + tcgen05 FP4 grouped GEMMs)
through the C ABI against the CPU oracle.

Stage 1: the GPU's NVFP4 h (per route) equals the oracle's except for rare flips at
rounding boundaries (h differs in fp32 accumulation order), each one code step or
one E4M3 scale step.  Stage 2: y equals the oracle's GEMM2 + combine computed from
the GPU's own h, within rel-L2 5e-3 and max-abs 2e-2 * rms.  Slot tables after each
layer call are bit-exact with the oracle's prefill state.
"""
import numpy as np
import pytest
import torch

import synth
from oracle.formats import e2m1_decode, e4m3_decode
from oracle.lru import SlotCache
from oracle.moe import prefill_from_h, prefill_layer
from parity import assert_close, oracle_experts

pytestmark = pytest.mark.gpu

MAX_FLIP_FRACTION = 1e-3


@pytest.fixture(scope="module")
def ft():
    import __graft_entry__ as entry
    entry.build()
    import expert_cache_gb300
    return expert_cache_gb300


def _split_debug(dbg, R, I):
    codes = dbg[: R * I // 2].reshape(R, I // 2)
    scales = dbg[R * I // 2: R * I // 2 + R * I // 16].reshape(R, I // 16)
    c = np.empty((R, I), np.uint8)
    c[:, 0::2] = codes & 0xF
    c[:, 1::2] = codes >> 4
    return c, scales


def _check_h(gc, gs, oc, os_, valid_rows):
    gc, gs, oc, os_ = gc[valid_rows], gs[valid_rows], oc[valid_rows], os_[valid_rows]
    sdiff = gs != os_
    if sdiff.any():
        step = np.abs(gs.astype(int) - os_.astype(int))
        assert step[sdiff].max() <= 1, "scale differs by more than one E4M3 step"
    assert sdiff.mean() <= MAX_FLIP_FRACTION, f"scale flips {sdiff.mean():.2e}"
    blk_same = np.repeat(~sdiff, 16, axis=1)
    cdiff = (gc != oc) & blk_same
    if cdiff.any():
        mag_g = np.abs(e2m1_decode(gc[cdiff]))
        mag_o = np.abs(e2m1_decode(oc[cdiff]))
        grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
        ig = np.searchsorted(grid, mag_g)
        io = np.searchsorted(grid, mag_o)
        assert np.abs(ig - io).max() <= 1, "code differs by more than one step"
    assert cdiff.mean() <= MAX_FLIP_FRACTION, f"code flips {cdiff.mean():.2e}"


def _run_chunk(ft, wl_mod, L, E, H, I, k, T, C, db, seed, check_state=True, layers=None):
    pool = wl_mod.build_pool(seed, L, E, H, I)
    cache = ft.ExpertCache(L, E, H, I, k, 1, C, pool.ptr, T_max=T)
    ref = SlotCache(L, E, C)
    experts = oracle_experts(seed, H, I)
    flags = ft.FT_PREFILL_DOUBLE_BUFFER if db else 0
    R = T * k
    dbg = torch.empty(R * (I // 2 + I // 16), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    for l in range(L):
        x = synth.prefill_x(seed, l, T, H, "cuda")
        ids, gates = synth.prefill_routes(seed, l, T, E, k, "cuda")
        ft.ft_moe_prefill_layer(cache.handle, l, x, ids, gates, T, k, y, flags, dbg)
        torch.cuda.synchronize()
        assert ft.ft_cache_status(cache.handle) == 0
        ref.prefill(l, db)
        if check_state:
            for a_, b_ in zip(ft.ft_cache_snapshot(cache.handle, L, E), ref.snapshot()):
                assert np.array_equal(np.asarray(a_), np.asarray(b_)), f"layer {l}"
        if layers is not None and l not in layers:
            continue
        xn, idn, gn = x.float().cpu().numpy(), ids.cpu().numpy(), gates.cpu().numpy()
        y_or, oc, os_ = prefill_layer(xn, idn, gn, l, E, experts)
        gc, gs = _split_debug(dbg.cpu().numpy(), R, I)
        _check_h(gc, gs, oc, os_, np.ones(R, bool))
        y_gpu = y.cpu().numpy()
        assert_close(y_gpu, prefill_from_h(gc, gs, idn, gn, l, E, experts), f"stage 2, layer {l}")
        assert_close(y_gpu, y_or, f"end to end, layer {l}")
    cache.close()
    pool.free()


@pytest.fixture(scope="module")
def wl_mod(ft):
    from expert_cache_gb300 import workloads
    return workloads


@pytest.mark.parametrize("db", [True, False])
def test_prefill_small_ragged(ft, wl_mod, db):
    # 200 tokens x top-4 over 8 experts: ~100 rows per expert, ragged 128-row tiles
    _run_chunk(ft, wl_mod, L=3, E=8, H=256, I=256, k=4, T=200, C=16 if db else 8, db=db, seed=3)


def test_prefill_wider_shapes(ft, wl_mod):
    # several N and K tiles per expert (H 1024 -> 4 GEMM2 tiles, I 512 -> 4 GEMM1 tiles)
    _run_chunk(ft, wl_mod, L=2, E=16, H=1024, I=512, k=4, T=300, C=40, db=True, seed=4)


def test_prefill_capacity_errors(ft, wl_mod):
    L, E, H, I, k, T = 2, 8, 256, 256, 2, 16
    pool = wl_mod.build_pool(5, L, E, H, I)
    cache = ft.ExpertCache(L, E, H, I, k, 1, 12, pool.ptr, T_max=T)
    x = synth.prefill_x(5, 0, T, H, "cuda")
    ids, gates = synth.prefill_routes(5, 0, T, E, k, "cuda")
    y = torch.empty((T, H), device="cuda")
    with pytest.raises(ft.FtError) as ei:
        ft.ft_moe_prefill_layer(cache.handle, 0, x, ids, gates, T, k, y, ft.FT_PREFILL_DOUBLE_BUFFER)
    assert ei.value.status == ft.FT_ERR_CAPACITY
    with pytest.raises(ft.FtError) as ei:
        ft.ft_moe_prefill_layer(cache.handle, 0, x, ids, gates, T + 1, k, y, 0)
    assert ei.value.status == ft.FT_ERR_ARG
    cache.close()
    pool.free()


def test_prefill_then_decode_hands_over_the_buffers(ft, wl_mod):
    """After a chunk the buffers hold layers L-2 and L-1; decode starts from them."""
    L, E, H, I, k, T, C = 3, 8, 256, 256, 2, 64, 20
    pool = wl_mod.build_pool(6, L, E, H, I)
    cache = ft.ExpertCache(L, E, H, I, k, 1, C, pool.ptr, T_max=T)
    ref = SlotCache(L, E, C)
    y = torch.empty((T, H), device="cuda")
    for l in range(L):
        x = synth.prefill_x(6, l, T, H, "cuda")
        ids, gates = synth.prefill_routes(6, l, T, E, k, "cuda")
        ft.ft_moe_prefill_layer(cache.handle, l, x, ids, gates, T, k, y)
        ref.prefill(l, True)
    ids = torch.tensor([[1, 5]], dtype=torch.int32, device="cuda")
    w = torch.tensor([[0.5, 0.5]], device="cuda")
    xd = synth.decode_x(6, 0, L - 1, L, 1, H, "cuda")
    yd = torch.empty((1, H), device="cuda")
    d = torch.empty((1, 2), dtype=torch.int32, device="cuda")
    ct = torch.empty(4, dtype=torch.int32, device="cuda")
    ft.ft_moe_decode(cache.handle, L - 1, xd, ids, w, 1, 2, yd, d, None, ct)
    r = ref.decode(L - 1, ids.cpu().numpy())
    assert ct.cpu().tolist() == [r.n_hit, r.m, r.q, r.n_def_routes] == [2, 0, 0, 0]
    for a_, b_ in zip(ft.ft_cache_snapshot(cache.handle, L, E), ref.snapshot()):
        assert np.array_equal(np.asarray(a_), np.asarray(b_))
    cache.close()
    pool.free()


def test_prefill_qwen_shaped_full_size_sampled(ft, wl_mod):
    """8192 tokens x top-8 over 256 experts (H 2048, I 512), two layers with the double
    buffer in the launch configuration the benchmark times; outputs of sampled tokens
    against the oracle (tokens are independent through the quantisers)."""
    from expert_cache_gb300.workloads import SHAPES
    s = SHAPES["qwen_prefill"]
    L, T = 2, s.T
    pool = wl_mod.build_pool(0, L, s.E, s.H, s.I)
    cache = ft.ExpertCache(L, s.E, s.H, s.I, s.k, 1, s.C, pool.ptr, T_max=T)
    experts = oracle_experts(0, s.H, s.I)
    y = torch.empty((T, s.H), device="cuda")
    rows = np.array([0, 1, 777, 4095, 5000, T - 1])
    for l in range(L):
        x = synth.prefill_x(0, l, T, s.H, "cuda")
        ids, gates = synth.prefill_routes(0, l, T, s.E, s.k, "cuda")
        ft.ft_moe_prefill_layer(cache.handle, l, x, ids, gates, T, s.k, y)
        torch.cuda.synchronize()
        assert ft.ft_cache_status(cache.handle) == 0
        xn = x.float().cpu().numpy()[rows]
        y_or, _, _ = prefill_layer(xn, ids.cpu().numpy()[rows], gates.cpu().numpy()[rows], l, s.E, experts)
        assert_close(y.cpu().numpy()[rows], y_or, f"layer {l}")
    cache.close()
    pool.free()
