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
from oracle.formats import e2m1_decode, e2m1_encode, e4m3_decode
from oracle.lru import SlotCache
from oracle.moe import prefill_from_h, prefill_layer
from parity import assert_close, oracle_experts

pytestmark = pytest.mark.gpu

# Boundary flips (GPU and oracle h differ in fp32 accumulation order and in the
# rounding of silu): at most this fraction of the h codes, and of the h scales.
MAX_FLIP_FRACTION = 1e-4
# A code may differ from the oracle's only where the oracle's v/s lies within this
# relative distance of an E2M1 rounding midpoint; a scale only where the oracle's
# amax/6 lies within it of an E4M3 midpoint.
MIDPOINT_REL = 1e-5

_GRID = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
_MIDS = (_GRID[1:] + _GRID[:-1]) / 2


@pytest.fixture(scope="module")
def ft():
    import __graft_entry__ as entry
    entry.build()
    import expert_cache_gb300
    return expert_cache_gb300


def _unpack(packed, n):
    c = np.empty((packed.shape[0], n), np.uint8)
    c[:, 0::2] = packed & 0xF
    c[:, 1::2] = packed >> 4
    return c


def _split_debug(dbg, R, I, H=None):
    """h codes [R, I] and scales [R, I/16] by route; with H also the debug-x part:
    (route_pos [R], x codes packed [R, H/2], x scales [R, H/16]) in sorted rows."""
    codes = dbg[: R * I // 2].reshape(R, I // 2)
    o = R * I // 2
    scales = dbg[o: o + R * I // 16].reshape(R, I // 16)
    out = [_unpack(codes, I), scales]
    if H is not None:
        o += R * I // 16
        pos = dbg[o: o + 4 * R].view(np.int32)
        o += 4 * R
        xc = dbg[o: o + R * H // 2].reshape(R, H // 2)
        o += R * H // 2
        xs = dbg[o: o + R * H // 16].reshape(R, H // 16)
        out += [pos, xc, xs]
    return out


def _debug_bytes(R, I, H, with_x):
    return R * (I // 2 + I // 16) + (R * (4 + H // 2 + H // 16) if with_x else 0)


def _near_midpoint(v, mids):
    a = np.abs(np.asarray(v, np.float64))
    d = np.min(np.abs(a[..., None] - mids), axis=-1)
    return d <= MIDPOINT_REL * a


def _check_h(gc, gs, oc, os_, h32, rows):
    """Stage 1: GPU h codes/scales equal the oracle's except legitimate boundary flips.
    Returns (code flips, scale flips, largest relative midpoint distance of a flip)."""
    gc, gs, oc, os_, h32 = gc[rows], gs[rows], oc[rows], os_[rows], h32[rows]
    n, I = gc.shape
    blocks = h32.reshape(n, I // 16, 16)
    e4m3_vals = e4m3_decode(np.arange(0x7F))
    worst = 0.0
    # scales: equal, or one E4M3 step where the oracle's amax/6 sits on a midpoint
    sdiff = gs != os_
    if sdiff.any():
        assert np.abs(gs.astype(int) - os_.astype(int))[sdiff].max() <= 1, "scale more than one step off"
        t = (np.max(np.abs(blocks), axis=2) / np.float32(6.0)).astype(np.float32)[sdiff]
        lo = np.minimum(gs, os_)[sdiff].astype(int)
        mid = (e4m3_vals[lo] + e4m3_vals[lo + 1]) / 2
        dist = np.abs(t - mid) / t
        assert np.all(dist <= MIDPOINT_REL), f"scale flip {dist.max():.2e} from an E4M3 midpoint"
        worst = max(worst, float(dist.max()))
    assert sdiff.mean() <= MAX_FLIP_FRACTION, f"scale flips {sdiff.mean():.2e}"
    # codes: against the oracle's h quantised with the scale the GPU used (the
    # oracle's own codes where the scales agree)
    s_used = e4m3_decode(gs).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        vs = (blocks / s_used[..., None]).astype(np.float32).reshape(n, I)
    vs = np.where(np.repeat(s_used, 16, axis=1) == 0, np.float32(0), vs)
    want = oc.copy()
    if sdiff.any():
        alt = e2m1_encode(vs)
        blk = np.repeat(sdiff, 16, axis=1)
        want[blk] = alt[blk]
    cdiff = gc != want
    if cdiff.any():
        mg = np.abs(e2m1_decode(gc[cdiff]))
        mo = np.abs(e2m1_decode(want[cdiff]))
        step = np.abs(np.searchsorted(_GRID, mg) - np.searchsorted(_GRID, mo))
        assert step.max() <= 1, "code more than one step off"
        v = vs[cdiff]
        neg = (gc[cdiff] & 8) != 0
        assert not np.any(neg & (v > 0)), "negative code for a positive h"
        assert np.all(_near_midpoint(v, _MIDS)), "code flip away from an E2M1 midpoint"
        a = np.abs(v.astype(np.float64))
        worst = max(worst, float((np.min(np.abs(a[:, None] - _MIDS), axis=1) / a).max()))
    assert cdiff.mean() <= MAX_FLIP_FRACTION, f"code flips {cdiff.mean():.2e}"
    return int(cdiff.sum()), int(sdiff.sum()), worst


def _check_x(x_f32, k, pos, xc_packed, xs, routes=None):
    """The GPU's quantised activations (sorted rows) equal the oracle quantiser's
    codes and scales of each route's token, bit for bit."""
    from oracle.formats import pack_nibbles, quantize_act
    R = pos.shape[0]
    r = np.arange(R) if routes is None else np.asarray(routes)
    r = r[pos[r] >= 0]
    t = r // k
    want_c, want_s = quantize_act(x_f32[np.unique(t)])
    row_of = {tt: i for i, tt in enumerate(np.unique(t).tolist())}
    idx = np.array([row_of[tt] for tt in t.tolist()])
    assert np.array_equal(xc_packed[pos[r]], pack_nibbles(want_c)[idx]), "x codes"
    assert np.array_equal(xs[pos[r]], want_s[idx]), "x scales"
    return len(r)


def _run_chunk(ft, wl_mod, L, E, H, I, k, T, C, db, seed, check_state=True, layers=None,
               on_demand=False, extra_flags=0):
    """One chunk through L layers; db: ask for the double buffer; on_demand: the
    oracle state follows the on-demand fallback (routed union through the LRU)."""
    pool = wl_mod.build_pool(seed, L, E, H, I)
    cache = ft.ExpertCache(L, E, H, I, k, 1, C, pool.ptr, T_max=T)
    ref = SlotCache(L, E, C)
    experts = oracle_experts(seed, H, I)
    flags = (ft.FT_PREFILL_DOUBLE_BUFFER if db else 0) | ft.FT_PREFILL_DEBUG_X | extra_flags
    R = T * k
    dbg = torch.empty(_debug_bytes(R, I, H, True), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    for l in range(L):
        x = synth.prefill_x(seed, l, T, H, "cuda")
        ids, gates = synth.prefill_routes(seed, l, T, E, k, "cuda")
        ft.ft_moe_prefill_layer(cache.handle, l, x, ids, gates, T, k, y, flags, dbg)
        torch.cuda.synchronize()
        assert ft.ft_cache_status(cache.handle) == 0
        if on_demand:
            ref.prefill_on_demand(l, ids.cpu().numpy())
        else:
            ref.prefill(l, db)
        if check_state:
            for a_, b_ in zip(ft.ft_cache_snapshot(cache.handle, L, E), ref.snapshot()):
                assert np.array_equal(np.asarray(a_), np.asarray(b_)), f"layer {l}"
        if layers is not None and l not in layers:
            continue
        xn, idn, gn = x.float().cpu().numpy(), ids.cpu().numpy(), gates.cpu().numpy()
        y_or, oc, os_, h32 = prefill_layer(xn, idn, gn, l, E, experts, return_h32=True)
        gc, gs, pos, xc, xs = _split_debug(dbg.cpu().numpy(), R, I, H)
        assert _check_x(xn, k, pos, xc, xs) == R
        _check_h(gc, gs, oc, os_, h32, np.ones(R, bool))
        y_gpu = y.cpu().numpy()
        assert_close(y_gpu, prefill_from_h(gc, gs, idn, gn, l, E, experts), f"stage 2, layer {l}")
        assert_close(y_gpu, y_or, f"end to end, layer {l}")
    # hand-off: decode continues from what prefill left resident
    if on_demand or check_state:
        rng = np.random.default_rng(seed)
        for call in range(6):
            l = call % L
            ids_d = np.stack([rng.choice(E, k, replace=False)]).astype(np.int32)
            xd = synth.decode_x(seed, call, l, L, 1, H, "cuda")
            yd = torch.empty((1, H), device="cuda")
            dd = torch.empty((1, k), dtype=torch.int32, device="cuda")
            ct = torch.empty(4, dtype=torch.int32, device="cuda")
            ft.ft_moe_decode(cache.handle, l, xd, torch.from_numpy(ids_d).cuda(),
                             torch.full((1, k), 1.0 / k, device="cuda"), 1, k, yd, dd, None, ct)
            r = ref.decode(l, ids_d)
            assert ct.cpu().tolist() == [r.n_hit, r.m, r.q, r.n_def_routes], f"decode call {call}"
        for a_, b_ in zip(ft.ft_cache_snapshot(cache.handle, L, E), ref.snapshot()):
            assert np.array_equal(np.asarray(a_), np.asarray(b_)), "tables after the hand-off"
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


def test_prefill_argument_errors(ft, wl_mod):
    L, E, H, I, k, T = 2, 8, 256, 256, 2, 16
    pool = wl_mod.build_pool(5, L, E, H, I)
    cache = ft.ExpertCache(L, E, H, I, k, 1, 12, pool.ptr, T_max=T)
    x = synth.prefill_x(5, 0, T, H, "cuda")
    ids, gates = synth.prefill_routes(5, 0, T, E, k, "cuda")
    y = torch.empty((T, H), device="cuda")
    for bad in (dict(T=T + 1), dict(flags=64), dict(layer=L), dict(k=k + 1)):
        kw = dict(layer=0, T=T, k=k, flags=0)
        kw.update(bad)
        with pytest.raises(ft.FtError) as ei:
            ft.ft_moe_prefill_layer(cache.handle, kw["layer"], x, ids, gates, kw["T"], kw["k"], y,
                                    kw["flags"])
        assert ei.value.status == ft.FT_ERR_ARG, bad
    cache.close()
    pool.free()


@pytest.mark.parametrize("C,flags", [(6, 0), (12, 1), (20, 1), (40, 4)])
def test_prefill_on_demand_fallback(ft, wl_mod, C, flags):
    """Capacity below two layers (with the double buffer asked for) or below one
    layer: the call falls back to the routed union on demand; C = 6 takes three
    groups per layer, 12 two, 20 one; C = 40 asks for the on-demand path directly.
    Tables after every layer, x, h and y as in the whole-layer path, then decode
    from what the prefill left resident."""
    _run_chunk(ft, wl_mod, L=3, E=16, H=256, I=256, k=4, T=200, C=C,
               db=bool(flags & 1), seed=7, on_demand=True, extra_flags=flags & 4)


def test_prefill_on_demand_sparse_union(ft, wl_mod):
    """A short chunk routes to few experts: only the union is loaded (hits from the
    previous layers' calls stay), one group."""
    _run_chunk(ft, wl_mod, L=4, E=64, H=256, I=256, k=2, T=5, C=24, db=False, seed=8,
               on_demand=True, extra_flags=4)


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


def test_prefill_x_quantisation_ties(ft, wl_mod):
    """The activation quantiser of the prefill path against the oracle's, bit for bit,
    on blocks built to land on rounding ties: E2M1 midpoints (v/s = .25, .75, 1.25,
    1.75, 2.5, 3.5, 5), an E4M3 scale midpoint (amax/6 = 1.0625, between 1 and 1.125),
    a subnormal scale midpoint (amax/6 = 2.5 * 2^-9), saturation, zero blocks and
    signed zeros, plus random rows."""
    L, E, H, I, k, T, C = 1, 8, 256, 256, 2, 64, 8
    x = synth.prefill_x(21, 0, T, H, "cpu").float().numpy()
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    x[0, :16] = [6.0] + mids + [-m for m in mids] + [0.0]          # s = 1, every tie
    x[1, :16] = [6.375] + [0.0] * 15                                # amax/6 = 1.0625: tie
    x[1, 16:32] = [6.0 * 2.5 * 2.0 ** -9] + [2.0 ** -9] * 15        # subnormal scale tie
    x[2, :16] = [-0.0] * 16                                         # zero block, signed zeros
    x[2, 16:32] = [3.0, -0.0] + [2.0 ** -20] * 14                    # tiny values round to +0
    x[3, :16] = [7.0] + [6.875] * 15                                # amax/6 rounds down: saturate
    for r in range(4, 12):                                          # ties at other scales
        s_ = 2.0 ** (r - 8)
        x[r, :16] = [6.0 * s_] + [m * s_ for m in mids] + [-m * s_ for m in mids] + [s_]
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(xb.float(), torch.from_numpy(x)), "tie values must be exact in bf16"
    pool = wl_mod.build_pool(21, L, E, H, I)
    cache = ft.ExpertCache(L, E, H, I, k, 1, C, pool.ptr, T_max=T)
    ids, gates = synth.prefill_routes(21, 0, T, E, k, "cuda")
    ids[5, 1] = E + 3                                               # one masked route
    R = T * k
    dbg = torch.empty(_debug_bytes(R, I, H, True), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ft.ft_moe_prefill_layer(cache.handle, 0, xb.cuda(), ids, gates, T, k, y, ft.FT_PREFILL_DEBUG_X, dbg)
    torch.cuda.synchronize()
    assert ft.ft_cache_status(cache.handle) == ft.FT_DEV_BAD_ID
    _, _, pos, xc, xs = _split_debug(dbg.cpu().numpy(), R, I, H)
    assert pos[5 * k + 1] == -1
    assert _check_x(xb.float().numpy(), k, pos, xc, xs) == R - 1
    cache.close()
    pool.free()


@pytest.fixture(scope="module")
def qwen_prefill_pool(wl_mod):
    from expert_cache_gb300.workloads import SHAPES
    s = SHAPES["qwen_prefill"]
    pool = wl_mod.build_pool(0, s.L, s.E, s.H, s.I)
    yield pool
    pool.free()


def test_prefill_qwen_shaped_full_chunk(ft, wl_mod, qwen_prefill_pool):
    """One 8192-token chunk through all 40 layers (256 experts, top-8, H 2048, I 512,
    600 slots) with the double buffer, in the launch configuration the benchmark
    times: slot tables bit-exact after every layer; on the first, a middle and the
    last layer the quantised x of every route bit-exact, and h (stage 1), y from the
    GPU's h (stage 2) and y end to end on sampled tokens (tokens are independent
    through the quantisers, so the oracle computes only those)."""
    from expert_cache_gb300.workloads import SHAPES
    s = SHAPES["qwen_prefill"]
    L, T, E, H, I, k = s.L, s.T, s.E, s.H, s.I, s.k
    cache = ft.ExpertCache(L, E, H, I, k, 1, s.C, qwen_prefill_pool.ptr, T_max=T)
    ref = SlotCache(L, E, s.C)
    experts = oracle_experts(0, H, I)
    R = T * k
    dbg = torch.empty(_debug_bytes(R, I, H, True), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, H), device="cuda")
    rows = np.array([0, 1, 777, 4095, 5000, T - 1])
    routes = (rows[:, None] * k + np.arange(k)).reshape(-1)
    checked = {0, L // 2, L - 1}
    flips = []
    for l in range(L):
        x = synth.prefill_x(0, l, T, H, "cuda")
        ids, gates = synth.prefill_routes(0, l, T, E, k, "cuda")
        flags = ft.FT_PREFILL_DOUBLE_BUFFER | (ft.FT_PREFILL_DEBUG_X if l in checked else 0)
        ft.ft_moe_prefill_layer(cache.handle, l, x, ids, gates, T, k, y, flags,
                                dbg if l in checked else None)
        ref.prefill(l, True)
        for a_, b_ in zip(ft.ft_cache_snapshot(cache.handle, L, E), ref.snapshot()):
            assert np.array_equal(np.asarray(a_), np.asarray(b_)), f"tables after layer {l}"
        assert ft.ft_cache_status(cache.handle) == 0
        if l not in checked:
            continue
        xn = x.float().cpu().numpy()
        idn, gn = ids.cpu().numpy(), gates.cpu().numpy()
        gc, gs, pos, xc, xs = _split_debug(dbg.cpu().numpy(), R, I, H)
        assert _check_x(xn, k, pos, xc, xs) == R
        y_or, oc, os_, h32 = prefill_layer(xn[rows], idn[rows], gn[rows], l, E, experts, return_h32=True)
        flips.append(_check_h(gc[routes], gs[routes], oc, os_, h32, np.ones(len(routes), bool)))
        y_rows = y.cpu().numpy()[rows]
        assert_close(y_rows, prefill_from_h(gc[routes], gs[routes], idn[rows], gn[rows], l, E, experts),
                     f"stage 2, layer {l}")
        assert_close(y_rows, y_or, f"end to end, layer {l}")
    # after the chunk the two buffers hold layers L-2 and L-1 (decode's first cache)
    sfi = ft.ft_cache_snapshot(cache.handle, L, E)[0].reshape(L, E)
    assert np.array_equal(sfi[L - 1], (L - 1) % 2 * E + np.arange(E))
    assert np.array_equal(sfi[L - 2], (L - 2) % 2 * E + np.arange(E))
    assert np.all(sfi[:L - 2] == -1)
    print("h flips (codes, scales, worst midpoint distance) per checked layer:", flips)
    cache.close()


def test_prefill_qwen_shaped_on_demand(ft, wl_mod, qwen_prefill_pool):
    """The Qwen-shaped 8192-token chunk with 200 slots (fewer than one layer's 256
    experts): every layer falls back to on-demand loading in two groups.  Tables
    after every layer; x, h and y on sampled tokens of two layers."""
    from expert_cache_gb300.workloads import SHAPES
    s = SHAPES["qwen_prefill"]
    L, T, E, H, I, k, C = 6, s.T, s.E, s.H, s.I, s.k, 200
    cache = ft.ExpertCache(L, E, H, I, k, 1, C, qwen_prefill_pool.ptr, T_max=T)
    ref = SlotCache(L, E, C)
    experts = oracle_experts(0, H, I)
    R = T * k
    dbg = torch.empty(_debug_bytes(R, I, H, True), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, H), device="cuda")
    rows = np.array([3, 2048, T - 2])
    routes = (rows[:, None] * k + np.arange(k)).reshape(-1)
    for l in range(L):
        x = synth.prefill_x(0, l, T, H, "cuda")
        ids, gates = synth.prefill_routes(0, l, T, E, k, "cuda")
        checked = l in (0, L - 1)
        flags = ft.FT_PREFILL_DOUBLE_BUFFER | (ft.FT_PREFILL_DEBUG_X if checked else 0)
        ft.ft_moe_prefill_layer(cache.handle, l, x, ids, gates, T, k, y, flags, dbg if checked else None)
        groups = ref.prefill_on_demand(l, ids.cpu().numpy())
        assert len(groups) == 2
        for a_, b_ in zip(ft.ft_cache_snapshot(cache.handle, L, E), ref.snapshot()):
            assert np.array_equal(np.asarray(a_), np.asarray(b_)), f"tables after layer {l}"
        assert ft.ft_cache_status(cache.handle) == 0
        if not checked:
            continue
        xn, idn, gn = x.float().cpu().numpy(), ids.cpu().numpy(), gates.cpu().numpy()
        gc, gs, pos, xc, xs = _split_debug(dbg.cpu().numpy(), R, I, H)
        assert _check_x(xn, k, pos, xc, xs, routes) == len(routes)
        y_or, oc, os_, h32 = prefill_layer(xn[rows], idn[rows], gn[rows], l, E, experts, return_h32=True)
        _check_h(gc[routes], gs[routes], oc, os_, h32, np.ones(len(routes), bool))
        y_rows = y.cpu().numpy()[rows]
        assert_close(y_rows, prefill_from_h(gc[routes], gs[routes], idn[rows], gn[rows], l, E, experts),
                     f"stage 2, layer {l}")
        assert_close(y_rows, y_or, f"end to end, layer {l}")
    cache.close()
