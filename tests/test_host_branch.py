"""The host share of decode (the CPU branch) against the oracle, on the CPU: the
branch's workers compute the deferred routes from a pool of records in host memory;
their partial must equal the oracle's decode_layer restricted to those routes.  Also
the backend choice of the bandwidth profile against the oracle's rule, and the branch's
argument checks.  (The GPU-side hand-off, the join and the profile itself run in
test_gpu_host_branch.py.)"""
import numpy as np
import pytest

import synth
from oracle.formats import encode_record, record_layout
from oracle.moe import decode_layer
from oracle.qrule import recommend_backend, split_from_overlap
from tests.parity import assert_close, oracle_experts


@pytest.fixture(scope="module")
def ft():
    import expert_cache_gb300 as m
    return m


def _pool(seed, L, E, H, I, fmt="nvfp4", flats=None):
    """Records of the oracle's quantiser in one host array (only `flats` filled)."""
    rb = record_layout(H, I, fmt)["bytes"]
    pool = np.zeros(L * E * rb, np.uint8)
    for f in (range(L * E) if flats is None else flats):
        w_gu, w_d = synth.expert_weights(seed, f, H, I, "cpu")
        pool[f * rb:(f + 1) * rb] = encode_record(w_gu.numpy(), w_d.numpy(), fmt)
    return pool


def _bf16_bits(x):
    """bf16 bit patterns (uint16) of float32 values that are already bf16-exact."""
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _case(seed, B, k, L, E, layer, H):
    rng = np.random.default_rng(seed)
    x = synth.decode_x(seed, 0, layer, L, B, H, "cpu").float().numpy()
    ids = rng.integers(0, E, size=(B, k)).astype(np.int32)
    w = rng.random((B, k)).astype(np.float32)
    host = rng.random((B, k)) < 0.6                       # the routes left to the host
    deferred = np.where(host, layer * E + ids, -1).astype(np.int32)
    return x, ids, w, host, deferred


def _host_partial(ft, pool, L, E, H, I, x, deferred, w, B, k, n_threads, fmt="nvfp4"):
    hb = ft.HostBranch(L, E, H, I, k, max(B, 1), pool.ctypes.data, n_threads, fmt=fmt, mailbox=False)
    try:
        y = np.full((B, H), np.nan, np.float32)
        ft.ft_host_moe(hb.handle, _bf16_bits(x), deferred, w, B, k, y)
        return y
    finally:
        hb.close()


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_host_share_matches_oracle_tiny(ft, fmt):
    """B = 3 tokens, k = 4, about 60 % of the routes on the host, repeated experts
    within and across tokens: the partial equals the oracle's, in fp32 accuracy."""
    L, E, H, I, k, B, layer, seed = 2, 16, 64, 32, 4, 3, 1, 5
    pool = _pool(seed, L, E, H, I, fmt)
    x, ids, w, host, deferred = _case(seed, B, k, L, E, layer, H)
    ids[1, 2] = ids[1, 0]                                 # a token that lists an expert twice
    deferred = np.where(host, layer * E + ids, -1).astype(np.int32)
    deferred[1, 0] = layer * E + ids[1, 0]
    deferred[1, 2] = layer * E + ids[1, 2]
    y = _host_partial(ft, pool, L, E, H, I, x, deferred, w, B, k, 4, fmt)
    y_ref = decode_layer(x, ids, w, layer, E, oracle_experts(seed, H, I, fmt), include=deferred >= 0)
    assert_close(y, y_ref, "host share")
    rel = np.linalg.norm(y - y_ref) / np.linalg.norm(y_ref)
    assert rel < 1e-5, rel                                 # fp32 sums of exact products


def test_host_share_no_routes_is_zero(ft):
    L, E, H, I, k, B = 1, 8, 64, 32, 2, 2
    pool = _pool(1, L, E, H, I)
    x = synth.decode_x(1, 0, 0, L, B, H, "cpu").float().numpy()
    y = _host_partial(ft, pool, L, E, H, I, x, np.full((B, k), -1, np.int32), np.ones((B, k), np.float32),
                      B, k, 2)
    assert np.all(y == 0.0)


def test_host_share_deterministic_over_thread_counts(ft):
    """Every row is computed by one worker in a fixed order, so 1, 3 and 8 workers give
    the same bits."""
    L, E, H, I, k, B, layer, seed = 2, 16, 128, 64, 4, 2, 0, 9
    pool = _pool(seed, L, E, H, I)
    x, ids, w, host, deferred = _case(seed, B, k, L, E, layer, H)
    ys = [_host_partial(ft, pool, L, E, H, I, x, deferred, w, B, k, n) for n in (1, 3, 8)]
    assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])


def test_host_share_qwen_shape(ft):
    """The benchmark's layer shape (H 2048, I 512): two host experts, one token."""
    L, E, H, I, k, B, layer, seed = 1, 8, 2048, 512, 8, 1, 0, 3
    ids = np.array([[0, 1, 2, 3, 4, 5, 6, 7]], np.int32)
    deferred = np.full((1, k), -1, np.int32)
    deferred[0, 2], deferred[0, 5] = 2, 5
    pool = _pool(seed, L, E, H, I, flats=(2, 5))
    x = synth.decode_x(seed, 0, 0, L, B, H, "cpu").float().numpy()
    w = np.linspace(0.1, 0.8, k, dtype=np.float32)[None]
    y = _host_partial(ft, pool, L, E, H, I, x, deferred, w, B, k, 4)
    y_ref = decode_layer(x, ids, w, layer, E, oracle_experts(seed, H, I), include=deferred >= 0)
    assert_close(y, y_ref, "host share at H 2048, I 512")


def test_host_branch_argument_errors(ft):
    L, E, H, I = 1, 8, 64, 32
    pool = _pool(1, L, E, H, I)
    bad = dict(L=L, E=E, H=96, I=I)
    with pytest.raises(ft.FtError):
        ft.HostBranch(bad["L"], bad["E"], bad["H"], bad["I"], 2, 1, pool.ctypes.data, 2, mailbox=False)
    with pytest.raises(ft.FtError):
        ft.HostBranch(L, E, H, I, 2, 1, pool.ctypes.data, 0, mailbox=False)
    hb = ft.HostBranch(L, E, H, I, 2, 1, pool.ctypes.data, 2, mailbox=False)
    try:
        x = np.zeros((2, H), np.uint16)
        d = np.full((2, 2), -1, np.int32)
        w = np.ones((2, 2), np.float32)
        y = np.zeros((2, H), np.float32)
        with pytest.raises(ft.FtError):                   # B above B_max
            ft.ft_host_moe(hb.handle, x, d, w, 2, 2, y)
        with pytest.raises(ft.FtError):                   # k above k_max
            ft.ft_host_moe(hb.handle, x, np.full((1, 3), -1, np.int32), np.ones((1, 3), np.float32), 1, 3, y)
        assert ft.ft_host_branch_stats(hb.handle) == (0, 0)
        ft.ft_host_moe(hb.handle, x[:1], d[:1], w[:1], 1, 2, y)
        assert ft.ft_host_branch_stats(hb.handle) == (1, 0)
    finally:
        hb.close()
    assert ft.ft_host_mailbox_bytes(2048, 8, 1) > 2048 * 6
    with pytest.raises(ft.FtError):
        ft.ft_host_mailbox_bytes(2048, 0, 1)


def test_recommend_rule_pins():
    """[BWRATIO "第一层带宽比"]: hybrid iff cpu > 2 x pcie; exactly 2 x stays offload."""
    assert recommend_backend(100.0, 49.9) == "hybrid"
    assert recommend_backend(100.0, 50.0) == "offload"
    assert recommend_backend(100.0, 211.0) == "offload"
    assert recommend_backend(1.0, 0.0) == "hybrid"


def test_recommend_and_overlap_split_match_the_library(ft):
    rng = np.random.default_rng(0)
    for _ in range(200):
        cpu, pcie = rng.uniform(1, 500, size=2)
        want = ft.FT_BACKEND_HYBRID if recommend_backend(cpu, pcie) == "hybrid" else ft.FT_BACKEND_OFFLOAD
        assert ft.ft_recommend_backend(cpu, pcie) == want
        assert ft.ft_split_from_overlap(pcie, cpu) == split_from_overlap(pcie, cpu)
    assert ft.ft_recommend_backend(100.0, 50.0) == ft.FT_BACKEND_OFFLOAD


def test_host_share_large_activations(ft):
    """x scaled by 2^20 (beyond the f16 range): the per-token power-of-two prescale keeps
    the f16 copy of x exact, so the partial still matches the oracle in fp32 accuracy."""
    L, E, H, I, k, B, layer, seed = 1, 8, 64, 32, 2, 2, 0, 4
    pool = _pool(seed, L, E, H, I)
    x = synth.decode_x(seed, 0, 0, L, B, H, "cpu").float().numpy() * np.float32(2.0 ** 20)
    ids = np.array([[1, 5], [5, 2]], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5]], np.float32)
    deferred = ids.astype(np.int32).copy()
    y = _host_partial(ft, pool, L, E, H, I, x, deferred, w, B, k, 2)
    with np.errstate(over="ignore"):                     # silu of large negative g: e^-g -> inf, silu -> 0
        y_ref = decode_layer(x, ids, w, layer, E, oracle_experts(seed, H, I), include=deferred >= 0)
    rel = np.linalg.norm(y - y_ref) / np.linalg.norm(y_ref)
    assert rel < 1e-5, rel
