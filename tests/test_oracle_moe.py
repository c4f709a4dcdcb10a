"""Pins for oracle.moe: expert outputs, the exact GPU/CPU merge, prefill."""
import math

import numpy as np
import pytest

from oracle import formats as F
from oracle.lru import SlotCache
from oracle.moe import (RecordSource, decode_layer, decode_layer_dense, prefill_from_h,
                        prefill_layer)
from synth import decode_gates, expert_weights, locality_trace, prefill_routes, prefill_x

L, E, K, H, I = 2, 16, 2, 64, 32


@pytest.fixture(scope="module")
def tiny():
    recs = {f: F.encode_record(*[w.numpy() for w in expert_weights(0, f, H, I)])
            for f in range(L * E)}
    return RecordSource(lambda f: recs[f], H, I)


def _record_from_codes(gu_codes, d_codes):
    """Record with every block scale 1.0 (E4M3 0x38) and unit tensor scales."""
    two_i, h = gu_codes.shape
    i = two_i // 2
    lay = F.record_layout(h, i)
    rec = np.zeros(lay["bytes"], np.uint8)
    for name, arr in (("gu_codes", F.pack_nibbles(gu_codes)),
                      ("gu_scales", np.full((two_i, h // 16), 0x38, np.uint8)),
                      ("d_codes", F.pack_nibbles(d_codes)),
                      ("d_scales", np.full((h, i // 16), 0x38, np.uint8)),
                      ("s_gu", np.float32([1.0]).view(np.uint8)),
                      ("s_d", np.float32([1.0]).view(np.uint8))):
        off, size = lay[name]
        rec[off:off + size] = arr.reshape(-1)
    return rec


def test_swiglu_closed_form():
    # x = x0 * e_0; gate row i sees g_i * x0, up row i sees u_i * x0:
    # h_i = silu(g_i x0) * u_i x0 and o_r = sum_i D[r, i] h_i.
    hh = ii = 16
    enc = {v: c for c, v in enumerate(F.e2m1_decode(np.arange(16)).tolist()) if c != 8}
    gvals = [1.0, -2.0, 0.5, 3.0, -1.5, 4.0, 0.0, -6.0, 2.0, 1.5, -0.5, 6.0, -3.0, 1.0, -4.0, 0.5]
    uvals = [-1.0, 0.5, 2.0, -3.0, 6.0, -0.5, 1.5, 4.0, -2.0, 1.0, 3.0, -1.5, 0.5, -6.0, 2.0, -4.0]
    gu = np.zeros((2 * ii, hh), np.uint8)
    for i in range(ii):
        gu[i, 0] = enc[gvals[i]]
        gu[ii + i, 0] = enc[uvals[i]]
    dvals = np.array([[((r * 7 + i * 3) % 15) - 7 for i in range(ii)] for r in range(hh)], float)
    dvals = np.clip(dvals, -6, 6)
    dvals[np.isin(np.abs(dvals), [5.0])] = 4.0
    d = np.vectorize(lambda v: enc[float(v)])(dvals).astype(np.uint8)
    rec = _record_from_codes(gu, d)
    x0 = 0.75
    x = np.zeros((1, hh))
    x[0, 0] = x0
    src = RecordSource(lambda f: rec, hh, ii)
    y = decode_layer(x, np.array([[0]]), np.float32([[1.0]]), 0, 1, src)[0]
    for r in range(hh):
        want = 0.0
        for i in range(ii):
            g = gvals[i] * x0
            want += dvals[r, i] * (g / (1.0 + math.exp(-g))) * (uvals[i] * x0)
        assert abs(y[r] - want) <= 1e-12 * max(1.0, abs(want))


def test_per_route_loop_equals_dense_einsum(tiny):
    rng = np.random.default_rng(0)
    B = 3
    ids = rng.integers(0, E, (B, K))
    gates = rng.random((B, K)).astype(np.float32)
    x = rng.standard_normal((B, H))
    shared = tiny(5)
    for layer in range(L):
        a = decode_layer(x, ids, gates, layer, E, tiny, shared)
        b = decode_layer_dense(x, ids, gates, layer, E, tiny, shared)
        assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_merge_is_invariant_to_split_and_capacity(tiny):
    B, steps = 2, 12
    trace = locality_trace(0, L, E, K, B, steps, 0.5)
    gates = decode_gates(0, steps, L, B, K)
    rng = np.random.default_rng(1)
    xs = rng.standard_normal((steps, L, B, H))
    results = []
    for cap, full, f in ((8, True, 65536), (8, False, 32768), (8, False, 16384),
                         (3, False, 4096), (L * E, False, 43691)):
        cache = SlotCache(L, E, cap, full, f)
        ys = []
        for t in range(steps):
            for l in range(L):
                r = cache.decode(l, trace[t, l])
                y_gpu = decode_layer(xs[t, l], trace[t, l], gates[t, l], l, E, tiny,
                                     include=r.route_slot >= 0)
                y_cpu = decode_layer(xs[t, l], trace[t, l], gates[t, l], l, E, tiny,
                                     include=r.deferred >= 0)
                assert not ((r.route_slot >= 0) & (r.deferred >= 0)).any()
                ys.append(y_gpu + y_cpu)
        results.append(np.array(ys))
    ref = []
    for t in range(steps):
        for l in range(L):
            ref.append(decode_layer(xs[t, l], trace[t, l], gates[t, l], l, E, tiny))
    ref = np.array(ref)
    for ys in results:
        assert np.allclose(ys, ref, rtol=1e-12, atol=1e-15)


def test_prefill_against_unquantised_definition(tiny):
    T = 24
    x = prefill_x(0, 1, T, H).float().numpy()
    ids, gates = prefill_routes(0, 1, T, E, K)
    ids, gates = ids.numpy(), gates.numpy()
    y, hc, hs = prefill_layer(x, ids, gates, 1, E, tiny)
    assert np.array_equal(prefill_from_h(hc, hs, ids, gates, 1, E, tiny), y)
    exact = decode_layer(x, ids, gates, 1, E, tiny)
    rel = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel < 0.25          # two NVFP4 activation roundings, nothing structural
    perm = np.random.default_rng(0).permutation(T)
    y2, _, _ = prefill_layer(x[perm], ids[perm], gates[perm], 1, E, tiny)
    assert np.allclose(y2, y[perm], rtol=0, atol=0)


def test_prefill_routes_are_topk_of_logits():
    ids, gates = prefill_routes(3, 0, 64, E, 4)
    ids = ids.numpy()
    assert all(len(set(r)) == 4 for r in ids.tolist())
    assert np.allclose(gates.numpy().sum(1), 1.0, atol=1e-6)
    assert np.all(np.diff(gates.numpy(), axis=1) <= 0)      # sorted by logit
