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


# ---------------------------------------------------------------- prefill closed form
#
# Every value below is chosen so that both activation quantisations are exact or
# decided by a known rounding rule, and y is exact in fp64:
#   * token t has one non-zero x element, 6.0 at column c_t of the first 16-block:
#     amax 6 -> scale E4M3(1.0) (code 0x38), code of 6.0; the other blocks have
#     amax 0 -> scale 0, a zero block.  So g_i = 6 * Wg[i, c_t], u_i = 6 * Wu[i, c_t].
#   * "on" rows: Wg = 4 -> g = 24, silu(24) = 24 (1 - 3.8e-11), so the fp32 h is
#     exactly 144 * Wu (the relative deviation is far below half an fp32 ulp).
#     Each 16-row block of h holds one row with |Wu| = 6, so amax = 864, the block
#     scale is E4M3(864 / 6) = E4M3(144) = 144 exactly (code 0x71) and the code of an
#     on row is the code of Wu itself.
#   * the "mid" row: Wg = 3, Wu = 1 -> h = silu(18) * 6 = 108 (1 - 1.5e-8) in fp64,
#     which rounds to exactly 108.0 in fp32; 108 / 144 = 0.75 is the tie between
#     E2M1 0.5 and 1.0 and goes to the even code 2 (1.0).  Quantising the unrounded
#     fp64 value instead would give 0.5 (code 1).
#   * "neg" rows: Wg = -4 -> g = -24, |h| < 1e-8 -> code 0 (zero magnitudes are +0).
#   * "zero" rows: Wg = 0 -> h = 0 -> code 0.
# Gates are dyadic and not 1: a gate applied before h is quantised changes the
# block scale (0.75 * 864 / 6 = 108 is not an E4M3 value), so h codes catch it.

_E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _fp4_code(v):
    c = _E2M1_VALUES.index(abs(v))
    return c | (8 if v < 0 and c else 0)


def _fp4_value(c):
    return (-1.0 if c & 8 else 1.0) * _E2M1_VALUES[c & 7]


def _prefill_fixture():
    Hh, Ii, Ee, T, k = 64, 32, 4, 3, 2
    cols = [1, 6, 11]                                  # c_t, all in x's first 16-block
    ids = np.array([[0, 1], [1, 2], [3, 0]])
    gates = np.float32([[0.75, 0.25], [0.625, 0.375], [0.8125, 0.1875]])
    rng = np.random.default_rng(7)
    ladder = [0.5, -1.0, 1.5, -2.0, 3.0, -4.0, 0.5, 2.0, -1.5, 1.0]
    recs, h_want = [], {}
    for e in range(Ee):
        gu = rng.integers(0, 16, (2 * Ii, Hh)).astype(np.uint8)   # columns x never uses
        d = rng.integers(0, 16, (Hh, Ii)).astype(np.uint8)
        for c in cols:
            want = []
            for i in range(Ii):
                b, r = divmod(i, 16)
                if r == 0:                                   # on, |Wu| = 6: sets amax
                    wg, wu, code = 4.0, (6.0 if (e + c + b) % 2 else -6.0), None
                elif r <= 10:                                # on, varied Wu
                    wg, wu, code = 4.0, ladder[(r - 1 + e + c) % 10], None
                elif r == 11:                                # mid: the fp32 tie
                    wg, wu, code = 3.0, 1.0, 2
                elif r == 12:                                # neg, u > 0
                    wg, wu, code = -4.0, 2.0, 0
                elif r == 13:                                # neg, u < 0
                    wg, wu, code = -4.0, -3.0, 0
                elif r == 14:                                # zero gate
                    wg, wu, code = 0.0, 1.5, 0
                else:                                        # on, small
                    wg, wu, code = 4.0, -0.5, None
                gu[i, c] = _fp4_code(wg)
                gu[Ii + i, c] = _fp4_code(wu)
                want.append(_fp4_code(wu) if code is None else code)
            h_want[(e, c)] = want
        recs.append(_record_from_codes(gu, d))
    x = np.zeros((T, Hh), np.float32)
    for t, c in enumerate(cols):
        x[t, c] = 6.0
    return Hh, Ii, Ee, T, k, cols, ids, gates, recs, h_want


def test_prefill_closed_form():
    Hh, Ii, Ee, T, k, cols, ids, gates, recs, h_want = _prefill_fixture()
    x = np.zeros((T, Hh), np.float32)
    for t, c in enumerate(cols):
        x[t, c] = 6.0
    src = RecordSource(lambda f: recs[f], Hh, Ii)
    y, hc, hs, h32 = prefill_layer(x, ids, gates, 0, Ee, src, return_h32=True)
    # h per route row r = t*k + j: the codes worked out above, scale 144 (0x71)
    for t in range(T):
        for j in range(k):
            r = t * k + j
            want = h_want[(int(ids[t, j]), cols[t])]
            assert hc[r].tolist() == want, f"h codes of route ({t}, {j})"
            assert hs[r].tolist() == [0x71, 0x71], f"h scales of route ({t}, {j})"
            assert h32[r][11] == np.float32(108.0) and h32[r][27] == np.float32(108.0)
    # y by hand: o = W_d . hq with hq = code value * 144, then the gated sum over j
    d_vals = [F.unpack_nibbles(rec[F.record_layout(Hh, Ii)["d_codes"][0]:][:Hh * Ii // 2]
                               .reshape(Hh, Ii // 2)) for rec in recs]
    for t in range(T):
        want_y = [0.0] * Hh
        for j in range(k):
            e = int(ids[t, j])
            hq = [_fp4_value(cd) * 144.0 for cd in h_want[(e, cols[t])]]
            for row in range(Hh):
                o = sum(_fp4_value(int(d_vals[e][row, i])) * hq[i] for i in range(Ii))
                want_y[row] += float(gates[t, j]) * o
        assert y[t].tolist() == want_y, f"y of token {t}"
    # the second GEMM alone, from the same h
    assert np.array_equal(prefill_from_h(hc, hs, ids, gates, 0, Ee, src), y)


def test_prefill_closed_form_masks_and_order():
    """A route whose id is outside [0, E) contributes nothing and leaves its h row
    zero; swapping the two routes of a token (ids and gates together) moves the h
    rows to the swapped route indices and leaves y unchanged."""
    Hh, Ii, Ee, T, k, cols, ids, gates, recs, h_want = _prefill_fixture()
    x = np.zeros((T, Hh), np.float32)
    for t, c in enumerate(cols):
        x[t, c] = 6.0
    src = RecordSource(lambda f: recs[f], Hh, Ii)
    y, hc, hs = prefill_layer(x, ids, gates, 0, Ee, src)
    ids_sw, gates_sw = ids[:, ::-1].copy(), gates[:, ::-1].copy()
    y2, hc2, hs2 = prefill_layer(x, ids_sw, gates_sw, 0, Ee, src)
    for t in range(T):
        assert np.array_equal(hc2[t * k], hc[t * k + 1]) and np.array_equal(hc2[t * k + 1], hc[t * k])
    assert np.allclose(y2, y, rtol=1e-15, atol=0)
    ids_m = ids.copy()
    ids_m[1, 0] = Ee                                       # masked route (1, 0)
    y3, hc3, hs3 = prefill_layer(x, ids_m, gates, 0, Ee, src)
    assert not hc3[1 * k + 0].any() and not hs3[1 * k + 0].any()
    assert np.array_equal(y3[[0, 2]], y[[0, 2]])
    # token 1 keeps only route (1, 1): y = gate * o of that route (a one-route
    # layer over that route's h row)
    only = prefill_from_h(hc[[1 * k + 1]], hs[[1 * k + 1]], np.array([[ids[1, 1]]]),
                          gates[1:2, 1:2], 0, Ee, src)
    assert np.array_equal(y3[1], only[0])
