"""Pins for oracle.formats: the NVFP4 codecs, quantisers and the expert record."""
import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import formats as F

# The E2M1 value table of the OCP microscaling FP4 element format (codes 0..15).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_decode_every_code():
    got = F.e2m1_decode(np.arange(16))
    assert got.tolist() == E2M1_TABLE
    assert np.all(np.signbit(got[8:]))


def test_e4m3_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(0, 448, 20000), np.exp(rng.uniform(-16, 6, 20000)),
                        F.e4m3_decode(np.arange(0x7F)),
                        (F.e4m3_decode(np.arange(0x7E)) + F.e4m3_decode(np.arange(1, 0x7F))) / 2])
    v = v[(v >= 0) & (v <= 448)].astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode_unsigned(v), ref)


def test_e4m3_encode_saturates():
    assert F.e4m3_encode_unsigned(np.float32([449, 464, 1e30])).tolist() == [0x7E] * 3


def test_e2m1_encode_round_trip_and_ties():
    # every representable value round-trips (negative zero is canonicalised to +0)
    vals = np.array(E2M1_TABLE, np.float32)
    codes = F.e2m1_encode(vals)
    assert np.array_equal(F.e2m1_decode(codes), vals)
    assert codes[8] == 0
    # midpoints go to the even mantissa (code with bit 0 clear)
    mids = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert F.e2m1_decode(F.e2m1_encode(mids)).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert F.e2m1_decode(F.e2m1_encode(-mids)).tolist() == [0.0, -1.0, -1.0, -2.0, -2.0, -4.0, -4.0]
    # off-midpoint values go to the nearer neighbour
    eps = np.float32(1e-4)
    assert F.e2m1_decode(F.e2m1_encode(mids + eps)).tolist() == [0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert F.e2m1_decode(F.e2m1_encode(mids - eps)).tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0]
    # saturation
    assert F.e2m1_decode(F.e2m1_encode(np.float32([7, 1e9, -100]))).tolist() == [6.0, 6.0, -6.0]


def test_e2m1_encode_is_nearest():
    rng = np.random.default_rng(2)
    v = rng.uniform(-7, 7, 50000).astype(np.float32)
    dec = F.e2m1_decode(F.e2m1_encode(v))
    grid = np.array(sorted(set(abs(x) for x in E2M1_TABLE)))
    best = np.min(np.abs(np.abs(v)[:, None].astype(np.float64) - grid[None, :]), axis=1)
    assert np.allclose(np.abs(np.abs(v) - np.abs(dec)), best, rtol=0, atol=0)
    assert np.all((np.sign(dec) == np.sign(v)) | (dec == 0))


def test_weight_quantiser_exact_construction():
    # amax = 6c  ->  s_t = 6c / 2688,  block scale (6c/6)/s_t rounds to 448, and
    # blk * s_t = c up to the fp32 rounding of s_t, so every code is w / c.
    c = np.float32(0.0078125)
    row = np.array(E2M1_TABLE, np.float32)
    w = np.stack([row * c, row[::-1] * c]).astype(np.float32)
    codes, scales, s_t = F.quantize_weight(w)
    assert s_t == np.float32(6 * c) / np.float32(2688)
    assert np.all(scales == 0x7E)
    assert np.array_equal(F.e2m1_decode(codes) * float(c), w.astype(np.float64))
    assert np.allclose(F.dequant(codes, scales, s_t), w, rtol=2.0 ** -23, atol=0)


def test_weight_quantiser_error_bound():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    codes, scales, s_t = F.quantize_weight(w)
    dq = F.dequant(codes, scales, s_t)
    blk = F.e4m3_decode(scales).repeat(16, axis=1) * float(s_t)
    mag = np.abs(F.e2m1_decode(codes))
    # half the local code spacing (spacing 0.5 below 2, 1 in [2, 4), 2 at and above 4)
    half = np.where(mag < 2, 0.25, np.where(mag < 4, 0.5, 1.0)) * blk
    over = np.maximum(np.abs(w) / blk - 6.0, 0) * blk           # saturated tails
    assert np.all(np.abs(w - dq) <= half + over + 1e-6 * blk)
    # the element holding amax is reproduced to fp32 rounding
    i = np.unravel_index(np.argmax(np.abs(w)), w.shape)
    assert abs(dq[i] - w[i]) <= 1e-6 * abs(w[i])
    z_codes, z_scales, z_t = F.quantize_weight(np.zeros((4, 32), np.float32))
    assert z_t == 0 and not z_codes.any() and not z_scales.any()


def test_activation_quantiser_exact_and_ties():
    # a block whose amax is 6 * 2^j has scale exactly 2^j; codes are v / 2^j
    x = np.zeros((2, 32), np.float32)
    x[0, :16] = np.array(E2M1_TABLE, np.float32) * 4.0           # amax 24 -> s = 4
    x[1, 16:] = np.array(E2M1_TABLE, np.float32)[::-1] * 0.25    # amax 1.5 -> s = 0.25
    codes, scales = F.quantize_act(x)
    assert F.e4m3_decode(scales).tolist() == [[4.0, 0.0], [0.0, 0.25]]
    assert np.array_equal(F.dequant(codes, scales), x.astype(np.float64))
    # ties inside a block with scale 1: 2.5 -> 2, 3.5 -> 4, 5 -> 4
    t = np.zeros((1, 16), np.float32)
    t[0, :4] = [6.0, 2.5, 3.5, 5.0]
    c, s = F.quantize_act(t)
    assert F.dequant(c, s)[0, :4].tolist() == [6.0, 2.0, 4.0, 4.0]


def test_nibble_order_and_record_layout():
    packed = F.pack_nibbles(np.array([[1, 2, 15, 0]], np.uint8))
    assert packed.tolist() == [[0x21, 0x0F]]
    assert np.array_equal(F.unpack_nibbles(packed), [[1, 2, 15, 0]])
    # sizes: codes + scales of W_gu [2I,H] and W_d [H,I] + two fp32 tensor scales
    assert F.record_layout(64, 32)["raw_bytes"] == 3464
    assert F.record_layout(64, 32)["bytes"] == 3584
    assert F.record_layout(2048, 512)["raw_bytes"] == 1769480
    assert F.record_layout(4096, 2048)["raw_bytes"] == 14155784


def test_record_gate_rows_first_round_trip():
    H, I = 32, 16
    c = np.float32(0.5)
    row = np.array(E2M1_TABLE * 2, np.float32)[:H] * c
    w_gu = np.concatenate([np.tile(np.abs(row), (I, 1)), -np.tile(np.abs(row), (I, 1))])
    w_d = np.tile(np.array(E2M1_TABLE, np.float32) * c, (H, 1))
    rec = F.encode_record(w_gu, w_d)
    g, d = F.decode_record(rec, H, I)
    assert np.all(g[:I] >= 0) and np.all(g[I:] <= 0)
    f = F.record_fields(rec, H, I)
    assert np.array_equal(F.e2m1_decode(f["gu_codes"]) * float(c), w_gu.astype(np.float64))
    assert np.array_equal(F.e2m1_decode(f["d_codes"]) * float(c), w_d.astype(np.float64))
    assert np.allclose(g, w_gu, rtol=2.0 ** -23, atol=0) and np.allclose(d, w_d, rtol=2.0 ** -23, atol=0)


def test_pool_shape_matches_pages_bf16_pool():
    # [EXPLAINER §4.2]: the BF16 pool streamed per chunk is 64.4 GB.  Our record holds
    # the same 3*H*I weights per expert as nibbles (4 per 2 bytes of BF16).
    (L, E, H, I, bpw, gb, bp, lo, hi), = read_golden("prefill_chunk.txt")
    L, E, H, I, bpw = int(L), int(E), int(H), int(I), int(bpw)
    lay = F.record_layout(H, I)
    nibble_bytes = lay["gu_codes"][1] + lay["d_codes"][1]
    pool_bf16 = L * E * nibble_bytes * 2 * bpw
    assert abs(pool_bf16 / 1e9 - float(gb)) < 0.05
    t = pool_bf16 / (float(bp) * 1e9)
    assert float(lo) <= t + 0.01 and t <= float(hi) + 0.01


# ---------------------------------------------------------------- MXFP4

def test_e8m0_decode_matches_torch_float8_e8m0():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without float8_e8m0fnu")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = F.e8m0_decode(codes)
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def _brute_mx_block(v):
    """Shared exponent k with 2^(k+2) <= amax < 2^(k+3) found by search, and each code
    as the nearest of the 16 E2M1 values to v / 2^k (ties to the even code, beyond 6
    the largest)."""
    import math
    a = max(abs(float(x)) for x in v)
    if a == 0:
        k = -127
    else:
        k = -200
        while 2.0 ** (k + 3) <= a:
            k += 1
        k = max(-127, min(127, k))
    codes = []
    for x in v:
        t = float(x) / 2.0 ** k
        best = None
        for c in range(16):
            val = F.e2m1_decode(c)
            d = abs(float(val) - t)
            key = (d, c & 1, c)                 # nearest; ties: even mantissa bit
            if abs(t) > 6:
                key = (abs(abs(float(val)) - 6) + (0 if (val < 0) == (t < 0) else 9), 0, c)
            if best is None or key < best[0]:
                best = (key, c)
        c = best[1]
        if float(F.e2m1_decode(c)) == 0:
            c = 0                               # zero magnitudes are +0
        codes.append(c)
    return k + 127, codes


def test_quantize_mx_constructions():
    grid = [6.0, 4.0, -3.0, 0.5, 1.5, -2.0, 1.0, 0.0] * 4
    rows = []
    rows.append([g * 2.0 ** -7 for g in grid])                      # amax 6 * 2^-7 -> scale -7
    rows.append([7.0 * 2.0 ** 3] + [1.0 * 2.0 ** 3] * 31)           # amax 7 * 2^3: 7 saturates to 6
    rows.append([4.0 * 2.0 ** -2] + [-0.5 * 2.0 ** -2] * 31)        # amax 4 * 2^k: exponent k
    rows.append([3.9] + [0.25] * 31)                                 # floor(log2 3.9) = 1: shared -1
    rows.append([0.0] * 32)                                          # zero block -> code 0, scale 0
    rows.append([2.0 ** -130] + [0.0] * 31)                          # clamp at -127
    w = np.array(rows, np.float32)
    codes, scales = F.quantize_mx(w)
    assert scales.reshape(-1).tolist() == [120, 130, 125, 126, 0, 0]
    assert codes[0].tolist() == [F.e2m1_encode(g).item() for g in grid]
    assert codes[1, 0] == 7 and codes[1, 1] == 2
    assert codes[2, 0] == 6 and codes[2, 1] == 9
    assert codes[3, 0] == 7 and codes[3, 1] == 1              # 3.9 * 2 -> 6 (saturated), 0.25 * 2 = 0.5
    assert not codes[4].any()
    # 2^-130 * 2^127 = 1/8: rounds to 0 (below 0.25)
    assert codes[5, 0] == 0
    rng = np.random.default_rng(3)
    wr = (rng.standard_normal((6, 64)) * np.exp(rng.uniform(-12, 8, (6, 1)))).astype(np.float32)
    c2, s2 = F.quantize_mx(wr)
    for r in range(6):
        for b in range(2):
            sc, cc = _brute_mx_block(wr[r, 32 * b:32 * b + 32])
            assert s2[r, b] == sc and c2[r, 32 * b:32 * b + 32].tolist() == cc


def test_mx_record_layout_and_round_trip():
    H, I = 4096, 2048
    lay = F.record_layout(H, I, "mxfp4")
    assert lay["gu_scales"][1] == 2 * I * H // 32 and lay["d_scales"][1] == H * I // 32
    assert lay["raw_bytes"] == 3 * H * I // 2 + 3 * H * I // 32 + 8
    assert lay["bytes"] % 256 == 0
    rng = np.random.default_rng(4)
    h, i = 64, 32
    w_gu = (rng.standard_normal((2 * i, h)) * 0.02).astype(np.float32)
    w_d = (rng.standard_normal((h, i)) * 0.02).astype(np.float32)
    rec = F.encode_record(w_gu, w_d, "mxfp4")
    f = F.record_fields(rec, h, i, "mxfp4")
    assert f["s_gu"] == 1.0 and f["s_d"] == 1.0
    g, d = F.decode_record(rec, h, i, "mxfp4")
    c, s = F.quantize_mx(w_gu)
    assert np.array_equal(g, F.e2m1_decode(c) * np.repeat(2.0 ** (s.astype(np.int64) - 127), 32, axis=1))
    # every value of the decoded weights is on its block's E2M1 grid
    assert np.all(np.abs(d) <= 6 * np.repeat(F.e8m0_decode(f["d_scales"]), 32, axis=1))


def test_mx_and_nvfp4_records_of_the_same_values_decode_alike():
    """Blocks whose scales are powers of two inside E4M3's range: the MXFP4 record
    (E8M0 per 32) and an NVFP4 record with those scales (E4M3 per 16, tensor scale 1)
    hold the same weights."""
    rng = np.random.default_rng(5)
    h, i = 64, 32
    lay_n, lay_m = F.record_layout(h, i), F.record_layout(h, i, "mxfp4")
    recs = {"nvfp4": np.zeros(lay_n["bytes"], np.uint8), "mxfp4": np.zeros(lay_m["bytes"], np.uint8)}
    for name, rows, k in (("gu", 2 * i, h), ("d", h, i)):
        codes = rng.integers(0, 16, (rows, k)).astype(np.uint8)
        exps = rng.integers(-9, 9, (rows, k // 32))                 # E4M3 holds 2^-9 .. 2^8
        e4m3 = {F.e4m3_decode(c).item(): c for c in range(0x7F)}
        n_sc = np.repeat(np.vectorize(lambda e: e4m3[2.0 ** e])(exps), 2, axis=1).astype(np.uint8)
        for fmt, sc in (("nvfp4", n_sc), ("mxfp4", (exps + 127).astype(np.uint8))):
            lay = F.record_layout(h, i, fmt)
            off, size = lay[name + "_codes"]
            recs[fmt][off:off + size] = F.pack_nibbles(codes).reshape(-1)
            off, size = lay[name + "_scales"]
            recs[fmt][off:off + size] = sc.reshape(-1)
    for fmt in recs:
        lay = F.record_layout(h, i, fmt)
        for t in ("s_gu", "s_d"):
            off, size = lay[t]
            recs[fmt][off:off + size] = np.float32([1.0]).view(np.uint8)
    gn, dn = F.decode_record(recs["nvfp4"], h, i)
    gm, dm = F.decode_record(recs["mxfp4"], h, i, "mxfp4")
    assert np.array_equal(gn, gm) and np.array_equal(dn, dm)
