"""NVFP4 number formats and the per-flat-id expert record (oracle side).

TEST INFRASTRUCTURE: see the package docstring for who may import this.

What the pages fix, and what this module restates:
  * Experts are served as NVFP4 on the NVFP4 machines ([EXPLAINER §9.2], the 4060
    Laptop and RTX PRO 6000 rows; [JUHE] "先纠正一个容易混淆的模型": Qwen3.6-35B-A3B
    NVFP4).  NVFP4 = E2M1 element codes, an E4M3 scale per 16 consecutive elements
    and one fp32 tensor scale per stored matrix.
  * One flat id  id(l, e) = l*E + e  names one whole expert in every weight bank
    ([EXPLAINER §8.4]; [JUHE] "FTW 为什么能缩短启动时间").  Here the banks of one
    flat id are laid out back to back so that a cache fill is one contiguous copy.

Record layout (bytes, one per flat id, padded to a multiple of 256):
    [W_gu codes  2I*H/2][W_gu scales 2I*H/16][W_d codes H*I/2][W_d scales H*I/16]
    [s_gu fp32][s_d fp32][zero padding]
  W_gu is [2I, H] row-major (K = H contiguous), rows [0, I) = gate, [I, 2I) = up.
  W_d  is [H, I]  row-major (K = I contiguous).
  Two codes per byte, element 2j in the low nibble, element 2j+1 in the high one.
  Scales are unsigned E4M3 bytes, row-major [rows, K/16].

MXFP4 ([EXPLAINER §9.2] and the model table: DeepSeek-V4-Flash's routed experts are
natively MXFP4, and the engines consume those blocks bit-exactly): E2M1 codes as above,
one unsigned E8M0 scale (value 2^(c - 127), code 255 is NaN) per 32 consecutive
elements of a row, no tensor scale.  The MXFP4 record has the same layout with the
scale arrays [rows, K/32] and the two tensor-scale words fixed at 1.0.  Synthetic
MXFP4 pools are quantised with the conversion rule of the microscaling format
definition: shared exponent floor(log2(amax_32)) - 2 (2 = the largest E2M1
exponent), clamped to [-127, 127]; code = E2M1_RNE_sat(v / 2^shared).

Quantiser arithmetic is written as fp32 IEEE round-to-nearest steps (numpy float32
ops), so that a device implementation doing the same fp32 steps is bit-exact.
Decoding goes to fp64 and is exact.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------- E2M1 (FP4)

def e2m1_decode(codes) -> np.ndarray:
    """Value of 4-bit E2M1 codes: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.

    exponent 0 is subnormal (m * 0.5); otherwise 2^(e-1) * (1 + m/2).
    """
    c = np.asarray(codes).astype(np.int64) & 0xF
    s = c >> 3
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return np.where(s == 1, -mag, mag).astype(np.float64)


_E2M1_MAG = e2m1_decode(np.arange(8))          # 0, .5, 1, 1.5, 2, 3, 4, 6 (ascending)


def _nearest_even(a: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index of the nearest value of an ascending table; exact ties go to the even
    index (the even mantissa: consecutive codes alternate mantissa parity).
    Values above the last entry saturate to it."""
    a = np.asarray(a, dtype=np.float64)
    hi = np.searchsorted(table, a, side="left")          # table[hi-1] < a <= table[hi]
    hi = np.clip(hi, 1, len(table) - 1)
    lo = hi - 1
    dlo = a - table[lo]
    dhi = table[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(a <= table[0], 0, idx)
    idx = np.where(a >= table[-1], len(table) - 1, idx)
    return idx.astype(np.int64)


def e2m1_encode(v) -> np.ndarray:
    """Round-to-nearest-even E2M1 code of fp32 values, saturating at +-6.

    Zero magnitudes are always encoded as +0 (code 0): the sign bit is set only
    for a negative value whose rounded magnitude is non-zero.
    """
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("E2M1 encode of a non-finite value")
    mag = _nearest_even(np.abs(v), _E2M1_MAG)
    neg = (v < 0) & (mag != 0)
    return (mag | (neg.astype(np.int64) << 3)).astype(np.uint8)


# ---------------------------------------------------------------- E4M3 (FP8)

def e4m3_decode(codes) -> np.ndarray:
    """Value of 8-bit E4M3 codes (bias 7, no infinities; 0x7F/0xFF are NaN).

    exponent 0 is subnormal: m/8 * 2^-6; otherwise 2^(e-7) * (1 + m/8).
    """
    c = np.asarray(codes).astype(np.int64) & 0xFF
    s = c >> 7
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag).astype(np.float64)


_E4M3_POS = e4m3_decode(np.arange(0x7F))        # finite non-negative values, ascending


def e4m3_encode_unsigned(v) -> np.ndarray:
    """Round-to-nearest-even unsigned E4M3 code of non-negative fp32 values,
    saturating at 448 (code 0x7E)."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    if np.any(v < 0) or not np.all(np.isfinite(v)):
        raise ValueError("unsigned E4M3 encode needs finite values >= 0")
    return _nearest_even(v, _E4M3_POS).astype(np.uint8)


# ---------------------------------------------------------------- E8M0 (MX scale)

def e8m0_decode(codes) -> np.ndarray:
    """Value of unsigned 8-bit E8M0 scale codes: 2^(c - 127); code 255 is NaN."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    v = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, v).astype(np.float64)


# ---------------------------------------------------------------- quantisers

F32 = np.float32
BLOCK = 16


def quantize_weight(w) -> tuple[np.ndarray, np.ndarray, np.float32]:
    """NVFP4 weight quantiser, fp32 IEEE steps.

    s_t   = amax(W) / (6*448)                          (one fp32 tensor scale)
    blk   = E4M3_RNE((amax_block16 / 6) / s_t)
    code  = E2M1_RNE_sat(w / (blk * s_t));  a zero block scale gives a zero block.
    Returns (codes uint8 [rows, K] one code per element, scales uint8 [rows, K/16], s_t).
    """
    w = np.asarray(w, dtype=F32)
    rows, k = w.shape
    assert k % BLOCK == 0
    amax = F32(np.max(np.abs(w))) if w.size else F32(0)
    s_t = F32(amax / F32(6.0 * 448.0))
    if s_t == 0:
        return (np.zeros((rows, k), np.uint8), np.zeros((rows, k // BLOCK), np.uint8), F32(0))
    blocks = w.reshape(rows, k // BLOCK, BLOCK)
    amax_b = np.max(np.abs(blocks), axis=2).astype(F32)
    t = ((amax_b / F32(6.0)).astype(F32) / s_t).astype(F32)
    sc = e4m3_encode_unsigned(t)
    sc_val = e4m3_decode(sc).astype(F32)                 # exact
    denom = (sc_val * s_t).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        qv = (blocks / denom[..., None]).astype(F32)
    qv = np.where(denom[..., None] == 0, F32(0), qv)
    codes = e2m1_encode(qv).reshape(rows, k)
    return codes, sc, s_t


def quantize_act(x) -> tuple[np.ndarray, np.ndarray]:
    """NVFP4 activation quantiser with a unit tensor scale, fp32 IEEE steps.

    s    = E4M3_RNE(amax_block16 / 6)
    code = E2M1_RNE_sat(v / s);  s = 0 gives a zero block.
    Returns (codes uint8 [rows, K], scales uint8 [rows, K/16]).
    """
    x = np.asarray(x, dtype=F32)
    rows, k = x.shape
    assert k % BLOCK == 0
    blocks = x.reshape(rows, k // BLOCK, BLOCK)
    a = np.max(np.abs(blocks), axis=2).astype(F32)
    sc = e4m3_encode_unsigned((a / F32(6.0)).astype(F32))
    s = e4m3_decode(sc).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        qv = (blocks / s[..., None]).astype(F32)
    qv = np.where(s[..., None] == 0, F32(0), qv)
    return e2m1_encode(qv).reshape(rows, k), sc


MX_BLOCK = 32


def quantize_mx(w) -> tuple[np.ndarray, np.ndarray]:
    """MXFP4 quantiser (conversion rule of the microscaling format definition), fp32
    IEEE steps, per 32 consecutive elements of a row:
      shared = floor(log2(amax)) - 2, clamped to [-127, 127] (amax = 0: -127);
      scale code = shared + 127;  code = E2M1_RNE_sat(v * 2^-shared).
    floor(log2(amax)) is exact: the exponent of amax's binary representation.
    Returns (codes uint8 [rows, K] one code per element, scales uint8 [rows, K/32])."""
    w = np.asarray(w, dtype=F32)
    rows, k = w.shape
    assert k % MX_BLOCK == 0
    blocks = w.reshape(rows, k // MX_BLOCK, MX_BLOCK)
    amax = np.max(np.abs(blocks), axis=2).astype(F32)
    _, e = np.frexp(amax)                       # amax = m * 2^e, m in [0.5, 1)
    shared = np.where(amax > 0, e.astype(np.int64) - 1 - 2, -127)
    shared = np.clip(shared, -127, 127)
    mul = np.ldexp(np.float32(1.0), (-shared).astype(np.int32)).astype(F32)   # exact powers of two
    qv = (blocks * mul[..., None]).astype(F32)
    codes = e2m1_encode(qv).reshape(rows, k)
    return codes, (shared + 127).astype(np.uint8)


def dequant_mx(codes, scales) -> np.ndarray:
    """fp64 value of MXFP4 data: e2m1(code) * 2^(scale - 127) of its 32-block (exact)."""
    codes = np.asarray(codes)
    rows, k = codes.shape
    v = e2m1_decode(codes).reshape(rows, k // MX_BLOCK, MX_BLOCK)
    v = v * e8m0_decode(scales)[..., None]
    return v.reshape(rows, k)


def dequant(codes, scales, s_t=1.0) -> np.ndarray:
    """fp64 value of NVFP4 data: e2m1(code) * e4m3(scale of its 16-block) * s_t (exact)."""
    codes = np.asarray(codes)
    rows, k = codes.shape
    v = e2m1_decode(codes).reshape(rows, k // BLOCK, BLOCK)
    v = v * e4m3_decode(scales)[..., None] * float(s_t)
    return v.reshape(rows, k)


# ---------------------------------------------------------------- expert record

def pack_nibbles(codes) -> np.ndarray:
    """[rows, K] codes -> [rows, K/2] bytes, element 2j in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)


def unpack_nibbles(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


FORMATS = ("nvfp4", "mxfp4")


def record_layout(H: int, I: int, fmt: str = "nvfp4") -> dict:
    """Byte offsets and sizes of one expert record for hidden H, intermediate I."""
    sb = BLOCK if fmt == "nvfp4" else MX_BLOCK
    assert fmt in FORMATS and H % sb == 0 and I % sb == 0
    lay = {}
    off = 0
    for name, size in (("gu_codes", 2 * I * H // 2), ("gu_scales", 2 * I * H // sb),
                       ("d_codes", H * I // 2), ("d_scales", H * I // sb),
                       ("s_gu", 4), ("s_d", 4)):
        lay[name] = (off, size)
        off += size
    lay["raw_bytes"] = off
    lay["bytes"] = (off + 255) // 256 * 256
    return lay


def encode_record(w_gu, w_d, fmt: str = "nvfp4") -> np.ndarray:
    """Quantise fp32 W_gu [2I, H] and W_d [H, I] into one padded record (uint8)."""
    w_gu = np.asarray(w_gu, F32)
    w_d = np.asarray(w_d, F32)
    two_i, H = w_gu.shape
    I = two_i // 2
    assert w_d.shape == (H, I)
    lay = record_layout(H, I, fmt)
    rec = np.zeros(lay["bytes"], np.uint8)
    if fmt == "mxfp4":
        for w, cn, sn, tn in ((w_gu, "gu_codes", "gu_scales", "s_gu"), (w_d, "d_codes", "d_scales", "s_d")):
            c, sc = quantize_mx(w)
            _put(rec, lay[cn], pack_nibbles(c))
            _put(rec, lay[sn], sc)
            _put(rec, lay[tn], np.array([1.0], F32).view(np.uint8))
        return rec
    c, s, t = quantize_weight(w_gu)
    _put(rec, lay["gu_codes"], pack_nibbles(c))
    _put(rec, lay["gu_scales"], s)
    _put(rec, lay["s_gu"], np.array([t], F32).view(np.uint8))
    c, s, t = quantize_weight(w_d)
    _put(rec, lay["d_codes"], pack_nibbles(c))
    _put(rec, lay["d_scales"], s)
    _put(rec, lay["s_d"], np.array([t], F32).view(np.uint8))
    return rec


def _put(rec, where, arr):
    off, size = where
    b = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
    assert b.size == size
    rec[off:off + size] = b


def _get(rec, where):
    off, size = where
    return np.asarray(rec[off:off + size], np.uint8)


def record_fields(rec, H: int, I: int, fmt: str = "nvfp4") -> dict:
    """Split a record into its raw fields (codes unpacked, scales, tensor scales)."""
    lay = record_layout(H, I, fmt)
    sb = BLOCK if fmt == "nvfp4" else MX_BLOCK
    rec = np.asarray(rec, np.uint8)
    return {
        "gu_codes": unpack_nibbles(_get(rec, lay["gu_codes"]).reshape(2 * I, H // 2)),
        "gu_scales": _get(rec, lay["gu_scales"]).reshape(2 * I, H // sb),
        "d_codes": unpack_nibbles(_get(rec, lay["d_codes"]).reshape(H, I // 2)),
        "d_scales": _get(rec, lay["d_scales"]).reshape(H, I // sb),
        "s_gu": _get(rec, lay["s_gu"]).view(F32)[0],
        "s_d": _get(rec, lay["s_d"]).view(F32)[0],
    }


def decode_record(rec, H: int, I: int, fmt: str = "nvfp4") -> tuple[np.ndarray, np.ndarray]:
    """fp64 (W_gu [2I, H], W_d [H, I]) of a record."""
    f = record_fields(rec, H, I, fmt)
    if fmt == "mxfp4":
        return dequant_mx(f["gu_codes"], f["gu_scales"]), dequant_mx(f["d_codes"], f["d_scales"])
    return (dequant(f["gu_codes"], f["gu_scales"], f["s_gu"]),
            dequant(f["d_codes"], f["d_scales"], f["s_d"]))
