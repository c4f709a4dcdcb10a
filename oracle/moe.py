"""Dense fp64 definitions of the routed MoE layer output (decode and prefill).

TEST INFRASTRUCTURE: see the package docstring for who may import this.

Sources:
  [EXPLAINER §1.1]    h = sum over the top-k experts of p_e * Expert_{l,e}(x).
  [JUHE "为什么可以直接相加？"]  y = g1*E1(x) + ... + gk*Ek(x); splitting the expert set
                      between GPU and CPU only moves where each term is computed,
                      so y = y_gpu + y_cpu exactly (each route computed once).
  [EXPLAINER §6.2, §6.9]  the split keeps ids, k, gates, weights and the set of summed
                      outputs; only the floating-point reduction order may differ.
  [BWRATIO "代码全链路" §2]  GPU-side weights of CPU routes are zero, CPU-side ids of
                      GPU routes are -1, so the two partials are complementary.
  [JUHE "先纠正一个容易混淆的模型"]  Qwen3.6-35B-A3B: top-8 routed experts plus one
                      always-active shared expert.

Experts are SwiGLU: Expert(x) = W_d (silu(W_g x) * (W_u x)), silu(a) = a / (1 + e^-a),
with W_g, W_u the gate and up halves of the stored W_gu. Every weight is the exact
fp64 decode of its NVFP4 record. Reading for the shared expert (the pages do not
give its gate): weight 1, same shape as a routed expert.
"""
from __future__ import annotations

import numpy as np

from .formats import decode_record, dequant, quantize_act


def silu(a):
    return a / (1.0 + np.exp(-a))


def swiglu(w_gu: np.ndarray, w_d: np.ndarray, x: np.ndarray) -> np.ndarray:
    """Expert output for rows of x ([n, H] fp64) with fp64 weights."""
    I = w_gu.shape[0] // 2
    g = x @ w_gu[:I].T
    u = x @ w_gu[I:].T
    return (silu(g) * u) @ w_d.T


class RecordSource:
    """Decoded-expert lookup with a small memo, from a callable flat_id -> record bytes
    (records in format fmt: "nvfp4" or "mxfp4")."""

    def __init__(self, get_record, H: int, I: int, fmt: str = "nvfp4"):
        self.get_record, self.H, self.I, self.fmt = get_record, H, I, fmt
        self.memo = {}

    def __call__(self, flat: int):
        if flat not in self.memo:
            self.memo[flat] = decode_record(self.get_record(flat), self.H, self.I, self.fmt)
        return self.memo[flat]


def decode_layer(x, ids, gates, layer: int, E: int, experts: RecordSource,
                 shared=None, include=None) -> np.ndarray:
    """y[b] = sum_j gates[b,j] * Expert_{layer, ids[b,j]}(x[b])  (+ Shared(x[b])).

    x: [B, H] activations (bf16 values, taken exactly); gates: [B, k] fp32.
    include: optional bool [B, k]; routes outside it contribute nothing (used for
    the CPU partial: include = deferred >= 0, shared=None).
    Routes with ids outside [0, E) contribute nothing.
    """
    x = np.asarray(x, np.float64)
    ids = np.asarray(ids, np.int64)
    gates = np.asarray(gates, np.float32).astype(np.float64)
    B, k = ids.shape
    y = np.zeros((B, x.shape[1]), np.float64)
    for b in range(B):
        for j in range(k):
            e = int(ids[b, j])
            if not (0 <= e < E) or (include is not None and not include[b, j]):
                continue
            w_gu, w_d = experts(layer * E + e)
            y[b] += gates[b, j] * swiglu(w_gu, w_d, x[b:b + 1])[0]
        if shared is not None:
            y[b] += swiglu(shared[0], shared[1], x[b:b + 1])[0]
    return y


def decode_layer_dense(x, ids, gates, layer, E, experts: RecordSource, shared=None):
    """Brute-force twin of decode_layer: every expert of the layer on every token,
    weighted by a dense [B, E] gate matrix built from the routes."""
    x = np.asarray(x, np.float64)
    ids = np.asarray(ids, np.int64)
    gates = np.asarray(gates, np.float32).astype(np.float64)
    B, k = ids.shape
    G = np.zeros((B, E))
    for b in range(B):
        for j in range(k):
            if 0 <= ids[b, j] < E:
                G[b, ids[b, j]] += gates[b, j]
    outs = np.stack([swiglu(*experts(layer * E + e), x) for e in range(E)])  # [E, B, H]
    y = np.einsum("be,ebh->bh", G, outs)
    if shared is not None:
        y = y + swiglu(shared[0], shared[1], x)
    return y


# ---------------------------------------------------------------- prefill

def prefill_layer(x, ids, gates, layer: int, E: int, experts: RecordSource,
                  return_h32: bool = False):
    """Prefill expert compute for one layer with NVFP4 activations on both GEMMs.

    x [T, H] (bf16 values) is quantised with the unit-tensor-scale activation
    quantiser; each routed expert computes g||u from the decoded fp4 activations,
    h = silu(g) * u is rounded to fp32 and quantised the same way, then
    o = W_d h_q; y[t] = sum_j gates[t,j] * o_(t,j) in route order j = 0..k-1.

    Returns (y [T, H] fp64, h_codes [T*k, I] uint8, h_scales [T*k, I/16] uint8),
    h indexed by route r = t*k + j (rows of masked routes are zero); with
    return_h32 also the fp32 h [T*k, I] that was quantised (the value whose
    distance to a rounding boundary decides a code).
    """
    x = np.asarray(x, np.float32)
    ids = np.asarray(ids, np.int64)
    T, k = ids.shape
    xc, xs = quantize_act(x)
    xq = dequant(xc, xs)
    I = experts.I
    h_codes = np.zeros((T * k, I), np.uint8)
    h_scales = np.zeros((T * k, I // 16), np.uint8)
    h32_all = np.zeros((T * k, I), np.float32) if return_h32 else None
    for e in range(E):
        t_idx, j_idx = np.nonzero(ids == e)
        if t_idx.size == 0:
            continue
        w_gu, _ = experts(layer * E + e)
        g = xq[t_idx] @ w_gu[:I].T
        u = xq[t_idx] @ w_gu[I:].T
        h32 = (silu(g) * u).astype(np.float32)
        hc, hs = quantize_act(h32)
        r = t_idx * k + j_idx
        h_codes[r] = hc
        h_scales[r] = hs
        if return_h32:
            h32_all[r] = h32
    y = prefill_from_h(h_codes, h_scales, ids, gates, layer, E, experts)
    if return_h32:
        return y, h_codes, h_scales, h32_all
    return y, h_codes, h_scales


def prefill_from_h(h_codes, h_scales, ids, gates, layer, E, experts: RecordSource):
    """Second GEMM and combine of prefill from given per-route NVFP4 h."""
    ids = np.asarray(ids, np.int64)
    gates = np.asarray(gates, np.float32).astype(np.float64)
    T, k = ids.shape
    H = experts.H
    O = np.zeros((T * k, H))
    for e in range(E):
        t_idx, j_idx = np.nonzero(ids == e)
        if t_idx.size == 0:
            continue
        _, w_d = experts(layer * E + e)
        r = t_idx * k + j_idx
        hq = dequant(h_codes[r], h_scales[r])
        O[r] = gates[t_idx, j_idx][:, None] * (hq @ w_d.T)
    y = np.zeros((T, H))
    for j in range(k):
        y += O[j::k]
    return y
