"""The bandwidth-adaptive miss split: how many of the m unique misses are filled.

TEST INFRASTRUCTURE: see the package docstring for who may import this.

Sources:
  [EXPLAINER §6.4-6.5]  residual host bandwidth B_R = max(B_H - B_P, 0);
                        T_fill(q) = qS/B_P, T_cpu(m-q) = (m-q)S/(B_H-B_P);
                        equal times give q* = m * B_P / B_H; the system takes an
                        integer with at least one fill, and q -> m when B_H <= B_P.
  [BWRATIO "第二层带宽比", "数学推导"]  the fetch fraction f = pcie_bw / cpu_bw.
  [BWRATIO "实测版本"]   measured overlap form f = p_ov / (p_ov + c_ov), which equals
                        B_P/B_H when c_ov = B_H - B_P and p_ov = B_P.
  [BWRATIO "代码全链路" §3]  the device-side integer rule in Q16 fixed point: cost(F)
                        = max(F*(1-f), (M-F)*f); of the two integer neighbours lo =
                        floor(M*f) and lo+1 take the one with the smaller cost, lo on
                        a tie; then cap at M.
  [QIITA §8]            latency(q) = max(q/B_P, (m-q)/(B_H-B_P)) and the 27.6 % loss
                        of naive rounding on the 5090 Desktop at m = 8.
  [BWRATIO "第一层带宽比"]  the backend choice from the two measured bandwidths: the
                        hybrid backend only when the CPU expert path is more than twice
                        as fast as the fill path (ratio cpu/pcie > 2), else offload.

Reading adopted where the pages differ: the [BWRATIO] Q16 rule, then the "at least
one fill" clamp of [EXPLAINER §6.5] / [JUHE] "q*：为什么不是一半给 CPU、一半给 GPU",
then the capacity clamp q <= C - |H| (the pages are silent on a cache too small to
hold the fills; it never binds at the configured sizes).
"""
from __future__ import annotations

import math

Q16 = 1 << 16


def q_rule(m: int, f_q16: int) -> int:
    """Number of fills for m unique misses at Q16 fetch fraction f_q16 (1..65536)."""
    if m <= 0:
        return 0
    if not (0 < f_q16 <= Q16):
        raise ValueError("f_q16 must be in [1, 65536]")
    lo = (m * f_q16) >> 16
    cost_lo = max(lo * (Q16 - f_q16), (m - lo) * f_q16)
    cost_hi = max((lo + 1) * (Q16 - f_q16), (m - lo - 1) * f_q16)
    fetch = lo if cost_lo <= cost_hi else lo + 1
    return min(m, max(1, fetch))


def q_for_call(m: int, n_hit: int, capacity: int, full_offload: bool, f_q16: int) -> int:
    """q for one decode call: full offload fills every miss, the hybrid split uses
    q_rule; both are capped by the slots not holding this call's hits."""
    q = m if full_offload else q_rule(m, f_q16)
    return max(0, min(q, capacity - n_hit))


def f_to_q16(f: float) -> int:
    """Q16 of a fraction in (0, 1]: floor(f * 65536 + 0.5) in fp64, capped at 65536."""
    if not (f > 0):
        raise ValueError("fraction must be > 0")
    return int(min(Q16, math.floor(min(f, 1.0) * Q16 + 0.5)))


def split_from_bandwidth(b_p: float, b_h: float) -> int:
    """f = min(1, B_P / B_H) as Q16 ([EXPLAINER §6.5]; B_H <= B_P sends every miss to the GPU)."""
    if not (b_p > 0 and b_h > 0):
        raise ValueError("bandwidths must be > 0")
    return f_to_q16(min(1.0, b_p / b_h))


def split_from_overlap(p_ov: float, c_ov: float) -> int:
    """f = p_ov / (p_ov + c_ov) as Q16 ([BWRATIO] measured-overlap form)."""
    if not (p_ov > 0 and c_ov >= 0):
        raise ValueError("p_ov must be > 0 and c_ov >= 0")
    return f_to_q16(p_ov / (p_ov + c_ov))


def q_star_continuous(m: int, b_p: float, b_h: float) -> float:
    """The closed form q* = m * B_P / B_H of [EXPLAINER §6.5]."""
    return m * b_p / b_h


def exposed_latency(q: int, m: int, b_p: float, b_h: float, s: float = 1.0) -> float:
    """max(T_fill, T_cpu) of [EXPLAINER §6.4] with the residual host bandwidth
    B_R = max(B_H - B_P, 0); a CPU share on zero residual bandwidth never ends."""
    t_fill = q * s / b_p
    if q == m:
        return t_fill
    b_r = max(b_h - b_p, 0.0)
    return math.inf if b_r <= 0 else max(t_fill, (m - q) * s / b_r)


def recommend_backend(cpu_gbs: float, pcie_gbs: float, threshold: float = 2.0) -> str:
    """[BWRATIO "第一层带宽比"]: "hybrid" when cpu_gbs > threshold * pcie_gbs, else
    "offload" (a ratio of exactly the threshold stays with offload)."""
    return "hybrid" if cpu_gbs > threshold * pcie_gbs else "offload"
