"""Static expert placement vs the global LRU: miss rates on one layer's trace.

TEST INFRASTRUCTURE: see the package docstring for who may import this.

Sources:
  [QIITA §5]         llama.cpp fixes tensor placement at load time, KTransformers
                     pins the frequently used experts at prefill time; both are
                     static.  The article's simulation fixes the top-`cap` experts
                     by frequency over the first 512 steps and never changes them,
                     and compares that with an LRU over the unique ids of each step.
                     With locality LRU wins by a wide margin; with no locality LRU
                     is slightly worse.
  [EXPLAINER §11.2]  global LRU 16 % vs prefill-time placement 41 % vs static 62 %
                     (Qwen3.6 routing replay; the traces are not available).

Miss rate = misses / unique (per step) accesses, over every step of the trace.
"""
from __future__ import annotations

import numpy as np

from .lru import SlotCache


def static_resident(trace: np.ndarray, E: int, cap: int, warm: int = 512) -> set:
    """The `cap` most frequent ids over the first `warm` steps (ties: lower id)."""
    counts = np.bincount(np.asarray(trace[:warm]).reshape(-1), minlength=E)
    order = np.lexsort((np.arange(E), -counts))
    return set(int(e) for e in order[:cap])


def static_miss_rate(trace: np.ndarray, E: int, cap: int, warm: int = 512) -> float:
    resident = static_resident(trace, E, cap, warm)
    acc = miss = 0
    for row in np.asarray(trace):
        for e in set(int(v) for v in row):
            acc += 1
            miss += e not in resident
    return miss / acc


def lru_miss_rate(trace: np.ndarray, E: int, cap: int) -> float:
    """Miss rate of the global LRU slot cache (one layer, full offload: q = m)."""
    cache = SlotCache(1, E, cap, full_offload=True)
    acc = miss = 0
    for row in np.asarray(trace):
        r = cache.decode(0, np.asarray(row)[None, :])
        acc += r.n_hit + r.m
        miss += r.m
    return miss / acc
