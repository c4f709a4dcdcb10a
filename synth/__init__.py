"""Seeded synthetic inputs shared by the CUDA path and the oracle.

This module holds none of the method's arithmetic: no quantiser, no cache policy,
no split rule, no expert math. It only draws numbers.

  * Gaussian-shaped values come from a counter-based generator: a 32-bit integer
    hash of (key, element index) picks one of 65,536 equiprobable N(0, 1) quantiles
    (midpoints of 65,536 equal-probability bins, computed in fp64 with
    scipy.special.ndtri and rounded once to fp32).  Each 32-bit hash feeds two
    elements (its low and high 16 bits).  Only integer ops and a table gather are
    involved, so the same key gives bit-identical values on the CPU and on a GPU,
    which lets the oracle regenerate any single expert of a pool the GPU built.
  * Routing traces and decode gates use numpy's default_rng (small arrays, CPU).

Streams (the `stream` argument of `key`):
  1 routed expert weights (index = flat id, sub 0 = W_gu, 1 = W_d), std 0.02
  2 shared expert weights (index = layer), std 0.02
  3 decode activations (index = step * L + layer), std 1, rounded to bf16
  4 prefill activations (index = layer), std 1, rounded to bf16
  5 prefill router logits (index = layer)
"""
from __future__ import annotations

import functools

import numpy as np
import torch

MASK32 = 0xFFFFFFFF


def _splitmix64(z: int) -> int:
    z = (z + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    return z ^ (z >> 31)


def key(seed: int, stream: int, index: int, sub: int = 0) -> tuple[int, int]:
    """Two 32-bit keys for one generated tensor."""
    z = _splitmix64(_splitmix64(_splitmix64(_splitmix64(seed) ^ stream) ^ index) ^ sub)
    return z & MASK32, (z >> 32) & MASK32


def _hash32(x: torch.Tensor) -> torch.Tensor:
    """Bijective 32-bit integer mixer on int64 tensors holding values < 2^32.
    Multipliers are < 2^31 so no product overflows int64."""
    x = x ^ (x >> 16)
    x = (x * 0x7FEB352D) & MASK32
    x = x ^ (x >> 15)
    x = (x * 0x5BD1E995) & MASK32
    return x ^ (x >> 16)


@functools.lru_cache(maxsize=None)
def _quantile_table_np(scale: float) -> np.ndarray:
    from scipy.special import ndtri
    p = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
    return (scale * ndtri(p)).astype(np.float32)


_TABLES: dict = {}


def _table(scale: float, device) -> torch.Tensor:
    k = (scale, str(device))
    if k not in _TABLES:
        _TABLES[k] = torch.from_numpy(_quantile_table_np(scale)).to(device)
    return _TABLES[k]


def gaussian_indices(keys: tuple[int, int], n: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """16-bit quantile indices (int64) of elements offset .. offset+n-1 of a stream."""
    assert n % 2 == 0 and offset % 2 == 0
    k1, k2 = keys
    i = torch.arange(offset // 2, (offset + n) // 2, dtype=torch.int64, device=device)
    h = _hash32(_hash32(i ^ k1) ^ k2)
    return torch.stack((h & 0xFFFF, h >> 16), dim=1).reshape(-1)


def gaussian(keys, shape, std: float, device="cpu") -> torch.Tensor:
    """fp32 tensor of the given shape, N(0, std^2)-shaped, bit-identical on any device."""
    n = int(np.prod(shape))
    idx = gaussian_indices(keys, n + (n & 1), device)[:n]
    return _table(std, device)[idx].reshape(shape)


def gaussian_batch(key_list, shape, std: float, device="cpu") -> torch.Tensor:
    """Stack of gaussian(keys, shape) for every keys pair of key_list, in one pass."""
    n = int(np.prod(shape))
    assert n % 2 == 0
    k = torch.tensor(key_list, dtype=torch.int64, device=device)      # [m, 2]
    i = torch.arange(n // 2, dtype=torch.int64, device=device)[None, :]
    h = _hash32(_hash32(i ^ k[:, :1]) ^ k[:, 1:])
    idx = torch.stack((h & 0xFFFF, h >> 16), dim=2).reshape(len(key_list), n)
    return _table(std, device)[idx].reshape((len(key_list),) + tuple(shape))


# ------------------------------------------------------------- weights / inputs

def expert_weights(seed: int, flat_id: int, H: int, I: int, device="cpu"):
    """(W_gu [2I, H], W_d [H, I]) fp32, N(0, 0.02^2)-shaped, for one routed expert."""
    return (gaussian(key(seed, 1, flat_id, 0), (2 * I, H), 0.02, device),
            gaussian(key(seed, 1, flat_id, 1), (H, I), 0.02, device))


def expert_weights_batch(seed: int, flat0: int, n: int, H: int, I: int, device="cpu"):
    """expert_weights of flat ids flat0 .. flat0+n-1 as [n, 2I, H] and [n, H, I]."""
    return (gaussian_batch([key(seed, 1, f, 0) for f in range(flat0, flat0 + n)], (2 * I, H), 0.02, device),
            gaussian_batch([key(seed, 1, f, 1) for f in range(flat0, flat0 + n)], (H, I), 0.02, device))


def shared_weights(seed: int, layer: int, H: int, I: int, device="cpu"):
    return (gaussian(key(seed, 2, layer, 0), (2 * I, H), 0.02, device),
            gaussian(key(seed, 2, layer, 1), (H, I), 0.02, device))


def decode_x(seed: int, step: int, layer: int, L: int, B: int, H: int, device="cpu"):
    """bf16 [B, H] activations of one (step, layer), N(0, 1)-shaped."""
    return gaussian(key(seed, 3, step * L + layer), (B, H), 1.0, device).to(torch.bfloat16)


def decode_x_all(seed: int, steps: int, L: int, B: int, H: int, device="cpu"):
    """decode_x of every (step, layer) as one bf16 [steps, L, B, H] tensor."""
    keys = [key(seed, 3, t * L + l) for t in range(steps) for l in range(L)]
    return gaussian_batch(keys, (B, H), 1.0, device).to(torch.bfloat16).reshape(steps, L, B, H)


def prefill_x(seed: int, layer: int, T: int, H: int, device="cpu"):
    return gaussian(key(seed, 4, layer), (T, H), 1.0, device).to(torch.bfloat16)


def prefill_routes(seed: int, layer: int, T: int, E: int, k: int, device="cpu"):
    """Top-k of N(0,1)-shaped router logits [T, E] (ties -> lower expert id) and
    the fp32 softmax of the k selected logits (computed in fp64 on the CPU).
    Returns (ids int32 [T, k] on `device`, gates fp32 [T, k] on `device`)."""
    idx = gaussian_indices(key(seed, 5, layer), T * E + ((T * E) & 1), device)[:T * E]
    idx = idx.reshape(T, E)
    e = torch.arange(E, device=device, dtype=torch.int64)
    order_key = idx * E + (E - 1 - e)            # unique per row, larger = larger logit
    top = torch.topk(order_key, k, dim=1, largest=True, sorted=True).indices
    logits = _table(1.0, device)[torch.gather(idx, 1, top)]
    lg = logits.cpu().numpy().astype(np.float64)
    ex = np.exp(lg - lg.max(axis=1, keepdims=True))
    gates = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    return top.to(torch.int32), torch.from_numpy(gates).to(device)


def locality_trace(seed: int, L: int, E: int, k: int, B: int, steps: int, p: float) -> np.ndarray:
    """Routing trace int32 [steps, L, B, k] with short-term locality.

    Each (layer, token) keeps a working set of k distinct ids; every step each
    position is kept with probability p and otherwise replaced by a uniform id
    that is not already in the set.  The row is emitted after the update.
    """
    rng = np.random.default_rng([seed, 0])
    work = np.empty((L, B, k), np.int64)
    for l in range(L):
        for b in range(B):
            work[l, b] = rng.choice(E, k, replace=False)
    out = np.empty((steps, L, B, k), np.int32)
    for t in range(steps):
        for l in range(L):
            for b in range(B):
                row = work[l, b]
                u = rng.random(k)
                for j in range(k):
                    if u[j] > p:
                        while True:
                            c = int(rng.integers(0, E))
                            if c not in row:
                                break
                        row[j] = c
                out[t, l, b] = row
    return out


def decode_gates(seed: int, steps: int, L: int, B: int, k: int) -> np.ndarray:
    """fp32 [steps, L, B, k]: softmax (fp64) of k standard normals, rounded to fp32."""
    rng = np.random.default_rng([seed, 3])
    z = rng.standard_normal((steps, L, B, k))
    ex = np.exp(z - z.max(axis=-1, keepdims=True))
    return (ex / ex.sum(axis=-1, keepdims=True)).astype(np.float32)
