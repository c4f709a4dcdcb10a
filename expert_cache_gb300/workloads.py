"""Workload shapes and device-side setup for the routed-expert cache.

Builds the pinned host expert pool (fp32 weights drawn on the GPU by ``synth``,
quantised to NVFP4 records by ``ft_quantize_experts``, copied into pinned memory),
the device-resident shared experts, and the per-step decode inputs.  Nothing here
computes any part of the hot path.
"""
from __future__ import annotations

import numpy as np
import torch

import synth
from synth.shapes import SHAPES, Shape  # noqa: F401  (re-exported)
from . import (FT_SPLIT_FULL_OFFLOAD, FT_SPLIT_QSTAR, ExpertCache, PinnedBuffer,
               ft_moe_decode, ft_quantize_experts, ft_record_bytes)


def build_pool(seed: int, L: int, E: int, H: int, I: int, chunk_bytes: int = 1 << 30,
               device: str = "cuda", fmt: str = "nvfp4") -> PinnedBuffer:
    """Pinned host pool of L*E records (NVFP4 or MXFP4), flat id l*E + e."""
    rec = ft_record_bytes(H, I, fmt)
    n_all = L * E
    pool = PinnedBuffer(n_all * rec)
    host = pool.tensor()
    per = max(1, min(n_all, chunk_bytes // (3 * H * I * 4)))
    stage = torch.empty(per * rec, dtype=torch.uint8, device=device)
    for f0 in range(0, n_all, per):
        n = min(per, n_all - f0)
        w_gu = torch.empty((n, 2 * I, H), dtype=torch.float32, device=device)
        w_d = torch.empty((n, H, I), dtype=torch.float32, device=device)
        a, b = synth.expert_weights_batch(seed, f0, n, H, I, device)
        w_gu.copy_(a)
        w_d.copy_(b)
        del a, b
        ft_quantize_experts(w_gu, w_d, n, H, I, stage, fmt=fmt)
        host[f0 * rec:(f0 + n) * rec].copy_(stage[:n * rec])
    torch.cuda.synchronize()
    return pool


def build_shared(seed: int, L: int, H: int, I: int, device: str = "cuda",
                 fmt: str = "nvfp4") -> torch.Tensor:
    """Device records of the always-resident shared expert of each layer."""
    rec = ft_record_bytes(H, I, fmt)
    out = torch.empty(L * rec, dtype=torch.uint8, device=device)
    for l in range(L):
        a, b = synth.shared_weights(seed, l, H, I, device)
        ft_quantize_experts(a.contiguous(), b.contiguous(), 1, H, I, out[l * rec:(l + 1) * rec],
                            fmt=fmt)
    torch.cuda.synchronize()
    return out


class DecodeWorkload:
    """Resident decode inputs/outputs of a shape for `steps` steps."""

    def __init__(self, shape: Shape, seed: int = 0, steps: int | None = None, device="cuda"):
        s = shape
        self.shape = s
        self.steps = steps or s.steps
        self.trace = synth.locality_trace(seed, s.L, s.E, s.k, s.B, self.steps, s.p)
        self.gates = synth.decode_gates(seed, self.steps, s.L, s.B, s.k)
        self.ids = torch.from_numpy(self.trace).to(device)
        self.w = torch.from_numpy(self.gates).to(device)
        self.x = synth.decode_x_all(seed, self.steps, s.L, s.B, s.H, device)
        self.y = torch.empty((self.steps, s.L, s.B, s.H), dtype=torch.float32, device=device)
        self.deferred = torch.empty((self.steps, s.L, s.B, s.k), dtype=torch.int32, device=device)
        self.route_slot = torch.empty_like(self.deferred)
        self.counters = torch.empty((self.steps, s.L, 4), dtype=torch.int32, device=device)

        # raw addresses and per-(step, layer) strides: the per-layer call does integer
        # arithmetic only (no tensor views on the launch path)
        self._base = [(tsr.data_ptr(), tsr[0, 0].numel() * tsr.element_size())
                      for tsr in (self.x, self.ids, self.w, self.y, self.deferred,
                                  self.route_slot, self.counters)]

    def addresses(self, t: int, l: int):
        i = t * self.shape.L + l
        return [b + i * st for b, st in self._base]

    def run_layer(self, cache: ExpertCache, t: int, l: int, stream=None):
        s = self.shape
        x, ids, w, y, d, rs, ct = self.addresses(t, l)
        ft_moe_decode(cache.handle, l, x, ids, w, s.B, s.k, y, d, rs, ct, stream)

    def run_step(self, cache: ExpertCache, t: int, stream=None):
        for l in range(self.shape.L):
            self.run_layer(cache, t, l, stream)


class StepGraph:
    """One decode step (all L layer calls) captured as a CUDA graph over fixed
    staging buffers; `replay(t)` copies step t's inputs in, replays, and copies the
    outputs of the step back into the workload's arrays."""

    def __init__(self, wl: DecodeWorkload, cache: ExpertCache):
        self.wl, self.cache = wl, cache
        self.x = wl.x[0].clone()
        self.ids = wl.ids[0].clone()
        self.w = wl.w[0].clone()
        self.y = torch.empty_like(wl.y[0])
        self.d = torch.empty_like(wl.deferred[0])
        self.rs = torch.empty_like(wl.route_slot[0])
        self.ct = torch.empty_like(wl.counters[0])
        self.graph = None

    def capture(self):
        s = self.wl.shape
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        per = [(t.data_ptr(), t[0].numel() * t.element_size())
               for t in (self.x, self.ids, self.w, self.y, self.d, self.rs, self.ct)]
        with torch.cuda.graph(g, stream=side):
            st = torch.cuda.current_stream().cuda_stream
            for l in range(s.L):
                x, ids, w, y, d, rs, ct = [b + l * n for b, n in per]
                ft_moe_decode(self.cache.handle, l, x, ids, w, s.B, s.k, y, d, rs, ct, st)
        torch.cuda.current_stream().wait_stream(side)
        self.graph = g

    def replay(self, t: int):
        wl = self.wl
        self.x.copy_(wl.x[t], non_blocking=True)
        self.ids.copy_(wl.ids[t], non_blocking=True)
        self.w.copy_(wl.w[t], non_blocking=True)
        self.graph.replay()
        wl.y[t].copy_(self.y, non_blocking=True)
        wl.deferred[t].copy_(self.d, non_blocking=True)
        wl.route_slot[t].copy_(self.rs, non_blocking=True)
        wl.counters[t].copy_(self.ct, non_blocking=True)


def split_tuple(mode: str, f_q16: int = 65536):
    return (FT_SPLIT_FULL_OFFLOAD, 65536) if mode == "full" else (FT_SPLIT_QSTAR, int(f_q16))
