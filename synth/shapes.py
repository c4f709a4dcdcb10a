"""Workload shapes: layer counts, sizes, capacities, batch, step counts and the
locality of the synthetic routing traces.  Plain data (no arithmetic of the method,
no device code), so both the CUDA path's harness and the CPU oracle's timing read
the same shapes without loading the CUDA library."""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass
class Shape:
    name: str
    L: int
    E: int
    k: int
    H: int
    I: int
    C: int
    B: int = 1
    steps: int = 256
    p: float = 0.8
    shared: bool = False
    T: int = 0
    resize: dict = field(default_factory=dict)   # step -> new capacity


# The workloads: a tiny parity case, Qwen3.6-35B-A3B-shaped decode and prefill,
# DeepSeek-V4-Flash-shaped decode, and the elastic stress run.
SHAPES = {
    "tiny": Shape("tiny", L=2, E=16, k=2, H=64, I=32, C=8, B=1, steps=32, p=0.8),
    "qwen_decode": Shape("qwen_decode", L=40, E=256, k=8, H=2048, I=512, C=600, B=1,
                         steps=256, p=0.8, shared=True),
    "dsv4_decode": Shape("dsv4_decode", L=16, E=256, k=6, H=4096, I=2048, C=1024, B=1,
                         steps=256, p=0.8),
    "qwen_prefill": Shape("qwen_prefill", L=40, E=256, k=8, H=2048, I=512, C=600, T=8192),
    # the same prefill layer (8192 tokens over 256 experts) for two layers only:
    # profiling captures of the prefill kernels that hold about 2 GB on the device
    "qwen_prefill_small": Shape("qwen_prefill_small", L=2, E=256, k=8, H=2048, I=512, C=512, T=8192),
    # the Qwen-shaped layer over a small pool (4 x 64 experts, 64 slots): profiling
    # captures of the decode kernel that hold a few hundred MB on the device
    "qwen_decode_small": Shape("qwen_decode_small", L=4, E=64, k=8, H=2048, I=512, C=64, B=1,
                               steps=24, p=0.8, shared=True),
    "stress": Shape("stress", L=16, E=256, k=6, H=4096, I=2048, C=1024, B=16, steps=512,
                    p=0.3, resize={171: 256, 342: 768}),
}
