"""Benchmark of the routed-expert cache hot path on one GB300 (or N replicas).

Headline workload: Qwen3.6-35B-A3B-shaped decode (40 MoE layers x 256 routed experts,
top-8 + 1 shared expert, hidden 2048, intermediate 512, NVFP4 records in a pinned host
pool, 600-slot global LRU cache, batch 1, locality p = 0.8, full offload q = m).
A step is one decode token: all 40 layer calls (remap, load-through fills, gate/up,
down + gated combine), replayed as one CUDA graph.  Inputs are resident in HBM; `e2e`
times the same steps with each step's inputs copied from pinned host memory and y
copied back inside the timed region.  The device-timed pass and the e2e pass are
repeated (interleaved) and the medians reported with their spread.

Further lines in the same JSON object:
  prefill   the Qwen-shaped 8192-token chunk (40 layers) with and without the
            full-layer double buffer, interleaved with copy-only passes of the same
            bytes, plus the host-to-device rate of every 1 GiB window of the pool;
  legs      decode at the other benchmarked points: Qwen-shaped p in {0.5, 0.8,
            0.95} x {q = m, q*}; DeepSeek-V4-Flash-shaped B in {1, 4} x f in
            {2/3, 1/2, 1/4}; the elastic stress run (B 16, p 0.3, 512 steps, resized
            1024 -> 256 -> 768 slots), each with its roofline fraction;
  cpu_baseline  the CPU oracle on the host cores (one core, and all cores).
`--impl reference` times the CPU oracle alone (all host cores), whole tokens.

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE decode tok/s & prefill tok/s; % of HBM/PCIe/FP4 roofline"
HEADLINE = "qwen_decode"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=32)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--workload", default=HEADLINE, help="headline decode workload")
    ap.add_argument("--repeats", type=int, default=5, help="interleaved device / e2e passes")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-legs", action="store_true")
    ap.add_argument("--prefill-pairs", type=int, default=5)
    ap.add_argument("--prefill-workload", default="qwen_prefill")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prefill workload (its own pool; for profiling captures)")
    ap.add_argument("--oracle-workers", type=int, default=0, help="0: every host core")
    return ap.parse_args()


# ----------------------------------------------------------------- distributed

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons sampled every 200 ms."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 6:
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[2 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ----------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# From the ncu capture of decode_layer_kernel on qwen_decode_small (profiles/): DRAM
# bytes read per algorithmic HBM byte, the median of the captured launches.
DRAM_READ_PER_ALGORITHMIC_BYTE = 1.013


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def med_spread(xs):
    m = statistics.median(xs)
    return m, (max(xs) - min(xs)) / m if m else 0.0


def config_of(s, split_name, f_q16, rec_bytes):
    return {"workload": s.name, "L": s.L, "E": s.E, "top_k": s.k, "shared_expert": s.shared,
            "H": s.H, "I": s.I, "capacity": s.C, "B": s.B, "locality_p": s.p,
            "split": split_name, "f_q16": f_q16, "parallelism": "replicas",
            "l2": "inputs larger than L2 (slot cache %.2f GB, host pool %.1f GB)"
                  % (s.C * rec_bytes / 1e9, s.L * s.E * rec_bytes / 1e9)}


# ----------------------------------------------------------------- CPU oracle timing
# Worker processes (spawned, one BLAS thread each) hold the pool records of the layers
# assigned to them; the parent runs the state oracle (LRU + q rule) and hands each
# layer call's output computation (fp64 decode of every expert it reads + the dense
# SwiGLU definition) to the worker of that layer.  The record encoding is the pool
# being built (an input), done before the timed region.

_W = {}


def _worker_init(seed, H, I, L, E, shared):
    import synth
    from oracle.formats import decode_record, encode_record
    _W.update(seed=seed, H=H, I=I, L=L, E=E, recs={}, shared={}, has_shared=shared,
              enc=encode_record, dec=decode_record, synth=synth)


def _worker_prepare(items):
    """items: (layer, flat ids) whose records (and shared experts) this worker needs."""
    w = _W
    for l, flats in items:
        for f in flats:
            if f not in w["recs"]:
                w["recs"][f] = w["enc"](*[a.numpy() for a in w["synth"].expert_weights(w["seed"], f, w["H"], w["I"])])
        if w["has_shared"] and l not in w["shared"]:
            w["shared"][l] = w["enc"](*[a.numpy() for a in w["synth"].shared_weights(w["seed"], l, w["H"], w["I"])])
    return len(w["recs"])


def _worker_call(l, x, ids, gates):
    """One layer call's output through the oracle, timed: (y, seconds)."""
    from oracle.moe import RecordSource, decode_layer
    w = _W
    t0 = time.perf_counter()
    src = RecordSource(lambda f: w["recs"][f], w["H"], w["I"])      # fresh: decodes every expert
    sh = w["dec"](w["shared"][l], w["H"], w["I"]) if w["has_shared"] else None
    y = decode_layer(x, ids, gates, l, w["E"], src, sh)
    return y, time.perf_counter() - t0


class OraclePool:
    """n spawned single-threaded workers; layer l goes to worker l mod n."""

    def __init__(self, n, seed, s):
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        env = {"OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}
        old = {k: os.environ.get(k) for k in env}
        os.environ.update(env)
        ctx = mp.get_context("spawn")
        self.n = n
        self.ex = [ProcessPoolExecutor(1, mp_context=ctx, initializer=_worker_init,
                                       initargs=(seed, s.H, s.I, s.L, s.E, s.shared))
                   for _ in range(n)]
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v

    def prepare(self, s, trace):
        per = [[] for _ in range(self.n)]
        for l in range(s.L):
            flats = sorted({l * s.E + int(e) for e in trace[:, l].reshape(-1)})
            per[l % self.n].append((l, flats))
        futs = [ex.submit(_worker_prepare, items) for ex, items in zip(self.ex, per)]
        return sum(f.result() for f in futs)

    def submit(self, l, x, ids, gates):
        return self.ex[l % self.n].submit(_worker_call, l, x, ids, gates)

    def close(self):
        for ex in self.ex:
            ex.shutdown(wait=True)


def oracle_tokens(s, seed, n_workers, tokens, warmup=0, budget_s=None):
    """Whole decode tokens through the oracle: per token, the state oracle for its L
    layer calls (parent) and their outputs (workers, in parallel).  Returns a dict
    with the wall seconds of each timed token and the per-call compute seconds."""
    import synth
    from oracle.lru import SlotCache
    total = warmup + tokens
    trace = synth.locality_trace(seed, s.L, s.E, s.k, s.B, total, s.p)
    gates = synth.decode_gates(seed, total, s.L, s.B, s.k)
    pool = OraclePool(n_workers, seed, s)
    t_prep = time.perf_counter()
    pool.prepare(s, trace)
    t_prep = time.perf_counter() - t_prep
    cache = SlotCache(s.L, s.E, s.C)
    walls, calls = [], []
    t_all = time.perf_counter()
    for t in range(total):
        xs = [synth.decode_x(seed, t, l, s.L, s.B, s.H).float().numpy() for l in range(s.L)]
        t0 = time.perf_counter()
        futs = []
        for l in range(s.L):
            cache.decode(l, trace[t, l])
            futs.append(pool.submit(l, xs[l], trace[t, l], gates[t, l]))
        res = [f.result() for f in futs]
        wall = time.perf_counter() - t0
        if t >= warmup:
            walls.append(wall)
            calls.extend(r[1] for r in res)
        if budget_s is not None and t >= warmup and time.perf_counter() - t_all > budget_s:
            break
    pool.close()
    return {"walls": walls, "calls": calls, "prepare_s": t_prep}


def oracle_calls_single_core(s, seed, budget_s):
    """One worker, layer calls one after another: seconds per layer call."""
    import synth
    total = 4
    trace = synth.locality_trace(seed, s.L, s.E, s.k, s.B, total, s.p)
    gates = synth.decode_gates(seed, total, s.L, s.B, s.k)
    pool = OraclePool(1, seed, s)
    n_calls = max(1, min(total * s.L, int(budget_s / 0.25)))
    pool.prepare(s, trace[: (n_calls + s.L - 1) // s.L])
    spent, calls = 0.0, 0
    for i in range(total * s.L):
        t, l = divmod(i, s.L)
        x = synth.decode_x(seed, t, l, s.L, s.B, s.H).float().numpy()
        _, sec = pool.submit(l, x, trace[t, l], gates[t, l]).result()
        spent += sec
        calls += 1
        if spent > budget_s or calls >= n_calls:
            break
    pool.close()
    return spent / calls, calls


def cpu_baseline(s, seed, n_workers):
    sec_call, n_calls = oracle_calls_single_core(s, seed, budget_s=15.0)
    r = oracle_tokens(s, seed, n_workers, tokens=3, warmup=0)
    tok_s = s.B * len(r["walls"]) / sum(r["walls"])
    return {"value": tok_s, "unit": "tok/s", "cores": n_workers, "kind": "oracle",
            "sample": (f"{len(r['walls'])} whole decode tokens of {s.name} ({s.L} layer calls "
                       f"each: state oracle in order, fp64 outputs of the layer calls on "
                       f"{n_workers} worker processes at once), records encoded beforehand"),
            "cpu_model": cpu_model(), "blas_threads_per_worker": 1,
            "single_core": {"value": s.B / (sec_call * s.L), "unit": "tok/s", "cores": 1,
                            "blas_threads": 1,
                            "sample": f"{n_calls} decode layer calls one after another, "
                                      f"{sec_call * 1e3:.0f} ms each, x {s.L} layers per token"}}


# ----------------------------------------------------------------- native decode

def decode_counts(wl, t0, t1, rec_bytes, shared):
    import numpy as np
    ct = wl.counters[t0:t1].cpu().numpy().astype(np.int64)   # [K, L, 4]
    n_hit, n_miss, n_fill = ct[..., 0].sum(), ct[..., 1].sum(), ct[..., 2].sum()
    n_shared = (t1 - t0) * wl.shape.L if shared else 0
    return {"hits": int(n_hit), "misses": int(n_miss), "fills": int(n_fill),
            "deferred_routes": int(ct[..., 3].sum()),
            "hbm_bytes": int((n_hit + n_shared) * rec_bytes), "link_bytes": int(n_fill * rec_bytes)}


def roofline_ms(cnt, hbm_gbs, b_p):
    """Decode roofline: hit (+ shared) records at HBM bandwidth + fills at B_P."""
    return (cnt["hbm_bytes"] / (hbm_gbs * 1e9) + cnt["link_bytes"] / (b_p * 1e9)) * 1e3


class DecodeRun:
    """A decode workload over one cache: reset + warm-up + timed graph replays."""

    def __init__(self, ft, wlm, s, pool_ptr, shared, split, seed, steps, fmt="nvfp4", host_threads=0):
        self.ft, self.s = ft, s
        self.cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool_ptr, shared=shared,
                                    split=split, capacity_max=max([s.C] + list(s.resize.values())),
                                    fmt=fmt)
        self.host = None
        if host_threads:
            # the host share of every call computed by a pinned worker pool and joined into y
            self.host = ft.HostBranch(s.L, s.E, s.H, s.I, s.k, s.B, pool_ptr, host_threads, fmt=fmt)
            ft.ft_cache_set_host_branch(self.cache.handle, self.host.handle)
        self.wl = wlm.DecodeWorkload(s, seed=seed, steps=steps)
        self.graph = wlm.StepGraph(self.wl, self.cache)
        self.steps = steps

    def reset(self, capacity=None):
        c = capacity or self.s.C
        self.ft.ft_cache_resize(self.cache.handle, c, self.cache.slot_buf)
        self.graph.graph = None                      # the captured args carry C

    def run(self, t0, t1, graph=True):
        for t in range(t0, t1):
            if t in self.s.resize:
                self.reset(self.s.resize[t])
            if graph:
                if self.graph.graph is None:
                    self.graph.capture()
                self.graph.replay(t)
            else:
                self.wl.run_step(self.cache, t)

    def warm(self, warmup):
        """Emptied cache, warm-up steps 0..warmup-1: eager, then (after the graph is
        captured) the last one as a replay, so the timed replays run an uploaded graph."""
        self.reset()
        self.run(0, max(warmup - 1, 0), graph=False)
        if self.graph.graph is None:
            self.graph.capture()
        if warmup > 0:
            self.graph.replay(warmup - 1)

    def timed(self, warmup, world, stream):
        import torch
        self.warm(warmup)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        self.run(warmup, self.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1)

    def profiled(self, warmup):
        """Same steps eagerly with CUDA events around each decode launch."""
        import torch
        ft = self.ft
        self.reset()
        self.run(0, warmup, graph=False)
        ft.ft_profile_enable(self.cache.handle, 1)
        ft.ft_profile_read(self.cache.handle)
        self.run(warmup, self.steps, graph=False)
        torch.cuda.synchronize()
        prof = ft.ft_profile_read(self.cache.handle)
        ft.ft_profile_enable(self.cache.handle, False)
        return prof["decode"]

    def e2e(self, warmup, world, stream):
        """Step inputs H2D from pinned host memory and y D2H inside the timed region."""
        import torch
        wl, g = self.wl, self.graph
        hx = wl.x.cpu().pin_memory()
        hid = wl.ids.cpu().pin_memory()
        hw = wl.w.cpu().pin_memory()
        hy = torch.empty(wl.y.shape, dtype=wl.y.dtype).pin_memory()
        self.warm(warmup)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for t in range(warmup, self.steps):
            g.x.copy_(hx[t], non_blocking=True)
            g.ids.copy_(hid[t], non_blocking=True)
            g.w.copy_(hw[t], non_blocking=True)
            g.graph.replay()
            hy[t].copy_(g.y, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        h2d = g.x.numel() * g.x.element_size() + g.ids.numel() * 4 + g.w.numel() * 4
        return e0.elapsed_time(e1), h2d, g.y.numel() * 4

    def close(self):
        if self.host is not None:
            self.ft.ft_cache_set_host_branch(self.cache.handle, None)
        self.cache.close()
        if self.host is not None:
            self.host.close()


def busy_host_leg(ft, wlm, s, pool_ptr, shared, seed, rec_bytes, hbm_gbs, b_p, world, stream, n_threads):
    """Full offload (the headline's split) with n_threads host workers spinning on their
    cores and no branch attached: what idle host cores cost the host link's fills."""
    spin = ft.HostBranch(s.L, s.E, s.H, s.I, s.k, s.B, pool_ptr, n_threads, mailbox=False)
    try:
        leg = decode_leg(ft, wlm, s, pool_ptr, shared, "full", 65536, seed, 32, 256, rec_bytes, hbm_gbs, b_p,
                         world, stream)
    finally:
        spin.close()
    leg["note"] = (f"{n_threads} host worker threads spinning on their cores during the run (nothing "
                   "computed on the host); compare qwen_p0.8_full")
    return leg


def bandwidth_profile(ft, s, pool, shared, n_threads, n_records=64):
    """The two miss paths of this machine over n_records records of the pool: the GPU
    gather (fill path) and the host branch's GEMV, alone and together; the backend rule
    and the overlap split (ft_profile_bandwidth)."""
    cache = ft.ExpertCache(s.L, s.E, s.H, s.I, s.k, s.B, s.C, pool.ptr, shared=shared)
    hb = ft.HostBranch(s.L, s.E, s.H, s.I, s.k, s.B, pool.ptr, n_threads, mailbox=False)
    prof = ft.ft_profile_bandwidth(cache.handle, hb.handle, n_records)
    cache.close()
    hb.close()
    prof["host_threads"] = n_threads
    prof["recommend"] = "hybrid" if prof["recommend"] == ft.FT_BACKEND_HYBRID else "offload"
    prof["f_overlap"] = prof["f_q16"] / 65536
    prof["ratio_cpu_over_pcie"] = prof["cpu_gbs"] / prof["pcie_gbs"]
    prof["note"] = ("record bytes per second: pcie = GPU gather of the records from the pinned pool "
                    "into slots, cpu = the host branch computing one token through each record; "
                    "ov = both at once; hybrid iff cpu > 2 x pcie; f = pcie_ov / (pcie_ov + cpu_ov)")
    return prof


def measure_b_p(ft, pool, torch):
    """B_P: best of 5 copies of the pool's first 1 GiB, and one copy of every 1 GiB
    window of the pool (GB/s), pinned host -> device."""
    GiB = 1 << 30
    n = min(GiB, pool.nbytes)
    dev = torch.empty(n, dtype=torch.uint8, device="cuda")
    best = ft.ft_measure_h2d(pool.ptr, dev, n, 5)
    win = [round(ft.ft_measure_h2d(pool.ptr + off, dev, n, 1), 1)
           for off in range(0, pool.nbytes - n + 1, n)]
    del dev
    return best, win


def pool_numa(pool):
    """The pool mapping's NUMA placement as the kernel reports it (numa_maps)."""
    try:
        addr = "%x" % pool.ptr
        with open("/proc/self/numa_maps") as fh:
            for line in fh:
                if line.split()[0] == addr:
                    return " ".join(w for w in line.split()[1:] if w.startswith(("N", "kernelpagesize")))
    except OSError:
        pass
    return None


def native(args, rank, world):
    import torch
    import expert_cache_gb300 as ft
    from expert_cache_gb300 import workloads as wlm
    from dataclasses import replace

    hbm_gbs, _, peak_src = peaks()
    stream = torch.cuda.current_stream()
    s = wlm.SHAPES[args.workload]
    rec_bytes = ft.ft_record_bytes(s.H, s.I)
    t_build = time.perf_counter()
    pool = wlm.build_pool(args.seed, s.L, s.E, s.H, s.I)
    shared = wlm.build_shared(args.seed, s.L, s.H, s.I)
    t_build = time.perf_counter() - t_build
    b_p, b_p_windows = measure_b_p(ft, pool, torch)
    f_half = ft.ft_split_from_bandwidth(b_p, 2.0 * b_p)        # B_H = 2 B_P  ->  f = 1/2

    out = {}
    # ---- prefill first (same pool shape: 40 x 256 experts, H 2048, I 512)
    pf = None
    if not args.no_prefill:
        pf = native_prefill(args, ft, wlm, pool, b_p, world)
        pf["mxfp4"] = prefill_mx_leg(args, ft, wlm, world)

    # ---- headline: interleaved device-timed and e2e passes
    steps = args.warmup + args.steps
    run = DecodeRun(ft, wlm, s, pool.ptr, shared, wlm.split_tuple("full"), args.seed, steps)
    dev_ms, e2e_ms = [], []
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(args.repeats):
            dev_ms.append(max_over_ranks(run.timed(args.warmup, world, stream), world))
            if not args.no_e2e:
                ms, h2d, d2h = run.e2e(args.warmup, world, stream)
                e2e_ms.append(max_over_ranks(ms, world))
    cnt = decode_counts(run.wl, args.warmup, steps, rec_bytes, s.shared)
    t_dec_ms, n_dec = run.profiled(args.warmup)
    cnt_p = decode_counts(run.wl, args.warmup, steps, rec_bytes, s.shared)
    assert cnt_p == cnt, "the profiled pass made different decisions"
    assert ft.ft_cache_status(run.cache.handle) == 0
    run.close()

    ms, spread = med_spread(dev_ms)
    tok = args.steps * s.B * world
    roof_ms = roofline_ms(cnt, hbm_gbs, b_p)
    per_launch = (cnt["hbm_bytes"] + cnt["link_bytes"]) / n_dec
    t_launch = t_dec_ms / 1e3 / n_dec
    eff_peak = (cnt["hbm_bytes"] + cnt["link_bytes"]) / (roof_ms / 1e3)
    out.update({
        "metric": METRIC,
        "value": tok / (ms / 1e3),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 weights x bf16 activations, f32 accumulate",
        "data": "synthetic",
        "config": config_of(s, "full", 65536, rec_bytes),
        "repeats": {"device_ms": [round(v, 3) for v in dev_ms],
                    "e2e_ms": [round(v, 3) for v in e2e_ms],
                    "median_ms": ms, "spread": spread,
                    "order": "device, e2e, device, e2e, ... (each from an emptied cache)"},
        "decode_roofline": {"ms_per_step_roofline": roof_ms / args.steps,
                            "frac": roof_ms / ms,
                            "b_p_gbs": b_p, "hbm_gbs": hbm_gbs, "hbm_source": peak_src,
                            "hits_per_step": cnt["hits"] / args.steps,
                            "misses_per_step": cnt["misses"] / args.steps,
                            "fills_per_step": cnt["fills"] / args.steps,
                            "miss_rate": cnt["misses"] / max(cnt["hits"] + cnt["misses"], 1)},
        "roofline": {
            "kernel": "decode_layer_kernel (decision, hits from HBM, fills load-through from "
                      "pinned host, down, combine, table update)",
            "bound": "hbm",
            "achieved": per_launch / t_launch / 1e9,
            "peak": eff_peak / 1e9,
            "unit": "GB/s",
            "frac": (per_launch / t_launch) / eff_peak,
            "traffic": DRAM_READ_PER_ALGORITHMIC_BYTE * cnt["hbm_bytes"] / n_dec,
            "traffic_note": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of decode_layer_kernel "
                             "on workload qwen_decode_small (read = %.3f x algorithmic HBM bytes, "
                             "write 0), scaled to this run's HBM bytes per launch"
                             % DRAM_READ_PER_ALGORITHMIC_BYTE),
            "peak_note": (f"byte-mix peak of this kernel: HBM bytes at {hbm_gbs:.0f} GB/s ({peak_src} "
                          f"MEASURED_PEAKS hbm_gbs) plus host-link bytes at B_P = {b_p:.1f} GB/s "
                          "measured in this run; duration from CUDA events around each launch "
                          "of an eager pass over the same steps"),
            "hbm_bytes_per_launch": cnt["hbm_bytes"] / n_dec,
            "link_bytes_per_launch": cnt["link_bytes"] / n_dec,
        },
        "kernels": {"decode_layer_kernel": {"ms_total": t_dec_ms, "launches": n_dec,
                                            "us_per_launch": t_launch * 1e6}},
        "gpu_launches": args.steps * s.L,
        "step_execution": "one CUDA graph replay per step (%d layer calls, one kernel each)" % s.L,
        "clocks": clk.summary(),
        "host_link": {"b_p_gbs": b_p, "b_p_source": "best of 5 copies of the pool's first 1 GiB",
                      "b_p_windows_gbs": b_p_windows, "pool_numa": pool_numa(pool),
                      "pool_build_s": round(t_build, 1)},
    })
    if e2e_ms:
        em, esp = med_spread(e2e_ms)
        out["e2e"] = {"value": tok / (em / 1e3), "unit": "tok/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "spread": esp,
                      "note": "median of passes interleaved with the device-timed ones"}
    if pf is not None:
        out["prefill"] = pf
    if not args.no_legs:
        legs = {}
        for p in (0.5, 0.8, 0.95):
            for mode in ("full", "qstar"):
                sp = replace(s, p=p)
                f = 65536 if mode == "full" else f_half
                legs[f"qwen_p{p}_{mode}"] = decode_leg(ft, wlm, sp, pool.ptr, shared, mode, f,
                                                       args.seed, 32, 256, rec_bytes, hbm_gbs,
                                                       b_p, world, stream)
        # the host share computed as well (end to end), and the bandwidth profile that
        # picks the backend and the split on this machine
        n_host = max(1, cpu_cores() - 1)
        for p in (0.5, 0.8):
            sp = replace(s, p=p)
            legs[f"qwen_p{p}_qstar_hybrid"] = decode_leg(ft, wlm, sp, pool.ptr, shared, "qstar", f_half,
                                                         args.seed, 32, 256, rec_bytes, hbm_gbs, b_p,
                                                         world, stream, host_threads=n_host)
        # the same full-offload decode while the host's cores are busy (the branch's
        # workers spinning, nothing attached): the host link's fills depend on it
        legs["qwen_p0.8_full_busy_host"] = busy_host_leg(ft, wlm, replace(s, p=0.8), pool.ptr, shared, args.seed,
                                                         rec_bytes, hbm_gbs, b_p, world, stream, n_host)
        bw = bandwidth_profile(ft, s, pool, shared, n_host)
        out["bandwidth_profile"] = bw
        sp = replace(s, p=0.8)
        legs["qwen_p0.8_profiled_split_hybrid"] = decode_leg(
            ft, wlm, sp, pool.ptr, shared, "qstar", max(1, bw["f_q16"]), args.seed, 32, 256, rec_bytes,
            hbm_gbs, b_p, world, stream, host_threads=n_host)
        out["legs"] = legs
    del shared
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = args.oracle_workers or cpu_cores()
        out["cpu_baseline"] = cpu_baseline(s, args.seed, n)
    pool.free()
    if not args.no_legs:
        out["legs"].update(dsv4_legs(args, ft, wlm, hbm_gbs, world, stream))
    return out


def decode_leg(ft, wlm, s, pool_ptr, shared, mode, f_q16, seed, warmup, steps, rec_bytes,
               hbm_gbs, b_p, world, stream, fmt="nvfp4", host_threads=0):
    run = DecodeRun(ft, wlm, s, pool_ptr, shared, wlm.split_tuple(mode, f_q16), seed,
                    warmup + steps, fmt=fmt, host_threads=host_threads)
    ms = max_over_ranks(run.timed(warmup, world, stream), world)
    cnt = decode_counts(run.wl, warmup, warmup + steps, rec_bytes, s.shared)
    status = ft.ft_cache_status(run.cache.handle)
    host = None
    if run.host is not None:
        jobs, mailbox_jobs = ft.ft_host_branch_stats(run.host.handle)
        host = {"threads": host_threads, "calls_joined": mailbox_jobs,
                "note": "y includes the host share: deferred routes computed by the host branch "
                        "concurrently with the GPU share and added by the join kernel"}
    run.close()
    roof = roofline_ms(cnt, hbm_gbs, b_p)
    leg_out = {"host_branch": host} if host else {}
    return {**leg_out, "config": config_of(s, mode, f_q16, rec_bytes), "steps": steps, "warmup": warmup,
            "tok_s": steps * s.B * world / (ms / 1e3), "ms_per_step": ms / steps,
            "roofline_ms_per_step": roof / steps, "frac": roof / ms,
            "hits_per_step": cnt["hits"] / steps, "misses_per_step": cnt["misses"] / steps,
            "fills_per_step": cnt["fills"] / steps,
            "deferred_routes_per_step": cnt["deferred_routes"] / steps,
            "link_gbs_achieved": cnt["link_bytes"] / (ms / 1e3) / 1e9, "device_status": status}


def dsv4_legs(args, ft, wlm, hbm_gbs, world, stream):
    import torch
    from dataclasses import replace
    s = wlm.SHAPES["dsv4_decode"]
    rec_bytes = ft.ft_record_bytes(s.H, s.I)
    pool = wlm.build_pool(args.seed, s.L, s.E, s.H, s.I)
    b_p, _ = measure_b_p(ft, pool, torch)
    legs = {}
    for B in (1, 4):
        for name, f in (("2/3", 2 / 3), ("1/2", 0.5), ("1/4", 0.25)):
            sb = replace(s, B=B)
            f_q16 = ft.ft_split_from_bandwidth(f, 1.0)
            leg = decode_leg(ft, wlm, sb, pool.ptr, None, "qstar", f_q16, args.seed, 32, 256,
                             rec_bytes, hbm_gbs, b_p, world, stream)
            leg["b_h_over_b_p"] = round(1 / f, 3)
            legs[f"dsv4_B{B}_f{name}"] = leg
    st = wlm.SHAPES["stress"]
    f_q16 = ft.ft_split_from_overlap(48.0, 40.0)
    leg = decode_leg(ft, wlm, st, pool.ptr, None, "qstar", f_q16, args.seed, 0, st.steps,
                     rec_bytes, hbm_gbs, b_p, world, stream)
    leg["note"] = ("whole 512-step run from an empty cache, resizes 1024 -> 256 (step 171) -> "
                   "768 (step 342) inside the timed region; f = p_ov / (p_ov + c_ov) at 48 / 40 GB/s")
    legs["stress"] = leg
    for v in legs.values():
        v["b_p_gbs"] = b_p
    pool.free()
    # the same layers from natively MXFP4 records (E8M0 scale per 32)
    rec_mx = ft.ft_record_bytes(s.H, s.I, "mxfp4")
    pool = wlm.build_pool(args.seed, s.L, s.E, s.H, s.I, fmt="mxfp4")
    b_p_mx, _ = measure_b_p(ft, pool, torch)
    for B in (1, 4):
        sb = replace(s, B=B)
        leg = decode_leg(ft, wlm, sb, pool.ptr, None, "qstar", 32768, args.seed, 32, 256,
                         rec_mx, hbm_gbs, b_p_mx, world, stream, fmt="mxfp4")
        leg["b_p_gbs"] = b_p_mx
        leg["record_format"] = "mxfp4"
        legs[f"dsv4_mxfp4_B{B}_f1/2"] = leg
    pool.free()
    return legs


def native_prefill(args, ft, wlm, pool, b_p, world):
    """Qwen3.6-shaped prefill: one 8192-token chunk through 40 layers, the next layer
    streaming into the other full-layer buffer while the current one computes, and
    without the double buffer; each pair interleaved with a copy-only pass of the same
    40 layer copies (what the host link delivers at that moment)."""
    import torch
    import synth
    s = wlm.SHAPES[args.prefill_workload]
    T, L = s.T, s.L
    rec = ft.ft_record_bytes(s.H, s.I)
    layer_bytes = s.E * rec
    cache = ft.ExpertCache(L, s.E, s.H, s.I, s.k, 1, s.C, pool.ptr, T_max=T)
    xs = [synth.prefill_x(args.seed, l, T, s.H, "cuda") for l in range(L)]
    routes = [synth.prefill_routes(args.seed, l, T, s.E, s.k, "cuda") for l in range(L)]
    y = torch.empty((T, s.H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    host = pool.tensor()
    buf = torch.empty(2 * layer_bytes, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()

    def chunk(flags):
        for l in range(L):
            ids, gates = routes[l]
            ft.ft_moe_prefill_layer(cache.handle, l, xs[l], ids, gates, T, s.k, y, flags)

    def timed_chunk(flags, copy_events):
        if copy_events:
            ft.ft_profile_enable(cache.handle, 1 << 4)      # copy stream only
            ft.ft_profile_read(cache.handle)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        chunk(flags)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(e0.elapsed_time(e1), world)
        copy = None
        if copy_events:
            c_ms, c_n = ft.ft_profile_read(cache.handle)["prefill_copy"]
            ft.ft_profile_enable(cache.handle, False)
            copy = {"copies": c_n, "ms": c_ms,
                    "gbs": c_n * layer_bytes / (c_ms / 1e3) / 1e9 if c_n else None}
        return ms, copy

    def copy_only():
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(side):
            e0.record()
            for l in range(L):
                b = l % 2
                buf[b * layer_bytes:(b + 1) * layer_bytes].copy_(
                    host[l * layer_bytes:(l + 1) * layer_bytes], non_blocking=True)
            e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    DB = ft.FT_PREFILL_DOUBLE_BUFFER
    chunk(DB)
    chunk(0)                                            # warm-up chunks
    torch.cuda.synchronize()
    db_ms, sb_ms, cp_ms, db_copy = [], [], [], []
    for _ in range(args.prefill_pairs):
        cp_ms.append(copy_only())
        ms, cp = timed_chunk(DB, True)
        db_ms.append(ms)
        db_copy.append(cp["gbs"])
        sb_ms.append(timed_chunk(0, False)[0])
    # per-kernel breakdown from a separate chunk with CUDA events around every launch
    ft.ft_profile_enable(cache.handle, True)
    ft.ft_profile_read(cache.handle)
    chunk(0)
    torch.cuda.synchronize()
    prof = ft.ft_profile_read(cache.handle)
    ft.ft_profile_enable(cache.handle, False)
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
    del buf
    od = prefill_on_demand_leg(args, ft, wlm, pool, b_p, world, xs, routes, y)
    db, db_sp = med_spread(db_ms)
    sb, sb_sp = med_spread(sb_ms)
    cp, cp_sp = med_spread(cp_ms)
    streamed = L * s.E * rec
    link_ms = streamed / (b_p * 1e9) * 1e3
    flops = 2.0 * T * s.k * 3 * s.H * s.I * L
    _, bf16_tf, src = peaks()
    fp4_tf = bf16_tf * 6.0                              # nominal dense FP4 : BF16 ratio (13.5 / 2.25)
    comp_ms = flops / (fp4_tf * 1e12) * 1e3
    g1_ms, g1_n = prof["prefill_gemm1"]
    g2_ms, g2_n = prof["prefill_gemm2"]
    g1_flop = 2.0 * T * s.k * 2 * s.I * s.H
    g2_flop = 2.0 * T * s.k * s.H * s.I
    return {
        "workload": s.name, "T": T, "L": L, "capacity": s.C,
        "tok_s": T * world / (db / 1e3), "ms_per_chunk": db,
        "tok_s_single_buffer": T * world / (sb / 1e3), "ms_per_chunk_single_buffer": sb,
        "pairs": {"double_ms": [round(v, 2) for v in db_ms], "single_ms": [round(v, 2) for v in sb_ms],
                  "copy_engine_only_ms": [round(v, 2) for v in cp_ms],
                  "double_copy_gbs": [round(v, 1) if v else None for v in db_copy],
                  "spread": {"double": db_sp, "single": sb_sp, "copy_engine_only": cp_sp},
                  "order": "copy-engine-only, double, single; repeated",
                  "copy_engine_note": "the same 40 layer copies as cudaMemcpyAsync on another stream, "
                                      "nothing else running: what a copy engine delivers at that moment "
                                      "(on some boxes it drops to 80-110 GB/s; the chunks stream by SM loads)"},
        "roofline": {"bound": "host link (streamed bytes) vs FP4 tensor", "link_ms": link_ms,
                     "compute_ms_at_peak": comp_ms, "frac": max(link_ms, comp_ms) / db,
                     "copy_engine_only_gbs": streamed / (cp / 1e3) / 1e9,
                     "double_stream_gbs_median": statistics.median([v for v in db_copy if v]),
                     "streamed_bytes": streamed, "b_p_gbs": b_p,
                     "fp4_peak_tflops": fp4_tf, "fp4_peak_source": f"{src} bf16 x 6 (nominal ratio)"},
        "on_demand": od,
        "gemm": {"gemm1_tflops": g1_flop / (g1_ms / g1_n / 1e3) / 1e12 if g1_n else None,
                 "gemm2_tflops": g2_flop / (g2_ms / g2_n / 1e3) / 1e12 if g2_n else None,
                 "gemm1_ms_per_layer": g1_ms / g1_n if g1_n else None,
                 "gemm2_ms_per_layer": g2_ms / g2_n if g2_n else None,
                 "other_ms_per_layer": prof["prefill_other"][0] / max(g1_n, 1),
                 "copy_ms_per_layer": prof["prefill_copy"][0] / max(prof["prefill_copy"][1], 1),
                 "profiled_chunk": "single-buffered, events around every launch and copy"},
    }


def prefill_on_demand_leg(args, ft, wlm, pool, b_p, world, xs, routes, y, capacity=200):
    """The same chunk with fewer slots than one layer's experts: every layer falls back
    to loading its routed union on demand, in groups of at most `capacity` experts,
    each gathered in batches whose GEMMs run beside the next batch's gather (a group
    cannot overlap the previous group's GEMMs: its victims are their slots).  Bound:
    the records it fills over the host link at B_P."""
    import torch
    s = wlm.SHAPES[args.prefill_workload]
    T, L = s.T, s.L
    rec = ft.ft_record_bytes(s.H, s.I)
    cache = ft.ExpertCache(L, s.E, s.H, s.I, s.k, 1, capacity, pool.ptr, T_max=T)
    stream = torch.cuda.current_stream()

    def chunk():
        for l in range(L):
            ids, gates = routes[l]
            ft.ft_moe_prefill_layer(cache.handle, l, xs[l], ids, gates, T, s.k, y,
                                    ft.FT_PREFILL_DOUBLE_BUFFER)

    chunk()
    torch.cuda.synchronize()
    ms_all = []
    for _ in range(2):
        ft.ft_cache_resize(cache.handle, capacity, cache.slot_buf)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        chunk()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms_all.append(max_over_ranks(e0.elapsed_time(e1), world))
    # fills of one chunk from an emptied cache: every expert of every layer's union is
    # loaded once per layer (the union covers all experts at this chunk size), so the
    # streamed bytes are the unions' sizes times the record
    unions = sum(int(torch.unique(routes[l][0]).numel()) for l in range(L))
    ft.ft_profile_enable(cache.handle, True)
    ft.ft_profile_read(cache.handle)
    ft.ft_cache_resize(cache.handle, capacity, cache.slot_buf)
    chunk()
    torch.cuda.synchronize()
    prof = ft.ft_profile_read(cache.handle)
    ft.ft_profile_enable(cache.handle, False)
    assert ft.ft_cache_status(cache.handle) == 0
    cache.close()
    ms = statistics.median(ms_all)
    streamed = unions * rec
    link_ms = streamed / (b_p * 1e9) * 1e3
    g_ms, g_n = prof["prefill_copy"]
    return {"capacity": capacity, "groups_per_layer": (s.E + capacity - 1) // capacity,
            "ms_per_chunk": ms, "tok_s": T * world / (ms / 1e3), "repeats_ms": [round(v, 2) for v in ms_all],
            "streamed_bytes": streamed, "link_ms": link_ms, "frac": link_ms / ms,
            "gather_gbs": streamed / (g_ms / 1e3) / 1e9 if g_ms else None,
            "gemm1_ms_per_layer": prof["prefill_gemm1"][0] / L, "gemm2_ms_per_layer": prof["prefill_gemm2"][0] / L,
            "note": "chunk from an emptied cache each time; DOUBLE_BUFFER asked for, 200 < 2E slots: "
                    "on-demand fallback; a group's records are gathered in batches, each batch's GEMMs "
                    "beside the next batch's gather; groups follow one another"}


def prefill_mx_leg(args, ft, wlm, world):
    """The Qwen-shaped chunk from an MXFP4 pool (E8M0 scale per 32), double-buffered."""
    import torch
    import synth
    s = wlm.SHAPES[args.prefill_workload]
    T, L = s.T, s.L
    rec = ft.ft_record_bytes(s.H, s.I, "mxfp4")
    pool = wlm.build_pool(args.seed, L, s.E, s.H, s.I, fmt="mxfp4")
    b_p, _ = measure_b_p(ft, pool, torch)
    cache = ft.ExpertCache(L, s.E, s.H, s.I, s.k, 1, s.C, pool.ptr, T_max=T, fmt="mxfp4")
    xs = [synth.prefill_x(args.seed, l, T, s.H, "cuda") for l in range(L)]
    routes = [synth.prefill_routes(args.seed, l, T, s.E, s.k, "cuda") for l in range(L)]
    y = torch.empty((T, s.H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def chunk():
        for l in range(L):
            ft.ft_moe_prefill_layer(cache.handle, l, xs[l], routes[l][0], routes[l][1], T, s.k, y,
                                    ft.FT_PREFILL_DOUBLE_BUFFER)

    chunk()
    ms_all = []
    for _ in range(2):
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        chunk()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms_all.append(max_over_ranks(e0.elapsed_time(e1), world))
    status = ft.ft_cache_status(cache.handle)
    ft.ft_profile_enable(cache.handle, True)           # per-kernel times of one more chunk
    ft.ft_profile_read(cache.handle)
    chunk()
    torch.cuda.synchronize()
    prof = ft.ft_profile_read(cache.handle)
    ft.ft_profile_enable(cache.handle, False)
    cache.close()
    pool.free()
    ms = statistics.median(ms_all)
    link_ms = L * s.E * rec / (b_p * 1e9) * 1e3
    per_layer = {k: v[0] / L for k, v in prof.items() if v[1]}
    return {"record_format": "mxfp4", "record_bytes": rec, "ms_per_chunk": ms,
            "ms_per_layer_by_kind": per_layer,
            "tok_s": T * world / (ms / 1e3), "repeats_ms": [round(v, 2) for v in ms_all],
            "link_ms": link_ms, "frac": link_ms / ms, "b_p_gbs": b_p, "device_status": status}


def prefill_only(args, world):
    """The prefill workload alone, on a pool of its own shape."""
    import torch
    import expert_cache_gb300 as ft
    from expert_cache_gb300 import workloads as wlm
    s = wlm.SHAPES[args.prefill_workload]
    pool = wlm.build_pool(args.seed, s.L, s.E, s.H, s.I)
    b_p, _ = measure_b_p(ft, pool, torch)
    pf = native_prefill(args, ft, wlm, pool, b_p, world)
    pool.free()
    return {"metric": "prefill tok/s (prefill-only run)", "value": pf["tok_s"], "unit": "tok/s",
            "n_gpus": world, "higher_is_better": True, "data": "synthetic",
            "config": {"workload": s.name}, "prefill": pf}


# ----------------------------------------------------------------- reference arm

def reference(args, world):
    """The CPU oracle, as it stands, on every host core: whole decode tokens of the
    headline workload (state oracle for the token's 40 layer calls in order, their
    fp64 outputs on one worker process per core)."""
    from oracle.formats import record_layout
    from synth.shapes import SHAPES
    s = SHAPES[args.workload]
    n = args.oracle_workers or cpu_cores()
    warm = min(args.warmup, 2)
    t0 = time.perf_counter()
    r = oracle_tokens(s, args.seed, n, tokens=args.steps, warmup=warm, budget_s=150.0)
    wall = time.perf_counter() - t0
    k = len(r["walls"])
    sec = sum(r["walls"]) / k
    value = s.B / sec
    return {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": k, "warmup": warm, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": config_of(s, "full", 65536, record_layout(s.H, s.I)["bytes"]),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": n, "kind": "oracle",
                             "cpu_model": cpu_model(), "blas_threads_per_worker": 1,
                             "sample": (f"{k} whole decode tokens after {warm} warm-up tokens; "
                                        f"{s.L} layer calls per token, outputs on {n} worker "
                                        f"processes at once; records encoded beforehand "
                                        f"({r['prepare_s']:.0f} s, untimed); wall {wall:.0f} s")},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "product_libraries_loaded": product_libraries_loaded()}


def product_libraries_loaded():
    """Shared objects of this repository mapped into the process (none on the
    reference arm: it runs the oracle only)."""
    libs = set()
    try:
        with open("/proc/self/maps") as fh:
            for line in fh:
                path = line.split()[-1] if len(line.split()) >= 6 else ""
                if path.startswith(ROOT) and path.endswith(".so"):
                    libs.add(os.path.relpath(path, ROOT))
    except OSError:
        pass
    return sorted(libs)


def main():
    args = parse()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        if rank != 0:
            return
        print(json.dumps(reference(args, world)), flush=True)
        return
    rank, world = dist_setup(args)
    out = prefill_only(args, world) if args.prefill_only else native(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
