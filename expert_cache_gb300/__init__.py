"""Python binding of libft, the GB300 routed-expert cache (argument marshalling only).

Every function below forwards to the C function of the same name declared in
``include/ft.h``; tensors are passed as raw pointers (``tensor.data_ptr()``) and
streams as ``torch.cuda.Stream.cuda_stream`` handles.  No step of the hot path
runs in Python.  Importing this module fails loudly when ``libft.so`` has not
been built (``python -m expert_cache_gb300.build`` or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libft.so")

FT_OK, FT_ERR_ARG, FT_ERR_CUDA, FT_ERR_CAPACITY, FT_ERR_STATE, FT_ERR_TIMEOUT, FT_ERR_UNPINNED = range(7)
FT_DEV_BAD_ID, FT_DEV_TIMEOUT, FT_DEV_SCALE_RANGE = 0x1, 0x2, 0x4
FT_FORMAT_NVFP4, FT_FORMAT_MXFP4 = 0, 1
FORMATS = {"nvfp4": FT_FORMAT_NVFP4, "mxfp4": FT_FORMAT_MXFP4}
FT_SPLIT_FULL_OFFLOAD, FT_SPLIT_QSTAR = 0, 1
FT_PREFILL_DOUBLE_BUFFER = 1
FT_PREFILL_DEBUG_X = 2
FT_PREFILL_ON_DEMAND = 4
FT_BACKEND_OFFLOAD, FT_BACKEND_HYBRID = 0, 1
FT_PROF_KINDS = 5
PROF_NAMES = ("decode", "prefill_gemm1", "prefill_gemm2", "prefill_other", "prefill_copy")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() first")

_lib = ctypes.CDLL(LIB_PATH)

c_void_p, c_int32, c_uint32, c_int64, c_size_t, c_double = (
    ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_int64, ctypes.c_size_t,
    ctypes.c_double)


class FtSplit(ctypes.Structure):
    _fields_ = [("mode", c_int32), ("f_q16", c_uint32)]


class FtCacheDesc(ctypes.Structure):
    _fields_ = [("L", c_int32), ("E", c_int32), ("H", c_int32), ("I", c_int32),
                ("k_max", c_int32), ("B_max", c_int32), ("capacity", c_int32),
                ("capacity_max", c_int32), ("T_max", c_int32),
                ("host_pool", c_void_p), ("slot_buf", c_void_p), ("workspace", c_void_p),
                ("shared_experts", c_void_p), ("split", FtSplit), ("format", c_int32)]


class FtHostDesc(ctypes.Structure):
    _fields_ = [("L", c_int32), ("E", c_int32), ("H", c_int32), ("I", c_int32),
                ("k_max", c_int32), ("B_max", c_int32), ("format", c_int32),
                ("host_pool", c_void_p), ("n_threads", c_int32), ("cpus", c_void_p),
                ("mailbox", c_void_p)]


class FtBwProfile(ctypes.Structure):
    _fields_ = [("pcie_gbs", c_double), ("cpu_gbs", c_double), ("pcie_ov_gbs", c_double),
                ("cpu_ov_gbs", c_double), ("recommend", c_int32), ("f_q16", c_uint32),
                ("n_records", c_int32)]


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_P = ctypes.POINTER
_f = {
    "ft_record_bytes": _sig("ft_record_bytes", c_int32, c_int32, c_int32, _P(c_size_t)),
    "ft_record_bytes_format": _sig("ft_record_bytes_format", c_int32, c_int32, c_int32, c_int32,
                                   _P(c_size_t)),
    "ft_quantize_experts_mx": _sig("ft_quantize_experts_mx", c_int32, c_void_p, c_void_p, c_int32,
                                   c_int32, c_int32, c_void_p, c_void_p),
    "ft_cache_required_sizes": _sig("ft_cache_required_sizes", c_int32, _P(FtCacheDesc),
                                    _P(c_size_t), _P(c_size_t)),
    "ft_cache_create": _sig("ft_cache_create", c_int32, _P(FtCacheDesc), _P(c_void_p)),
    "ft_cache_destroy": _sig("ft_cache_destroy", None, c_void_p),
    "ft_cache_resize": _sig("ft_cache_resize", c_int32, c_void_p, c_int32, c_void_p, c_void_p),
    "ft_set_split": _sig("ft_set_split", c_int32, c_void_p, FtSplit),
    "ft_split_from_bandwidth": _sig("ft_split_from_bandwidth", c_uint32, c_double, c_double),
    "ft_split_from_overlap": _sig("ft_split_from_overlap", c_uint32, c_double, c_double),
    "ft_moe_decode": _sig("ft_moe_decode", c_int32, c_void_p, c_int32, c_void_p, c_void_p,
                          c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                          c_void_p),
    "ft_moe_decode_static": _sig("ft_moe_decode_static", c_int32, c_void_p, c_int32, c_void_p,
                                 c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_void_p),
    "ft_moe_prefill_layer": _sig("ft_moe_prefill_layer", c_int32, c_void_p, c_int32, c_void_p,
                                 c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_int32,
                                 c_void_p, c_void_p),
    "ft_cache_snapshot": _sig("ft_cache_snapshot", c_int32, c_void_p, c_void_p, c_void_p,
                              c_void_p, c_void_p),
    "ft_cache_restore": _sig("ft_cache_restore", c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_int64, c_void_p),
    "ft_cache_set_trace": _sig("ft_cache_set_trace", c_int32, c_void_p, c_void_p, c_int32),
    "ft_cache_capacity": _sig("ft_cache_capacity", c_int32, c_void_p, _P(c_int32)),
    "ft_cache_status": _sig("ft_cache_status", c_int32, c_void_p, _P(c_int32)),
    "ft_check_bounded_waits": _sig("ft_check_bounded_waits", c_int32, _P(c_uint32)),
    "ft_quantize_experts": _sig("ft_quantize_experts", c_int32, c_void_p, c_void_p, c_int32,
                                c_int32, c_int32, c_void_p, c_void_p),
    "ft_pinned_alloc": _sig("ft_pinned_alloc", c_int32, c_size_t, _P(c_void_p)),
    "ft_pinned_free": _sig("ft_pinned_free", c_int32, c_void_p),
    "ft_measure_h2d": _sig("ft_measure_h2d", c_int32, c_void_p, c_void_p, c_size_t, c_int32,
                           _P(c_double)),
    "ft_profile_enable": _sig("ft_profile_enable", c_int32, c_void_p, c_int32),
    "ft_profile_read": _sig("ft_profile_read", c_int32, c_void_p, _P(c_double), _P(c_int64)),
    "ft_host_mailbox_bytes": _sig("ft_host_mailbox_bytes", c_int32, c_int32, c_int32, c_int32,
                                  _P(c_size_t)),
    "ft_host_branch_create": _sig("ft_host_branch_create", c_int32, _P(FtHostDesc), _P(c_void_p)),
    "ft_host_branch_destroy": _sig("ft_host_branch_destroy", None, c_void_p),
    "ft_host_moe": _sig("ft_host_moe", c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                        c_int32, c_void_p),
    "ft_host_branch_stats": _sig("ft_host_branch_stats", c_int32, c_void_p, _P(c_int64), _P(c_int64)),
    "ft_cache_set_host_branch": _sig("ft_cache_set_host_branch", c_int32, c_void_p, c_void_p),
    "ft_profile_bandwidth": _sig("ft_profile_bandwidth", c_int32, c_void_p, c_void_p, c_int32,
                                 c_void_p, _P(FtBwProfile)),
    "ft_recommend_backend": _sig("ft_recommend_backend", c_int32, c_double, c_double),
    "ft_status_string": _sig("ft_status_string", ctypes.c_char_p, c_int32),
    "ft_last_error": _sig("ft_last_error", ctypes.c_char_p, c_void_p),
}

EXPORTED = tuple(_f)


class FtError(RuntimeError):
    def __init__(self, status, msg=""):
        super().__init__(f"{_f['ft_status_string'](status).decode()} ({status}) {msg}".strip())
        self.status = status


def _ptr(t):
    """Raw address of a tensor / ndarray / int / None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return s if isinstance(s, int) else s.cuda_stream


def _check(status, handle=None):
    if status != FT_OK:
        msg = _f["ft_last_error"](handle).decode() if handle else ""
        raise FtError(status, msg)


# ----------------------------------------------------------------- thin wrappers

def ft_record_bytes(H, I, fmt="nvfp4"):
    out = c_size_t()
    if fmt == "nvfp4":
        _check(_f["ft_record_bytes"](H, I, ctypes.byref(out)))
    else:
        _check(_f["ft_record_bytes_format"](FORMATS[fmt], H, I, ctypes.byref(out)))
    return out.value


def ft_cache_required_sizes(desc: FtCacheDesc):
    rb, wb = c_size_t(), c_size_t()
    _check(_f["ft_cache_required_sizes"](ctypes.byref(desc), ctypes.byref(rb), ctypes.byref(wb)))
    return rb.value, wb.value


def ft_cache_create(desc: FtCacheDesc):
    h = c_void_p()
    _check(_f["ft_cache_create"](ctypes.byref(desc), ctypes.byref(h)))
    return h.value


def ft_cache_destroy(handle):
    _f["ft_cache_destroy"](handle)


def ft_cache_resize(handle, new_capacity, new_slot_buf, stream=None):
    _check(_f["ft_cache_resize"](handle, new_capacity, _ptr(new_slot_buf), _stream(stream)), handle)


def ft_set_split(handle, mode, f_q16=65536):
    _check(_f["ft_set_split"](handle, FtSplit(mode, f_q16)), handle)


def ft_split_from_bandwidth(b_p, b_h):
    return int(_f["ft_split_from_bandwidth"](b_p, b_h))


def ft_split_from_overlap(p_ov, c_ov):
    return int(_f["ft_split_from_overlap"](p_ov, c_ov))


def ft_moe_decode(handle, layer, x, topk_ids, topk_w, B, k, y, deferred, route_slot=None,
                  counters=None, stream=None):
    _check(_f["ft_moe_decode"](handle, layer, _ptr(x), _ptr(topk_ids), _ptr(topk_w), B, k,
                               _ptr(y), _ptr(deferred), _ptr(route_slot), _ptr(counters),
                               _stream(stream)), handle)


def ft_moe_decode_static(handle, layer, x, topk_ids, topk_w, B, k, y, deferred, route_slot=None,
                         counters=None, stream=None):
    _check(_f["ft_moe_decode_static"](handle, layer, _ptr(x), _ptr(topk_ids), _ptr(topk_w), B, k,
                                      _ptr(y), _ptr(deferred), _ptr(route_slot), _ptr(counters),
                                      _stream(stream)), handle)


def ft_moe_prefill_layer(handle, layer, x, topk_ids, topk_w, T, k, y, flags=FT_PREFILL_DOUBLE_BUFFER,
                         debug_h=None, stream=None):
    _check(_f["ft_moe_prefill_layer"](handle, layer, _ptr(x), _ptr(topk_ids), _ptr(topk_w), T, k,
                                      _ptr(y), flags, _ptr(debug_h), _stream(stream)), handle)


def ft_cache_capacity(handle):
    c = c_int32()
    _check(_f["ft_cache_capacity"](handle, ctypes.byref(c)), handle)
    return c.value


def ft_cache_snapshot(handle, L, E):
    """(slot_for_id [L*E], id_of_slot [C], usage [C], tick) as numpy arrays / int."""
    C = ft_cache_capacity(handle)
    sfi = np.empty(L * E, np.int32)
    ios = np.empty(C, np.int32)
    usage = np.empty(C, np.int64)
    tick = np.empty(1, np.int64)
    _check(_f["ft_cache_snapshot"](handle, sfi.ctypes.data, ios.ctypes.data, usage.ctypes.data,
                                   tick.ctypes.data), handle)
    return sfi, ios, usage, int(tick[0])


def ft_cache_restore(handle, slot_for_id, id_of_slot, usage, tick, stream=None):
    sfi = np.ascontiguousarray(slot_for_id, np.int32)
    ios = np.ascontiguousarray(id_of_slot, np.int32)
    us = np.ascontiguousarray(usage, np.int64)
    _check(_f["ft_cache_restore"](handle, sfi.ctypes.data, ios.ctypes.data, us.ctypes.data,
                                  int(tick), _stream(stream)), handle)


# one stats-ring record: tick, layer, n_hit, m, q, n_def_routes, n_units, t_commit_ns
TRACE_DTYPE = np.dtype([("tick", np.int64), ("layer", np.int32), ("n_hit", np.int32),
                        ("m", np.int32), ("q", np.int32), ("n_def_routes", np.int32),
                        ("n_units", np.int32), ("t_commit_ns", np.int64)])
TRACE_HEADER_BYTES = 16


def ft_cache_set_trace(handle, ring, capacity):
    _check(_f["ft_cache_set_trace"](handle, _ptr(ring), int(capacity)), handle)


def trace_records(ring_bytes: np.ndarray, capacity: int):
    """(count, records in write order) of a stats ring copied to the host."""
    count = int(ring_bytes[:8].view(np.uint64)[0])
    recs = ring_bytes[TRACE_HEADER_BYTES:TRACE_HEADER_BYTES + capacity * TRACE_DTYPE.itemsize]
    recs = recs.view(TRACE_DTYPE)
    n = min(count, capacity)
    start = count % capacity if count > capacity else 0
    order = [(start + i) % capacity for i in range(n)]
    return count, recs[order]


def ft_cache_status(handle):
    s = c_int32()
    _check(_f["ft_cache_status"](handle, ctypes.byref(s)), handle)
    return s.value


def ft_check_bounded_waits():
    bits = c_uint32()
    _check(_f["ft_check_bounded_waits"](ctypes.byref(bits)))
    return bits.value


def ft_quantize_experts(w_gu, w_d, n, H, I, records, stream=None, fmt="nvfp4"):
    name = "ft_quantize_experts" if fmt == "nvfp4" else "ft_quantize_experts_mx"
    _check(_f[name](_ptr(w_gu), _ptr(w_d), n, H, I, _ptr(records), _stream(stream)))


def ft_pinned_alloc(nbytes):
    p = c_void_p()
    _check(_f["ft_pinned_alloc"](nbytes, ctypes.byref(p)))
    return p.value


def ft_pinned_free(ptr):
    _check(_f["ft_pinned_free"](ptr))


def ft_measure_h2d(pinned, dev, nbytes, reps=5):
    g = c_double()
    _check(_f["ft_measure_h2d"](_ptr(pinned), _ptr(dev), nbytes, reps, ctypes.byref(g)))
    return g.value


FT_PROF_ALL = (1 << FT_PROF_KINDS) - 1


def ft_profile_enable(handle, kinds=True):
    """kinds: True (all kinds), False (off) or a bit mask of kinds (bit i: kind i)."""
    mask = FT_PROF_ALL if kinds is True else (0 if kinds is False else int(kinds))
    _check(_f["ft_profile_enable"](handle, mask), handle)


def ft_profile_read(handle):
    ms = (c_double * FT_PROF_KINDS)()
    n = (c_int64 * FT_PROF_KINDS)()
    _check(_f["ft_profile_read"](handle, ms, n), handle)
    return {PROF_NAMES[i]: (ms[i], n[i]) for i in range(FT_PROF_KINDS)}


def ft_host_mailbox_bytes(H, k_max, B_max):
    n = c_size_t()
    _check(_f["ft_host_mailbox_bytes"](H, k_max, B_max, ctypes.byref(n)))
    return n.value


def ft_host_branch_create(desc: FtHostDesc):
    h = c_void_p()
    _check(_f["ft_host_branch_create"](ctypes.byref(desc), ctypes.byref(h)))
    return h.value


def ft_host_branch_destroy(hb):
    _f["ft_host_branch_destroy"](hb)


def ft_host_moe(hb, x, deferred, w, B, k, y):
    _check(_f["ft_host_moe"](hb, _ptr(x), _ptr(deferred), _ptr(w), B, k, _ptr(y)))


def ft_host_branch_stats(hb):
    jobs, mb = c_int64(), c_int64()
    _check(_f["ft_host_branch_stats"](hb, ctypes.byref(jobs), ctypes.byref(mb)))
    return jobs.value, mb.value


def ft_cache_set_host_branch(handle, hb):
    _check(_f["ft_cache_set_host_branch"](handle, hb), handle)


def ft_profile_bandwidth(handle, hb, n_records, stream=None):
    out = FtBwProfile()
    _check(_f["ft_profile_bandwidth"](handle, hb, n_records, _stream(stream), ctypes.byref(out)), handle)
    return {k: getattr(out, k) for k, _ in FtBwProfile._fields_}


def ft_recommend_backend(cpu_gbs, pcie_gbs):
    return _f["ft_recommend_backend"](cpu_gbs, pcie_gbs)


# ----------------------------------------------------------------- memory plumbing

class PinnedBuffer:
    """Page-locked, device-mapped host bytes from ft_pinned_alloc, viewed as a
    uint8 numpy array and a CPU torch tensor sharing the same memory."""

    def __init__(self, nbytes: int):
        self.nbytes = int(nbytes)
        self.ptr = ft_pinned_alloc(self.nbytes)
        self.array = np.ctypeslib.as_array((ctypes.c_uint8 * self.nbytes).from_address(self.ptr))

    def tensor(self):
        import torch
        return torch.from_numpy(self.array)

    def free(self):
        if self.ptr:
            ft_pinned_free(self.ptr)
            self.ptr = None
            self.array = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class ExpertCache:
    """Owns the device memory of one cache (slot buffer, workspace; torch allocations)
    and the ft_cache handle over a caller-provided pinned host pool."""

    def __init__(self, L, E, H, I, k_max, B_max, capacity, host_pool_ptr, shared=None,
                 split=(FT_SPLIT_FULL_OFFLOAD, 65536), capacity_max=0, T_max=0, device="cuda",
                 fmt="nvfp4"):
        import torch
        self.L, self.E, self.H, self.I = L, E, H, I
        self.desc = FtCacheDesc(L, E, H, I, k_max, B_max, capacity, capacity_max, T_max,
                                None, None, None, None, FtSplit(*split), FORMATS[fmt])
        self.rec_bytes, ws_bytes = ft_cache_required_sizes(self.desc)
        cmax = capacity_max or capacity
        self.slot_buf = torch.empty(cmax * self.rec_bytes, dtype=torch.uint8, device=device)
        self.workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        self.shared = shared
        self.desc.host_pool = host_pool_ptr
        self.desc.slot_buf = self.slot_buf.data_ptr()
        self.desc.workspace = self.workspace.data_ptr()
        self.desc.shared_experts = _ptr(shared)
        self.handle = ft_cache_create(self.desc)

    def close(self):
        if self.handle:
            ft_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostBranch:
    """Owns one host branch (ft_host_branch_create) and its pinned mailbox."""

    def __init__(self, L, E, H, I, k_max, B_max, host_pool_ptr, n_threads, cpus=None, fmt="nvfp4",
                 mailbox=True):
        self.H = H
        self.mailbox = PinnedBuffer(ft_host_mailbox_bytes(H, k_max, B_max)) if mailbox else None
        self._cpus = (ctypes.c_int32 * n_threads)(*cpus) if cpus is not None else None
        self.desc = FtHostDesc(L, E, H, I, k_max, B_max, FORMATS[fmt], host_pool_ptr, n_threads,
                               ctypes.addressof(self._cpus) if self._cpus is not None else None,
                               self.mailbox.ptr if self.mailbox else None)
        self.handle = ft_host_branch_create(self.desc)

    def close(self):
        if self.handle:
            ft_host_branch_destroy(self.handle)
            self.handle = None
        if self.mailbox is not None:
            self.mailbox.free()
            self.mailbox = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
