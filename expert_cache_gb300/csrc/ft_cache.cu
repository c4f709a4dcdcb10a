// Host side of the C ABI: cache creation over caller-owned memory, the decode
// call sequence, resize at a safe point, snapshots, the split helpers, pinned
// memory, the H2D probe and per-kernel profiling.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <new>

#include <vector>
#include "ft_internal.cuh"
#include "ft_prefill.cuh"
#include "ft_umma.cuh"

namespace ft {

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

WsLayout ws_layout(const ft_cache_desc& d) {
    WsLayout w{};
    const int cmax = d.capacity_max > 0 ? d.capacity_max : d.capacity;
    const size_t R = (size_t)d.B_max * d.k_max;
    const size_t P = R + d.B_max;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    w.slot_for_id = take((size_t)d.L * d.E * 4);
    w.id_of_slot = take((size_t)cmax * 4);
    w.usage = take((size_t)cmax * 8);
    w.lru_order = take((size_t)cmax * 4);
    w.scalars = take(sizeof(DevScalars));
    w.sync = take(kSyncWords * 4);
    w.h = take(P * (size_t)d.I * 8);
    w.yflag = take((size_t)(d.H / decode_rows(d.I)) * 8);
    w.h_end = w.yflag + (size_t)(d.H / decode_rows(d.I)) * 8;
    if (d.T_max > 0) {
        // at least one 128-row tile so a TMA box never exceeds the sorted buffers
        const size_t RT = std::max<size_t>((size_t)d.T_max * d.k_max, 128);
        w.pf_chunk_cnt = take((size_t)((d.T_max + 31) / 32) * d.E * 4);
        w.pf_offsets = take((size_t)(d.E + 1) * 4);
        w.pf_mtile = take((size_t)(d.E + 1) * 4);
        w.pf_perm = take(RT * 4);
        w.pf_route_pos = take(RT * 4);
        w.pf_a_codes = take(RT * d.H / 2);
        w.pf_a_scales = take(RT * d.H / 16);
        w.pf_h_codes = take(RT * d.I / 2);
        w.pf_h_scales = take(RT * d.I / 16);
        w.pf_o = take(RT * d.H * 4);
        w.pf_slot_of = take((size_t)d.E * 4);
        w.pf_gmtile = take((size_t)(d.E + 1) * 4);
        w.pf_fill_flat = take((size_t)d.E * 4);
        w.pf_fill_slot = take((size_t)d.E * 4);
        w.pf_nfill = take(4);
        w.pf_sub = take((size_t)2 * (ft::kOdSub + 1) * 4);
    }
    w.total = off;
    return w;
}

// SM count of the current device (looked up once per device).
int sm_count() {
    static std::atomic<int> n[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 1;
    }
    int v = n[dev].load(std::memory_order_relaxed);
    if (!v) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
            cudaGetLastError();
            v = 1;
        }
        n[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace ft

using namespace ft;

static const char* kStatusNames[] = {"ok", "bad argument", "CUDA error", "not enough capacity",
                                     "bad state", "device wait timed out", "host pool not pinned"};

static ft_status fail(ft_cache* c, ft_status s, const char* msg) {
    if (c) snprintf(c->err, sizeof(c->err), "%s", msg);
    return s;
}

static ft_status cuda_fail(ft_cache* c, cudaError_t e, const char* where) {
    if (c) snprintf(c->err, sizeof(c->err), "%s: %s", where, cudaGetErrorString(e));
    return FT_ERR_CUDA;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

static ft_status check_desc(const ft_cache_desc* d) {
    if (!d) return FT_ERR_ARG;
    const int cmax = d->capacity_max > 0 ? d->capacity_max : d->capacity;
    if (d->L < 1 || d->E < 1 || d->E > kMaxE) return FT_ERR_ARG;
    if (d->H < 64 || d->H % 64 || d->H > kMaxH) return FT_ERR_ARG;
    if (d->I < 32 || d->I % 32 || d->I > kMaxI) return FT_ERR_ARG;
    if (d->k_max < 1 || d->k_max > kMaxK || d->B_max < 1 || d->B_max > kMaxB) return FT_ERR_ARG;
    if (d->B_max * d->k_max > kMaxRoutes) return FT_ERR_ARG;
    if (d->capacity < 1 || d->capacity > kMaxC || cmax < d->capacity || cmax > kMaxC) return FT_ERR_ARG;
    if ((long long)d->L * d->E > (1LL << 30) || d->T_max < 0) return FT_ERR_ARG;
    if (d->split.mode != FT_SPLIT_FULL_OFFLOAD && d->split.mode != FT_SPLIT_QSTAR) return FT_ERR_ARG;
    if (d->split.mode == FT_SPLIT_QSTAR && (d->split.f_q16 < 1 || d->split.f_q16 > 65536)) return FT_ERR_ARG;
    if (d->format != FT_FORMAT_NVFP4 && d->format != FT_FORMAT_MXFP4) return FT_ERR_ARG;
    return FT_OK;
}

namespace ft {

// Arguments of a decode call except the per-call scratch (h, o, sync).
DecodeArgs decode_args(ft_cache* c, int layer, const void* x, const int32_t* ids, const float* w,
                       int B, int k, float* y, int32_t* deferred, int32_t* route_slot,
                       int32_t* counters) {
    uint8_t* ws = c->workspace;
    DecodeArgs a{};
    a.slot_for_id = reinterpret_cast<int32_t*>(ws + c->ws.slot_for_id);
    a.id_of_slot = reinterpret_cast<int32_t*>(ws + c->ws.id_of_slot);
    a.usage = reinterpret_cast<long long*>(ws + c->ws.usage);
    a.lru_order = reinterpret_cast<int32_t*>(ws + c->ws.lru_order);
    a.sc = reinterpret_cast<DevScalars*>(ws + c->ws.scalars);
    a.host_pool = c->host_pool_dev;
    a.slot_buf = c->slot_buf;
    a.shared = static_cast<const uint8_t*>(c->d.shared_experts);
    a.rec_bytes = c->rec.bytes;
    a.off_gu_scales = c->rec.gu_scales;
    a.off_d_codes = c->rec.d_codes;
    a.off_d_scales = c->rec.d_scales;
    a.off_s_gu = c->rec.s_gu;
    a.off_s_d = c->rec.s_d;
    a.L = c->d.L; a.E = c->d.E; a.H = c->d.H; a.I = c->d.I; a.C = c->C;
    a.layer = layer; a.B = B; a.k = k;
    a.R_cap = c->d.B_max * c->d.k_max;
    a.mx = c->d.format == FT_FORMAT_MXFP4 ? 1 : 0;
    a.split_mode = c->d.split.mode;
    a.f_q16 = c->d.split.f_q16;
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.ids = ids;
    a.w = w;
    a.y = y;
    a.deferred = deferred;
    a.route_slot = route_slot;
    a.counters = counters;
    a.trace = static_cast<unsigned long long*>(c->trace);
    a.trace_cap = c->trace ? (unsigned)c->trace_cap : 0u;
    if (c->host) {
        a.mb = c->mb_dev;
        a.mb_x = (unsigned)c->ml.x;
        a.mb_def = (unsigned)c->ml.def;
        a.mb_w = (unsigned)c->ml.w;
    }
    return a;
}

}  // namespace ft

// TMA maps of the prefill GEMM operands (only when the cache supports prefill).
static bool prefill_maps(ft_cache* c) {
    const ft_cache_desc& d = c->d;
    if (d.T_max <= 0 || d.H % 256 || d.I % 256) return false;
    const uint64_t RT = std::max<uint64_t>((uint64_t)d.T_max * d.k_max, 128);
    uint8_t* ws = c->workspace;
    bool ok = make_map_2d(&c->map_a1, ws + c->ws.pf_a_codes, d.H / 2, RT);
    ok = ok && make_map_2d(&c->map_a2, ws + c->ws.pf_h_codes, d.I / 2, RT);
    ok = ok && make_map_3d(&c->map_b1, c->slot_buf + c->rec.gu_codes, d.H / 2, 2 * (uint64_t)d.I,
                           (uint64_t)c->C, c->rec.bytes, 128);
    ok = ok && make_map_3d(&c->map_b2, c->slot_buf + c->rec.d_codes, d.I / 2, (uint64_t)d.H,
                           (uint64_t)c->C, c->rec.bytes, 256);
    return ok;
}

extern "C" {

ft_status ft_record_bytes(int32_t H, int32_t I, size_t* bytes) {
    if (!bytes || H < 64 || H % 64 || I < 32 || I % 32) return FT_ERR_ARG;
    *bytes = record_layout(H, I).bytes;
    return FT_OK;
}

ft_status ft_record_bytes_format(int32_t format, int32_t H, int32_t I, size_t* bytes) {
    if (format != FT_FORMAT_NVFP4 && format != FT_FORMAT_MXFP4) return FT_ERR_ARG;
    if (!bytes || H < 64 || H % 64 || I < 32 || I % 32) return FT_ERR_ARG;
    *bytes = record_layout(H, I, format).bytes;
    return FT_OK;
}

ft_status ft_cache_required_sizes(const ft_cache_desc* d, size_t* record_bytes,
                                  size_t* workspace_bytes) {
    ft_status s = check_desc(d);
    if (s != FT_OK) return s;
    if (record_bytes) *record_bytes = record_layout(d->H, d->I, d->format).bytes;
    if (workspace_bytes) *workspace_bytes = ws_layout(*d).total;
    return FT_OK;
}

ft_status ft_cache_create(const ft_cache_desc* d, ft_cache** out) {
    if (!out) return FT_ERR_ARG;
    *out = nullptr;
    ft_status s = check_desc(d);
    if (s != FT_OK) return s;
    if (!d->host_pool || !d->slot_buf || !d->workspace) return FT_ERR_ARG;
    if (!aligned(d->slot_buf, 256) || !aligned(d->workspace, 256) || !aligned(d->host_pool, 256))
        return FT_ERR_ARG;
    if (d->shared_experts && !aligned(d->shared_experts, 256)) return FT_ERR_ARG;

    cudaPointerAttributes pa;
    cudaError_t e = cudaPointerGetAttributes(&pa, d->host_pool);
    if (e != cudaSuccess || pa.type != cudaMemoryTypeHost || !pa.devicePointer) {
        cudaGetLastError();
        return FT_ERR_UNPINNED;
    }
    cudaPointerAttributes pw, psb;
    if (cudaPointerGetAttributes(&pw, d->workspace) != cudaSuccess ||
        cudaPointerGetAttributes(&psb, d->slot_buf) != cudaSuccess ||
        (pw.type != cudaMemoryTypeDevice && pw.type != cudaMemoryTypeManaged) ||
        (psb.type != cudaMemoryTypeDevice && psb.type != cudaMemoryTypeManaged)) {
        cudaGetLastError();
        return FT_ERR_ARG;
    }

    ft_cache* c = new (std::nothrow) ft_cache();
    if (!c) return FT_ERR_ARG;
    c->d = *d;
    if (c->d.capacity_max <= 0) c->d.capacity_max = d->capacity;
    c->rec = record_layout(d->H, d->I, d->format);
    c->ws = ws_layout(c->d);
    c->C = d->capacity;
    c->host_pool_dev = static_cast<const uint8_t*>(pa.devicePointer);
    c->slot_buf = static_cast<uint8_t*>(d->slot_buf);
    c->workspace = static_cast<uint8_t*>(d->workspace);
    c->buffer_layer[0] = c->buffer_layer[1] = -1;
    c->copy_pending = false;
    c->prof = 0;
    c->prof_n = 0;
    c->trace = nullptr;
    c->trace_cap = 0;
    c->host = nullptr;
    c->mb_dev = nullptr;
    c->err[0] = 0;
    c->grid_decode = decode_grid(d->H, d->I, d->E, d->B_max * d->k_max);
    if (c->grid_decode < 2) {
        delete c;
        return FT_ERR_CUDA;
    }

    if ((e = cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking)) != cudaSuccess) {
        delete c;
        return FT_ERR_CUDA;
    }
    for (int i = 0; i < 2; ++i) {
        cudaEventCreateWithFlags(&c->copy_done[i], cudaEventDisableTiming);
        cudaEventCreateWithFlags(&c->compute_done[i], cudaEventDisableTiming);
    }
    cudaEventCreateWithFlags(&c->entry_ev, cudaEventDisableTiming);
    for (int i = 0; i <= kOdSub; ++i) cudaEventCreateWithFlags(&c->od_ev[i], cudaEventDisableTiming);
    c->maps_ok = prefill_maps(c);
    uint8_t* ws = c->workspace;
    e = launch_init_tables(reinterpret_cast<int32_t*>(ws + c->ws.slot_for_id), d->L * d->E,
                           reinterpret_cast<int32_t*>(ws + c->ws.id_of_slot),
                           reinterpret_cast<long long*>(ws + c->ws.usage),
                           reinterpret_cast<int32_t*>(ws + c->ws.lru_order), c->C,
                           reinterpret_cast<DevScalars*>(ws + c->ws.scalars), true, c->copy_stream);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(ws + c->ws.sync, 0, c->ws.h_end - c->ws.sync, c->copy_stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->copy_stream);
    if (e != cudaSuccess) {
        ft_cache_destroy(c);
        return FT_ERR_CUDA;
    }
    *out = c;
    return FT_OK;
}

void ft_cache_destroy(ft_cache* c) {
    if (!c) return;
    cudaStreamSynchronize(c->copy_stream);
    for (int i = 0; i < 2; ++i) {
        cudaEventDestroy(c->copy_done[i]);
        cudaEventDestroy(c->compute_done[i]);
    }
    cudaEventDestroy(c->entry_ev);
    for (int i = 0; i <= kOdSub; ++i) cudaEventDestroy(c->od_ev[i]);
    if (c->prof_n >= 0) {
        for (int i = 0; i < ft_cache::kProfEvents; ++i)
            if (c->prof_ev[i]) cudaEventDestroy(c->prof_ev[i]);
    }
    cudaStreamDestroy(c->copy_stream);
    delete c;
}

ft_status ft_cache_capacity(const ft_cache* c, int32_t* capacity) {
    if (!c || !capacity) return FT_ERR_ARG;
    *capacity = c->C;
    return FT_OK;
}

ft_status ft_set_split(ft_cache* c, ft_split s) {
    if (!c) return FT_ERR_ARG;
    if (s.mode != FT_SPLIT_FULL_OFFLOAD && s.mode != FT_SPLIT_QSTAR)
        return fail(c, FT_ERR_ARG, "split mode");
    if (s.mode == FT_SPLIT_QSTAR && (s.f_q16 < 1 || s.f_q16 > 65536))
        return fail(c, FT_ERR_ARG, "f_q16 outside [1, 65536]");
    c->d.split = s;
    return FT_OK;
}

static uint32_t frac_q16(double f) {
    if (!(f > 0)) return 0;
    if (f > 1) f = 1;
    double q = std::floor(f * 65536.0 + 0.5);
    return q > 65536.0 ? 65536u : (uint32_t)q;
}

uint32_t ft_split_from_bandwidth(double B_P, double B_H) {
    if (!(B_P > 0) || !(B_H > 0)) return 0;
    return frac_q16(B_P / B_H);
}

uint32_t ft_split_from_overlap(double p_ov, double c_ov) {
    if (!(p_ov > 0) || !(c_ov >= 0)) return 0;
    return frac_q16(p_ov / (p_ov + c_ov));
}

// ------------------------------------------------------------------ profiling

static void prof_fold(ft_cache* c) {
    if (c->prof_n == 0) return;
    for (int i = 0; i < c->prof_n; ++i) {
        float ms = 0.f;
        cudaEventSynchronize(c->prof_ev[2 * i + 1]);   // pairs may sit on different streams
        if (cudaEventElapsedTime(&ms, c->prof_ev[2 * i], c->prof_ev[2 * i + 1]) == cudaSuccess) {
            c->prof_ms[c->prof_kind[i]] += ms;
            c->prof_launches[c->prof_kind[i]] += 1;
        }
    }
    c->prof_n = 0;
}

}  // extern "C"

namespace ft {

// Records the "before" event of a launch of `kind`; returns the pair index or -1.
int prof_begin(ft_cache* c, int kind, cudaStream_t s) {
    if (!(c->prof & (1u << kind))) return -1;
    if (c->prof_n * 2 + 2 > ft_cache::kProfEvents) prof_fold(c);
    const int i = c->prof_n++;
    c->prof_kind[i] = kind;
    cudaEventRecord(c->prof_ev[2 * i], s);
    return i;
}

void prof_end(ft_cache* c, int i, cudaStream_t s) {
    if (i >= 0) cudaEventRecord(c->prof_ev[2 * i + 1], s);
}

}  // namespace ft

extern "C" {

ft_status ft_profile_enable(ft_cache* c, int32_t enable) {
    if (!c) return FT_ERR_ARG;
    if (enable && !c->prof_ev[0]) {
        for (int i = 0; i < ft_cache::kProfEvents; ++i)
            if (cudaEventCreate(&c->prof_ev[i]) != cudaSuccess) return FT_ERR_CUDA;
    }
    if (!enable) prof_fold(c);
    c->prof = (unsigned)enable & ((1u << FT_PROF_KINDS) - 1);
    return FT_OK;
}

ft_status ft_profile_read(ft_cache* c, double* total_ms, int64_t* launches) {
    if (!c) return FT_ERR_ARG;
    prof_fold(c);
    for (int k = 0; k < FT_PROF_KINDS; ++k) {
        if (total_ms) total_ms[k] = c->prof_ms[k];
        if (launches) launches[k] = c->prof_launches[k];
        c->prof_ms[k] = 0;
        c->prof_launches[k] = 0;
    }
    return FT_OK;
}

// ------------------------------------------------------------------ decode

ft_status ft_moe_decode(ft_cache* c, int32_t layer, const void* x, const int32_t* topk_ids,
                        const float* topk_w, int32_t B, int32_t k, float* y,
                        int32_t* deferred, int32_t* route_slot, int32_t* counters,
                        void* stream) {
    NvtxRange range("ft_moe_decode");
    if (!c) return FT_ERR_ARG;
    if (layer < 0 || layer >= c->d.L) return fail(c, FT_ERR_ARG, "layer out of range");
    if (B < 1 || B > c->d.B_max) return fail(c, FT_ERR_ARG, "B outside [1, B_max]");
    if (k < 1 || k > c->d.k_max) return fail(c, FT_ERR_ARG, "k outside [1, k_max]");
    if (!x || !topk_ids || !topk_w || !y || !deferred) return fail(c, FT_ERR_ARG, "NULL argument");
    if (!aligned(x, 16)) return fail(c, FT_ERR_ARG, "x must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (c->copy_pending) {   // a prefill stream-in may still be writing slots
        cudaStreamWaitEvent(s, c->copy_done[0], 0);
        cudaStreamWaitEvent(s, c->copy_done[1], 0);
        c->copy_pending = false;
    }
    c->buffer_layer[0] = c->buffer_layer[1] = -1;   // decode may evict prefill buffers

    DecodeArgs a = decode_args(c, layer, x, topk_ids, topk_w, B, k, y, deferred, route_slot,
                               counters);
    a.h = reinterpret_cast<unsigned long long*>(c->workspace + c->ws.h);
    a.sync = reinterpret_cast<unsigned*>(c->workspace + c->ws.sync);
    a.yflag = reinterpret_cast<unsigned long long*>(c->workspace + c->ws.yflag);
    a.scrub = a.h;
    a.scrub_words = (c->ws.h_end - c->ws.h) / 8;
    const int p = prof_begin(c, 0, s);
    cudaError_t e = launch_decode(a, c->grid_decode, s);
    prof_end(c, p, s);
    if (e == cudaSuccess && c->host)
        e = launch_host_join(c->mb_dev, (unsigned)c->ml.y, y, B * c->d.H, &a.sc->counters[3], &a.sc->status, s);
    if (e != cudaSuccess) return cuda_fail(c, e, "decode launch");
    return FT_OK;
}

// ------------------------------------------------------------------ resize / state

ft_status ft_cache_resize(ft_cache* c, int32_t new_capacity, void* new_slot_buf, void* stream) {
    NvtxRange range("ft_cache_resize");
    if (!c) return FT_ERR_ARG;
    if (new_capacity < 1 || new_capacity > c->d.capacity_max)
        return fail(c, FT_ERR_ARG, "new_capacity outside [1, capacity_max]");
    if (!new_slot_buf || !aligned(new_slot_buf, 256)) return fail(c, FT_ERR_ARG, "slot buffer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return cuda_fail(c, cudaGetLastError(), "capture query");
    if (cs != cudaStreamCaptureStatusNone) return fail(c, FT_ERR_STATE, "resize while capturing");
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->copy_stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "resize drain");
    c->C = new_capacity;
    c->slot_buf = static_cast<uint8_t*>(new_slot_buf);
    c->maps_ok = prefill_maps(c);
    c->buffer_layer[0] = c->buffer_layer[1] = -1;
    c->copy_pending = false;
    uint8_t* ws = c->workspace;
    e = launch_init_tables(reinterpret_cast<int32_t*>(ws + c->ws.slot_for_id), c->d.L * c->d.E,
                           reinterpret_cast<int32_t*>(ws + c->ws.id_of_slot),
                           reinterpret_cast<long long*>(ws + c->ws.usage),
                           reinterpret_cast<int32_t*>(ws + c->ws.lru_order), c->C,
                           reinterpret_cast<DevScalars*>(ws + c->ws.scalars), false, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(c, e, "resize rebuild");
    return FT_OK;
}

ft_status ft_cache_snapshot(ft_cache* c, int32_t* slot_for_id, int32_t* id_of_slot,
                            int64_t* usage, int64_t* tick) {
    if (!c) return FT_ERR_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    const uint8_t* ws = c->workspace;
    if (e == cudaSuccess && slot_for_id)
        e = cudaMemcpy(slot_for_id, ws + c->ws.slot_for_id, (size_t)c->d.L * c->d.E * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && id_of_slot)
        e = cudaMemcpy(id_of_slot, ws + c->ws.id_of_slot, (size_t)c->C * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && usage)
        e = cudaMemcpy(usage, ws + c->ws.usage, (size_t)c->C * 8, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && tick)
        e = cudaMemcpy(tick, ws + c->ws.scalars + offsetof(DevScalars, tick), 8, cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? FT_OK : cuda_fail(c, e, "snapshot");
}

ft_status ft_cache_restore(ft_cache* c, const int32_t* slot_for_id, const int32_t* id_of_slot,
                           const int64_t* usage, int64_t tick, void* stream) {
    NvtxRange range("ft_cache_restore");
    if (!c) return FT_ERR_ARG;
    if (!slot_for_id || !id_of_slot || !usage || tick < 0) return fail(c, FT_ERR_ARG, "NULL table or tick < 0");
    const int C = c->C;
    const long long n_ids = (long long)c->d.L * c->d.E;
    // consistency of the tables (host side, before anything is written)
    for (int s = 0; s < C; ++s) {
        const int f = id_of_slot[s];
        if (f < -1 || f >= n_ids) return fail(c, FT_ERR_ARG, "id_of_slot entry out of range");
        if (f >= 0 && slot_for_id[f] != s) return fail(c, FT_ERR_ARG, "id_of_slot / slot_for_id disagree");
        if (f < 0 && usage[s] != -1) return fail(c, FT_ERR_ARG, "free slot with usage != -1");
        if (f >= 0 && (usage[s] < 0 || usage[s] > tick)) return fail(c, FT_ERR_ARG, "usage outside [0, tick]");
    }
    for (long long f = 0; f < n_ids; ++f) {
        const int s = slot_for_id[f];
        if (s < -1 || s >= C) return fail(c, FT_ERR_ARG, "slot_for_id entry out of range");
        if (s >= 0 && id_of_slot[s] != f) return fail(c, FT_ERR_ARG, "slot_for_id / id_of_slot disagree");
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return cuda_fail(c, cudaGetLastError(), "capture query");
    if (cs != cudaStreamCaptureStatusNone) return fail(c, FT_ERR_STATE, "restore while capturing");
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->copy_stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "restore drain");
    // LRU order: free slots ascending, then ascending (usage, slot)
    int32_t* order = new (std::nothrow) int32_t[C];
    if (!order) return fail(c, FT_ERR_ARG, "host allocation for the LRU order failed");
    for (int s = 0; s < C; ++s) order[s] = s;
    std::stable_sort(order, order + C, [&](int a, int b) { return usage[a] < usage[b]; });
    uint8_t* ws = c->workspace;
    e = cudaMemcpy(ws + c->ws.slot_for_id, slot_for_id, (size_t)n_ids * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(ws + c->ws.id_of_slot, id_of_slot, (size_t)C * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(ws + c->ws.usage, usage, (size_t)C * 8, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(ws + c->ws.lru_order, order, (size_t)C * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = cudaMemcpy(ws + c->ws.scalars + offsetof(DevScalars, tick), &tick, 8, cudaMemcpyHostToDevice);
    delete[] order;
    if (e != cudaSuccess) return cuda_fail(c, e, "restore copy");
    c->buffer_layer[0] = c->buffer_layer[1] = -1;
    c->copy_pending = false;
    return FT_OK;
}

ft_status ft_cache_set_trace(ft_cache* c, void* ring, int32_t capacity) {
    if (!c || capacity < 0) return FT_ERR_ARG;
    if (ring && !aligned(ring, 16)) return fail(c, FT_ERR_ARG, "trace ring must be 16-byte aligned");
    c->trace = capacity > 0 ? ring : nullptr;
    c->trace_cap = c->trace ? capacity : 0;
    return FT_OK;
}

ft_status ft_cache_set_host_branch(ft_cache* c, ft_host_branch* hb) {
    if (!c) return FT_ERR_ARG;
    cudaError_t e = cudaDeviceSynchronize();   // no call of c still publishing to the old branch
    if (e != cudaSuccess) return cuda_fail(c, e, "host branch attach");
    if (!hb) {
        c->host = nullptr;
        c->mb_dev = nullptr;
        return FT_OK;
    }
    ft::HostBranchInfo hi;
    if (!ft::host_branch_info(hb, &hi)) return fail(c, FT_ERR_ARG, "host branch");
    if (hi.pool != c->d.host_pool || hi.L != c->d.L || hi.E != c->d.E || hi.H != c->d.H || hi.I != c->d.I ||
        hi.format != c->d.format || hi.B_max < c->d.B_max || hi.k_max < c->d.k_max || !hi.mailbox)
        return fail(c, FT_ERR_ARG, "host branch of another pool, shape or format, or without a mailbox");
    void* dev = nullptr;
    e = cudaHostGetDevicePointer(&dev, hi.mailbox, 0);
    if (e != cudaSuccess) return cuda_fail(c, e, "mailbox is not mapped pinned memory");
    c->mb_dev = static_cast<uint8_t*>(dev);
    c->ml = ft::mailbox_layout(hi.H, hi.k_max, hi.B_max);
    c->host = hb;
    return FT_OK;
}

int32_t ft_recommend_backend(double cpu_gbs, double pcie_gbs) {
    return cpu_gbs > 2.0 * pcie_gbs ? FT_BACKEND_HYBRID : FT_BACKEND_OFFLOAD;
}

ft_status ft_profile_bandwidth(ft_cache* c, ft_host_branch* hb, int32_t n, void* stream, ft_bw_profile* out) {
    NvtxRange range("ft_profile_bandwidth");
    if (!c) return FT_ERR_ARG;
    if (!hb || !out) return fail(c, FT_ERR_ARG, "NULL argument");
    ft::HostBranchInfo hi;
    if (!ft::host_branch_info(hb, &hi) || hi.pool != c->d.host_pool || hi.H != c->d.H || hi.I != c->d.I ||
        hi.format != c->d.format || hi.L != c->d.L || hi.E != c->d.E)
        return fail(c, FT_ERR_ARG, "host branch of another pool or shape");
    if (n < 1 || n > c->C || n > c->d.L * c->d.E) return fail(c, FT_ERR_ARG, "n_records outside [1, min(C, L*E)]");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return cuda_fail(c, cudaGetLastError(), "capture query");
    if (cs != cudaStreamCaptureStatusNone) return fail(c, FT_ERR_STATE, "profile while capturing");
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->copy_stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "profile drain");
    // the GPU fill path: records 0..n-1 gathered into slots 0..n-1
    std::vector<int32_t> lists(2 * (size_t)n + 4);
    for (int i = 0; i < n; ++i) { lists[i] = i; lists[n + i] = i; }
    lists[2 * n] = n;
    int32_t* dv = nullptr;
    e = cudaMalloc(&dv, lists.size() * 4);
    if (e != cudaSuccess) return cuda_fail(c, e, "profile lists");
    ft::PrefillGatherArgs ga{};
    ga.host_pool = c->host_pool_dev;
    ga.slot_buf = c->slot_buf;
    ga.rec_bytes = c->rec.bytes;
    ga.fill_flat = dv;
    ga.fill_slot = dv + n;
    ga.n_fill = dv + 2 * n;
    cudaEvent_t ev[2] = {nullptr, nullptr};
    float ms = 0.f;
    double t_p = 0, t_c = 0, t_pov = 0, t_cov = 0;
    int reps = 1;
    const double bytes = (double)n * (double)c->rec.bytes;
    e = cudaMemcpy(dv, lists.data(), lists.size() * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaEventCreate(&ev[0]);
    if (e == cudaSuccess) e = cudaEventCreate(&ev[1]);
    if (e == cudaSuccess) e = ft::launch_pf_gather(ga, false, s);          // warm-up
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaEventRecord(ev[0], s);
    if (e == cudaSuccess) e = ft::launch_pf_gather(ga, false, s);
    if (e == cudaSuccess) e = cudaEventRecord(ev[1], s);
    if (e == cudaSuccess) e = cudaEventSynchronize(ev[1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, ev[0], ev[1]);
    t_p = ms / 1e3;
    // the host branch alone (one warm-up run)
    if (e == cudaSuccess) {
        ft::host_branch_run_flats(hb, lists.data(), n);
        t_c = ft::host_branch_run_flats(hb, lists.data(), n);
        if (t_c <= 0) e = cudaErrorInvalidValue;
    }
    // both together: enough gathers to cover the host run
    if (e == cudaSuccess) {
        reps = (int)std::max(1.0, std::min(64.0, std::round(t_c / std::max(t_p, 1e-9))));
        e = cudaEventRecord(ev[0], s);
        for (int r = 0; r < reps && e == cudaSuccess; ++r) e = ft::launch_pf_gather(ga, false, s);
        if (e == cudaSuccess) e = cudaEventRecord(ev[1], s);
    }
    if (e == cudaSuccess) {
        t_cov = ft::host_branch_run_flats(hb, lists.data(), n);
        e = cudaEventSynchronize(ev[1]);
    }
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, ev[0], ev[1]);
    t_pov = ms / 1e3 / reps;
    for (auto v : ev) if (v) cudaEventDestroy(v);
    cudaFree(dv);
    // the gathers overwrote slots 0..n-1 behind the tables: empty the cache
    if (e == cudaSuccess) {
        uint8_t* ws = c->workspace;
        c->buffer_layer[0] = c->buffer_layer[1] = -1;
        e = launch_init_tables(reinterpret_cast<int32_t*>(ws + c->ws.slot_for_id), c->d.L * c->d.E,
                               reinterpret_cast<int32_t*>(ws + c->ws.id_of_slot),
                               reinterpret_cast<long long*>(ws + c->ws.usage),
                               reinterpret_cast<int32_t*>(ws + c->ws.lru_order), c->C,
                               reinterpret_cast<DevScalars*>(ws + c->ws.scalars), false, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    if (e != cudaSuccess) return cuda_fail(c, e, "bandwidth profile");
    out->n_records = n;
    out->pcie_gbs = bytes / t_p / 1e9;
    out->cpu_gbs = bytes / t_c / 1e9;
    out->pcie_ov_gbs = bytes / t_pov / 1e9;
    out->cpu_ov_gbs = t_cov > 0 ? bytes / t_cov / 1e9 : 0.0;
    out->recommend = ft_recommend_backend(out->cpu_gbs, out->pcie_gbs);
    out->f_q16 = ft_split_from_overlap(out->pcie_ov_gbs, out->cpu_ov_gbs);
    return FT_OK;
}

ft_status ft_cache_status(ft_cache* c, int32_t* device_status) {
    if (!c || !device_status) return FT_ERR_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    int* st = reinterpret_cast<int*>(c->workspace + c->ws.scalars + offsetof(DevScalars, status));
    if (e == cudaSuccess) e = cudaMemcpy(device_status, st, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(st, 0, 4);
    // a decode wait that ran out may have left its read counter non-zero
    if (e == cudaSuccess && (*device_status & FT_DEV_TIMEOUT))
        e = cudaMemset(c->workspace + c->ws.sync + 8, 0, 4);
    return e == cudaSuccess ? FT_OK : cuda_fail(c, e, "status");
}

// ------------------------------------------------------------------ utilities

ft_status ft_quantize_experts(const float* w_gu, const float* w_d, int32_t n, int32_t H,
                              int32_t I, void* records, void* stream) {
    if (!w_gu || !w_d || !records || n < 1 || H < 64 || H % 64 || I < 32 || I % 32) return FT_ERR_ARG;
    if (!aligned(w_gu, 16) || !aligned(w_d, 16) || !aligned(records, 256)) return FT_ERR_ARG;
    cudaError_t e = launch_quantize(w_gu, w_d, n, H, I, static_cast<uint8_t*>(records),
                                    record_layout(H, I).bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

ft_status ft_quantize_experts_mx(const float* w_gu, const float* w_d, int32_t n, int32_t H,
                                 int32_t I, void* records, void* stream) {
    if (!w_gu || !w_d || !records || n < 1 || H < 64 || H % 64 || I < 32 || I % 32) return FT_ERR_ARG;
    if (!aligned(w_gu, 16) || !aligned(w_d, 16) || !aligned(records, 256)) return FT_ERR_ARG;
    cudaError_t e = launch_quantize_mx(w_gu, w_d, n, H, I, static_cast<uint8_t*>(records),
                                       record_layout(H, I, FT_FORMAT_MXFP4).bytes,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

ft_status ft_pinned_alloc(size_t bytes, void** out) {
    if (!out || !bytes) return FT_ERR_ARG;
    *out = nullptr;
    cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *out = nullptr;
        return FT_ERR_CUDA;
    }
    return FT_OK;
}

ft_status ft_pinned_free(void* p) {
    if (!p) return FT_ERR_ARG;
    return cudaFreeHost(p) == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

ft_status ft_check_bounded_waits(uint32_t* expired) {
    if (!expired) return FT_ERR_ARG;
    unsigned bits = 0;
    if (check_bounded_waits(&bits) != cudaSuccess) return FT_ERR_CUDA;
    *expired = bits;
    return FT_OK;
}

ft_status ft_measure_h2d(const void* pinned, void* dev, size_t bytes, int32_t reps, double* gbps) {
    if (!pinned || !dev || !bytes || reps < 1 || !gbps) return FT_ERR_ARG;
    cudaStream_t s;
    cudaEvent_t a, b;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return FT_ERR_CUDA;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    float best = 0.f;
    cudaError_t e = cudaSuccess;
    for (int r = 0; r <= reps && e == cudaSuccess; ++r) {   // first copy is a warm-up
        cudaEventRecord(a, s);
        e = cudaMemcpyAsync(dev, pinned, bytes, cudaMemcpyHostToDevice, s);
        cudaEventRecord(b, s);
        if (e == cudaSuccess) e = cudaEventSynchronize(b);
        float ms = 0.f;
        cudaEventElapsedTime(&ms, a, b);
        if (r > 0 && (best == 0.f || ms < best)) best = ms;
    }
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaStreamDestroy(s);
    if (e != cudaSuccess || best <= 0.f) return FT_ERR_CUDA;
    *gbps = (double)bytes / (best * 1e-3) / 1e9;
    return FT_OK;
}

const char* ft_status_string(ft_status s) {
    if (s < 0 || s > 6) return "unknown status";
    return kStatusNames[s];
}

const char* ft_last_error(const ft_cache* c) { return c ? c->err : ""; }

}  // extern "C"
