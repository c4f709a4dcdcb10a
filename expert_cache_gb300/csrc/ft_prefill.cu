// Prefill of one MoE layer over a chunk of T tokens with full-layer double buffering.
//
// [EXPLAINER §4.1-4.3]: borrow two whole-layer buffers from the global slot pool;
// while layer l computes from buffer l mod 2, every expert of layer l+1 streams
// into the other buffer; T_layer ~ max(T_compute, T_link) instead of the sum.
// [JUHE "Prefill 为什么不能也按需加载"]: double buffering needs cache_size >= 2E.
// Without the flag only buffer 0 is used and each layer is loaded, then computed.
//
// When two whole layers do not fit (capacity < 2E with the double buffer asked for,
// capacity < E without it), or when FT_PREFILL_ON_DEMAND asks for it, the call falls
// back to loading on demand ([EXPLAINER §4.3]): the routed union of the layer (every
// expert some token routes to) goes through the global LRU like decode misses with
// every miss filled, in groups of at most C experts in ascending id; per group the
// table kernel picks the victims, a gather kernel streams the missing records from
// the pinned pool into them over the host link, and the two GEMMs run on the group's
// rows before the next group may evict them.  A group is gathered in kOdSub batches
// on the copy stream (one CTA on half of the SMs), and the GEMMs of batch j run on
// the caller's stream as soon as its records are in, beside the gather of batch j+1:
// a batch's victims are slots no other expert of the group uses, so the batches need
// no other order.  (8 batches per group measured best against 2, 4 and 16, and half of
// the SMs for the gathers against a quarter and all.)
//
// Streams: the caller's stream computes; the cache's copy stream moves whole layers
// (E contiguous records of the pool into E contiguous slots: one streaming kernel of
// SM loads from the device-mapped pool per layer.  On some boxes a copy-engine
// transfer issued on this stream ran at 72-90 GB/s while copies on another stream ran
// at 211 GB/s; SM loads do not depend on the copy engine a stream is given), and the
// on-demand batches.
//   copy(l+1 -> buffer b')  waits for everything enqueued before this call (the
//                            previous layer, the last reader of b');
//   compute(l)              waits for copy(l -> b).
#include <algorithm>
#include <cstdio>

#include "ft_prefill.cuh"
#include "ft_umma.cuh"

using namespace ft;

extern "C" ft_status ft_moe_prefill_layer(ft_cache* c, int32_t layer, const void* x,
                                          const int32_t* topk_ids, const float* topk_w,
                                          int32_t T, int32_t k, float* y, int32_t flags,
                                          void* debug_h, void* stream) {
    NvtxRange range("ft_moe_prefill_layer");
    if (!c) return FT_ERR_ARG;
    auto fail = [&](ft_status s, const char* m) { snprintf(c->err, sizeof(c->err), "%s", m); return s; };
    const ft_cache_desc& d = c->d;
    if (d.T_max <= 0) return fail(FT_ERR_STATE, "cache created without prefill support (T_max = 0)");
    if (d.H % 256 || d.I % 256) return fail(FT_ERR_ARG, "prefill needs H and I multiples of 256");
    if (layer < 0 || layer >= d.L) return fail(FT_ERR_ARG, "layer out of range");
    if (T < 1 || T > d.T_max) return fail(FT_ERR_ARG, "T outside [1, T_max]");
    if (k < 1 || k > d.k_max) return fail(FT_ERR_ARG, "k outside [1, k_max]");
    if (!x || !topk_ids || !topk_w || !y) return fail(FT_ERR_ARG, "NULL argument");
    if (((uintptr_t)x) % 16 || ((uintptr_t)y) % 16) return fail(FT_ERR_ARG, "x and y must be 16-byte aligned");
    if (flags & ~(FT_PREFILL_DOUBLE_BUFFER | FT_PREFILL_DEBUG_X | FT_PREFILL_ON_DEMAND))
        return fail(FT_ERR_ARG, "unknown prefill flag");
    if (!c->maps_ok) return fail(FT_ERR_CUDA, "TMA descriptors could not be built");

    // Which path: whole-layer buffers (double, or single when no double buffer is
    // asked for) when they fit; otherwise, or when asked, the routed union on demand.
    const bool force_od = (flags & FT_PREFILL_ON_DEMAND) != 0;
    const bool want_db = (flags & FT_PREFILL_DOUBLE_BUFFER) != 0;
    const bool db = want_db && !force_od && c->C >= 2 * d.E;
    const bool whole = !force_od && (db || (!want_db && c->C >= d.E));

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t rec = c->rec.bytes;
    const size_t layer_bytes = (size_t)d.E * rec;
    const int b = db ? layer % 2 : 0;
    uint8_t* ws = c->workspace;
    DevScalars* sc = reinterpret_cast<DevScalars*>(ws + c->ws.scalars);
    cudaError_t e = cudaSuccess;

    // whole-layer copy host pool -> buffer on the copy stream, after everything enqueued
    // on the caller's stream before this call (the last reader of the buffer)
    auto copy_layer = [&](int l, int buf) -> cudaError_t {
        cudaStreamWaitEvent(c->copy_stream, c->entry_ev, 0);
        cudaEvent_t e1 = nullptr;
        if ((c->prof & (1u << 4)) && c->prof_n * 2 + 2 <= ft_cache::kProfEvents) {
            const int i = c->prof_n++;
            c->prof_kind[i] = 4;
            cudaEventRecord(c->prof_ev[2 * i], c->copy_stream);
            e1 = c->prof_ev[2 * i + 1];
        }
        cudaError_t r = launch_pf_stream(c->host_pool_dev + (size_t)l * layer_bytes,
                                         c->slot_buf + (size_t)buf * layer_bytes, layer_bytes,
                                         c->copy_stream);
        if (e1) cudaEventRecord(e1, c->copy_stream);
        cudaEventRecord(c->copy_done[buf], c->copy_stream);
        c->buffer_layer[buf] = l;
        return r;
    };
    auto prof_kernel = [&](int kind, auto&& launch) -> cudaError_t {
        const int i = prof_begin(c, kind, s);
        cudaError_t r = launch();
        prof_end(c, i, s);
        return r;
    };

    if (whole) {
        // 1. layer -> buffer b (already there when the previous call prefetched it)
        cudaEventRecord(c->entry_ev, s);
        if (c->buffer_layer[b] != layer) {
            if ((e = copy_layer(layer, b)) != cudaSuccess) return fail(FT_ERR_CUDA, "layer copy");
        }
        cudaStreamWaitEvent(s, c->copy_done[b], 0);

        // 2. slot tables: layer -> buffer b, layer+1 -> the other buffer
        const int lb = (db && layer + 1 < d.L) ? layer + 1 : -1;
        PrefillTablesArgs ta;
        ta.slot_for_id = reinterpret_cast<int32_t*>(ws + c->ws.slot_for_id);
        ta.id_of_slot = reinterpret_cast<int32_t*>(ws + c->ws.id_of_slot);
        ta.usage = reinterpret_cast<long long*>(ws + c->ws.usage);
        ta.lru_order = reinterpret_cast<int32_t*>(ws + c->ws.lru_order);
        ta.sc = sc;
        ta.C = c->C;
        ta.E = d.E;
        ta.la = layer; ta.ba = b;
        ta.lb = lb; ta.bb = 1 - b;
        if ((e = launch_pf_tables(ta, s)) != cudaSuccess) return fail(FT_ERR_CUDA, "prefill table launch");

        // 3. stream layer+1 into the other buffer while this layer computes
        if (lb >= 0 && c->buffer_layer[1 - b] != lb) {
            if ((e = copy_layer(lb, 1 - b)) != cudaSuccess) return fail(FT_ERR_CUDA, "prefetch copy");
            c->copy_pending = true;
        }
    } else {
        // on demand: slots anywhere in the cache may be rewritten, so a stream-in of
        // an earlier double-buffered call must have landed, and no buffer stays valid
        if (c->copy_pending) {
            cudaStreamWaitEvent(s, c->copy_done[0], 0);
            cudaStreamWaitEvent(s, c->copy_done[1], 0);
            c->copy_pending = false;
        }
        c->buffer_layer[0] = c->buffer_layer[1] = -1;
    }

    // 4. compute
    PrefillArgs a;
    a.sc = sc;
    a.T = T; a.k = k; a.E = d.E; a.H = d.H; a.I = d.I;
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.ids = topk_ids;
    a.w = topk_w;
    a.y = y;
    a.chunk_cnt = reinterpret_cast<int32_t*>(ws + c->ws.pf_chunk_cnt);
    a.offsets = reinterpret_cast<int32_t*>(ws + c->ws.pf_offsets);
    a.mtile_prefix = reinterpret_cast<int32_t*>(ws + c->ws.pf_mtile);
    a.perm = reinterpret_cast<int32_t*>(ws + c->ws.pf_perm);
    a.route_pos = reinterpret_cast<int32_t*>(ws + c->ws.pf_route_pos);
    a.a_codes = ws + c->ws.pf_a_codes;
    a.a_scales = ws + c->ws.pf_a_scales;
    a.h_codes = ws + c->ws.pf_h_codes;
    a.h_scales = ws + c->ws.pf_h_scales;
    a.O = reinterpret_cast<float*>(ws + c->ws.pf_o);
    a.debug_h = static_cast<uint8_t*>(debug_h);
    const size_t RT = (size_t)T * k;
    if (debug_h) cudaMemsetAsync(debug_h, 0, RT * (d.I / 2 + d.I / 16), s);

    e = prof_kernel(3, [&] { return launch_pf_sort_quant(a, s); });
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, "route sort launch");
    if (debug_h && (flags & FT_PREFILL_DEBUG_X)) {
        // the quantised activations as the GEMM reads them (sorted rows) and the
        // sorted row of every route, after the h region of the debug buffer
        uint8_t* dx = static_cast<uint8_t*>(debug_h) + RT * (d.I / 2 + d.I / 16);
        e = cudaMemcpyAsync(dx, a.route_pos, RT * 4, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dx + RT * 4, a.a_codes, RT * (d.H / 2), cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dx + RT * (4 + d.H / 2), a.a_scales, RT * (d.H / 16),
                                cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return fail(FT_ERR_CUDA, "debug copy of the quantised x");
    }

    UmmaArgs g;
    g.E = d.E;
    g.R_max = std::max(d.T_max * d.k_max, 128);
    g.R_total = (int)RT;
    g.I = d.I; g.H = d.H;
    g.slot0 = b * d.E;
    g.slot_of = nullptr;
    g.mrange = nullptr;
    g.mx = d.format == FT_FORMAT_MXFP4 ? 1 : 0;
    g.slot_buf = c->slot_buf;
    g.rec_bytes = rec;
    g.offsets = a.offsets;
    g.mtile_prefix = a.mtile_prefix;
    g.perm = a.perm;
    g.w = topk_w;
    g.h_codes = a.h_codes;
    g.h_scales = a.h_scales;
    g.debug_h = a.debug_h;
    g.O = a.O;
    g.status = &sc->status;
    const int grid = sm_count();

    auto gemms = [&]() -> ft_status {
        g.kind = 1;
        g.K = d.H;
        g.n_tiles_n = d.I / 128;
        g.off_b_scales = c->rec.gu_scales;
        g.off_tscale = c->rec.s_gu;
        g.a_scales = a.a_scales;
        if (prof_kernel(1, [&] { return launch_umma(c->map_a1, c->map_b1, g, grid, s); }) != cudaSuccess)
            return fail(FT_ERR_CUDA, "GEMM1 launch");
        g.kind = 2;
        g.K = d.I;
        g.n_tiles_n = d.H / 256;
        g.off_b_scales = c->rec.d_scales;
        g.off_tscale = c->rec.s_d;
        g.a_scales = a.h_scales;
        if (prof_kernel(2, [&] { return launch_umma(c->map_a2, c->map_b2, g, grid, s); }) != cudaSuccess)
            return fail(FT_ERR_CUDA, "GEMM2 launch");
        return FT_OK;
    };

    if (whole) {
        const ft_status st = gemms();
        if (st != FT_OK) return st;
    } else {
        // the routed union in groups of at most C experts: tables, fills over the host
        // link into the victim slots, then the two GEMMs over the group's rows
        PrefillDemandArgs da;
        da.slot_for_id = reinterpret_cast<int32_t*>(ws + c->ws.slot_for_id);
        da.id_of_slot = reinterpret_cast<int32_t*>(ws + c->ws.id_of_slot);
        da.usage = reinterpret_cast<long long*>(ws + c->ws.usage);
        da.lru_order = reinterpret_cast<int32_t*>(ws + c->ws.lru_order);
        da.sc = sc;
        da.C = c->C;
        da.E = d.E;
        da.layer = layer;
        da.offsets = a.offsets;
        da.slot_of = reinterpret_cast<int32_t*>(ws + c->ws.pf_slot_of);
        da.mtile = reinterpret_cast<int32_t*>(ws + c->ws.pf_gmtile);
        da.fill_flat = reinterpret_cast<int32_t*>(ws + c->ws.pf_fill_flat);
        da.fill_slot = reinterpret_cast<int32_t*>(ws + c->ws.pf_fill_slot);
        da.n_fill = reinterpret_cast<int32_t*>(ws + c->ws.pf_nfill);
        da.sub_fill = reinterpret_cast<int32_t*>(ws + c->ws.pf_sub);
        da.sub_tile = da.sub_fill + (kOdSub + 1);
        PrefillGatherArgs ga;
        ga.host_pool = c->host_pool_dev;
        ga.slot_buf = c->slot_buf;
        ga.rec_bytes = rec;
        ga.fill_flat = da.fill_flat;
        ga.fill_slot = da.fill_slot;
        ga.n_fill = da.n_fill;
        ga.sub_fill = da.sub_fill;
        g.slot_of = da.slot_of;
        g.mtile_prefix = da.mtile;
        // a batch's gather on the copy stream, timed there when copies are profiled
        auto gather = [&](int j) -> cudaError_t {
            cudaEvent_t e1 = nullptr;
            if ((c->prof & (1u << 4)) && c->prof_n * 2 + 2 <= ft_cache::kProfEvents) {
                const int i = c->prof_n++;
                c->prof_kind[i] = 4;
                cudaEventRecord(c->prof_ev[2 * i], c->copy_stream);
                e1 = c->prof_ev[2 * i + 1];
            }
            ga.sub = j;
            const cudaError_t r = launch_pf_gather(ga, true, c->copy_stream);
            if (e1) cudaEventRecord(e1, c->copy_stream);
            return r;
        };
        const int groups = (d.E + c->C - 1) / c->C;
        for (int grp = 0; grp < groups; ++grp) {
            da.group = grp;
            if (prof_kernel(3, [&] { return launch_pf_demand_tables(da, s); }) != cudaSuccess)
                return fail(FT_ERR_CUDA, "on-demand table launch");
            cudaEventRecord(c->od_ev[kOdSub], s);
            cudaStreamWaitEvent(c->copy_stream, c->od_ev[kOdSub], 0);
            for (int j = 0; j < kOdSub; ++j) {
                if (gather(j) != cudaSuccess) return fail(FT_ERR_CUDA, "on-demand gather launch");
                cudaEventRecord(c->od_ev[j], c->copy_stream);
            }
            for (int j = 0; j < kOdSub; ++j) {
                cudaStreamWaitEvent(s, c->od_ev[j], 0);
                g.mrange = da.sub_tile + j;
                const ft_status st = gemms();
                if (st != FT_OK) return st;
            }
            g.mrange = nullptr;
        }
    }

    e = prof_kernel(3, [&] { return launch_pf_combine(a, s); });
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, "combine launch");
    if (whole) cudaEventRecord(c->compute_done[b], s);
    return FT_OK;
}
