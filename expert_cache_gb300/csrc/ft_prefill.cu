// Prefill of one MoE layer over a chunk of T tokens with full-layer double buffering.
//
// [EXPLAINER §4.1-4.3]: borrow two whole-layer buffers from the global slot pool;
// while layer l computes from buffer l mod 2, every expert of layer l+1 streams
// into the other buffer; T_layer ~ max(T_compute, T_link) instead of the sum.
// [JUHE "Prefill 为什么不能也按需加载"]: double buffering needs cache_size >= 2E.
// Without the flag only buffer 0 is used and each layer is loaded, then computed.
//
// Streams: the caller's stream computes; the cache's copy stream moves whole layers
// (E contiguous records of the pool into E contiguous slots: one copy per layer).
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
    const bool db = (flags & FT_PREFILL_DOUBLE_BUFFER) != 0;
    if (db && c->C < 2 * d.E) return fail(FT_ERR_CAPACITY, "double buffering needs capacity >= 2 * E");
    if (c->C < d.E) return fail(FT_ERR_CAPACITY, "prefill needs capacity >= E");
    if (!c->maps_ok) return fail(FT_ERR_CUDA, "TMA descriptors could not be built");

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t rec = c->rec.bytes;
    const size_t layer_bytes = (size_t)d.E * rec;
    const uint8_t* host = static_cast<const uint8_t*>(d.host_pool);
    const int b = db ? layer % 2 : 0;
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
        cudaError_t r = cudaMemcpyAsync(c->slot_buf + (size_t)buf * layer_bytes,
                                        host + (size_t)l * layer_bytes, layer_bytes,
                                        cudaMemcpyHostToDevice, c->copy_stream);
        if (e1) cudaEventRecord(e1, c->copy_stream);
        cudaEventRecord(c->copy_done[buf], c->copy_stream);
        c->buffer_layer[buf] = l;
        return r;
    };

    // 1. layer -> buffer b (already there when the previous call prefetched it)
    cudaEventRecord(c->entry_ev, s);
    if (c->buffer_layer[b] != layer) {
        if ((e = copy_layer(layer, b)) != cudaSuccess) return fail(FT_ERR_CUDA, "layer copy");
    }
    cudaStreamWaitEvent(s, c->copy_done[b], 0);

    // 2. slot tables: layer -> buffer b, layer+1 -> the other buffer
    const int lb = (db && layer + 1 < d.L) ? layer + 1 : -1;
    uint8_t* ws = c->workspace;
    PrefillTablesArgs ta;
    ta.slot_for_id = reinterpret_cast<int32_t*>(ws + c->ws.slot_for_id);
    ta.id_of_slot = reinterpret_cast<int32_t*>(ws + c->ws.id_of_slot);
    ta.usage = reinterpret_cast<long long*>(ws + c->ws.usage);
    ta.lru_order = reinterpret_cast<int32_t*>(ws + c->ws.lru_order);
    ta.sc = reinterpret_cast<DevScalars*>(ws + c->ws.scalars);
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

    // 4. compute
    PrefillArgs a;
    a.sc = ta.sc;
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

    auto prof_kernel = [&](int kind, auto&& launch) -> cudaError_t {
        cudaEvent_t e0 = nullptr, e1 = nullptr;
        if (c->prof & (1u << kind)) {
            if (c->prof_n * 2 + 2 > ft_cache::kProfEvents) return cudaErrorInvalidValue;
            const int i = c->prof_n++;
            c->prof_kind[i] = kind;
            e0 = c->prof_ev[2 * i];
            e1 = c->prof_ev[2 * i + 1];
            cudaEventRecord(e0, s);
        }
        cudaError_t r = launch();
        if (e1) cudaEventRecord(e1, s);
        return r;
    };

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
    g.status = &ta.sc->status;
    const int grid = sm_count();

    g.kind = 1;
    g.K = d.H;
    g.n_tiles_n = d.I / 128;
    g.off_b_scales = c->rec.gu_scales;
    g.off_tscale = c->rec.s_gu;
    g.a_scales = a.a_scales;
    e = prof_kernel(1, [&] { return launch_umma(c->map_a1, c->map_b1, g, grid, s); });
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, "GEMM1 launch");

    g.kind = 2;
    g.K = d.I;
    g.n_tiles_n = d.H / 256;
    g.off_b_scales = c->rec.d_scales;
    g.off_tscale = c->rec.s_d;
    g.a_scales = a.h_scales;
    e = prof_kernel(2, [&] { return launch_umma(c->map_a2, c->map_b2, g, grid, s); });
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, "GEMM2 launch");

    e = prof_kernel(3, [&] { return launch_pf_combine(a, s); });
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, "combine launch");
    cudaEventRecord(c->compute_done[b], s);
    return FT_OK;
}
