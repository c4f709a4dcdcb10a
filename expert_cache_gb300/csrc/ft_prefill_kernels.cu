// Prefill helper kernels: slot tables of the full-layer buffers, stable route sort
// by expert, NVFP4 activation quantisation into sorted row order, and the combine.
//
// [EXPLAINER §4.2-4.3] two whole-layer buffers borrowed from the global slot pool;
// what they hold afterwards is decode's initial cache.  [EXPLAINER §1.1] the MoE
// output y[t] = sum_j p_{t,j} Expert_{l,e_{t,j}}(x_t).  The activation quantiser
// (unit tensor scale, E4M3 per 16, E2M1 codes) runs in fp32 IEEE steps.
#include "ft_prefill.cuh"
#include "ft_quant.cuh"

namespace ft {

// ------------------------------------------------------------------ slot tables
// One CTA of 1024 threads.  Maps layer `la` into buffer ba (and, if lb >= 0, layer
// lb into buffer bb), with the same outcome as loading expert by expert: each
// buffer slot b*E + e ends up holding flat id l*E + e; an id evicted from a buffer
// slot is unmapped; a slot outside the buffers that held an expert of the loaded
// layer becomes free.  Then every buffer slot is stamped with the call's tick and
// the LRU order is rebuilt: free slots ascending, untouched occupied slots in their
// old order, then the touched slots ascending.
__global__ void __launch_bounds__(1024, 1) pf_tables_kernel(PrefillTablesArgs a) {
    __shared__ int s_scan[33];
    __shared__ long long s_tick;
    const int tid = threadIdx.x;
    const int C = a.C, E = a.E;
    if (tid == 0) {
        s_tick = a.sc->tick + 1;
        a.sc->tick = s_tick;
    }
    __syncthreads();
    for (int pass = 0; pass < 2; ++pass) {
        const int l = pass == 0 ? a.la : a.lb;
        const int b = pass == 0 ? a.ba : a.bb;
        if (l < 0) break;
        for (int s = tid; s < C; s += 1024) {
            const int f_old = a.id_of_slot[s];
            const bool in_buf = s >= b * E && s < b * E + E;
            if (in_buf) {
                const int f_new = l * E + (s - b * E);
                if (f_old >= 0 && f_old != f_new) a.slot_for_id[f_old] = -1;
            } else if (f_old >= 0 && f_old / E == l) {
                a.id_of_slot[s] = -1;
                a.usage[s] = -1;
            }
        }
        __syncthreads();
        for (int e = tid; e < E; e += 1024) {
            const int s = b * E + e;
            a.id_of_slot[s] = l * E + e;
            a.slot_for_id[l * E + e] = s;
        }
        __syncthreads();
    }
    // touched = slots of the loaded buffers
    auto touched = [&](int s) {
        return (s >= a.ba * E && s < a.ba * E + E) || (a.lb >= 0 && s >= a.bb * E && s < a.bb * E + E);
    };
    const int nc = (C + 1023) / 1024;
    // read the old order before rewriting it
    int old_loc[kSlotsPerThread];
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        const int pos = tid * nc + j;
        old_loc[j] = (j < nc && pos < C) ? a.lru_order[pos] : -1;
    }
    int n_free = 0, n_keep = 0, n_touch = 0;
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        const int s = tid * nc + j;          // slot-index order (free and touched)
        if (j < nc && s < C) {
            if (touched(s)) ++n_touch;
            else if (a.id_of_slot[s] < 0) ++n_free;
        }
        const int so = old_loc[j];           // old LRU order (kept occupied)
        if (so >= 0 && !touched(so) && a.id_of_slot[so] >= 0) ++n_keep;
    }
    int tot_free = 0, tot_keep = 0, tot_touch = 0;
    int r_free = block_exclusive_scan(n_free, &tot_free, s_scan);
    int r_keep = block_exclusive_scan(n_keep, &tot_keep, s_scan);
    int r_touch = block_exclusive_scan(n_touch, &tot_touch, s_scan);
    const long long tick = s_tick;
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        const int s = tid * nc + j;
        if (j < nc && s < C) {
            if (touched(s)) {
                a.usage[s] = tick;
                a.lru_order[tot_free + tot_keep + r_touch++] = s;
            } else if (a.id_of_slot[s] < 0) {
                a.lru_order[r_free++] = s;
            }
        }
        const int so = old_loc[j];
        if (so >= 0 && !touched(so) && a.id_of_slot[so] >= 0) a.lru_order[tot_free + r_keep++] = so;
    }
}

// ------------------------------------------------------------------ on-demand tables
// One CTA of 1024 threads per group.  Expert e belongs to thread e / ne (ne experts
// per thread, contiguous) and slot position p to thread p / nc, so block scans run
// in ascending expert id and ascending LRU position.
__global__ void __launch_bounds__(1024, 1) pf_demand_tables_kernel(PrefillDemandArgs a) {
    __shared__ int s_scan[33];
    __shared__ uint32_t s_hit[kMaxC / 32];        // slots held by a hit of this group
    __shared__ uint32_t s_touch[kMaxC / 32];      // hits and victims
    const int tid = threadIdx.x, E = a.E, C = a.C;
    const int ne = (E + 1023) / 1024, nc = (C + 1023) / 1024, nw = (C + 31) / 32;
    for (int w = tid; w < nw; w += 1024) { s_hit[w] = 0; s_touch[w] = 0; }
    // ---- union rank of every routed expert; group membership
    int used[kExpertsPerThread];
    int n_used = 0;
#pragma unroll
    for (int j = 0; j < kExpertsPerThread; ++j) {
        const int e = tid * ne + j;
        used[j] = (j < ne && e < E && a.offsets[e + 1] > a.offsets[e]) ? 1 : 0;
        n_used += used[j];
    }
    int U = 0;
    int rank = block_exclusive_scan(n_used, &U, s_scan);
    const int g0 = a.group * C;
    const int n_members = min(C, U - g0);
    int member[kExpertsPerThread], slot[kExpertsPerThread];
    int n_miss = 0;
#pragma unroll
    for (int j = 0; j < kExpertsPerThread; ++j) {
        member[j] = used[j] && rank >= g0 && rank < g0 + C;
        rank += used[j];
        slot[j] = -1;
        if (member[j]) {
            const int e = tid * ne + j;
            slot[j] = a.slot_for_id[a.layer * E + e];
            if (slot[j] >= 0) atomicOr(&s_hit[slot[j] >> 5], 1u << (slot[j] & 31));
            else ++n_miss;
        }
    }
    if (n_members <= 0) {                          // nothing in this group
#pragma unroll
        for (int j = 0; j < kExpertsPerThread; ++j) {
            const int e = tid * ne + j;
            if (j < ne && e < E) { a.slot_of[e] = -1; a.mtile[e] = 0; }
        }
        if (tid == 0) {
            a.mtile[E] = 0;
            *a.n_fill = 0;
            if (a.group == 0) a.sc->tick = a.sc->tick + 1;   // the call still ticks once
        }
        if (tid <= kOdSub) { a.sub_fill[tid] = 0; a.sub_tile[tid] = 0; }
        return;
    }
    int m = 0;
    int miss_rank = block_exclusive_scan(n_miss, &m, s_scan);   // also orders s_hit
    const long long tick = a.sc->tick + 1;
    // ---- victims: the first m entries of the LRU order that no hit holds
    int ent[kSlotsPerThread];
    int n_keep = 0;
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        const int pos = tid * nc + j;
        ent[j] = (j < nc && pos < C) ? a.lru_order[pos] : -1;
        if (ent[j] >= 0 && !((s_hit[ent[j] >> 5] >> (ent[j] & 31)) & 1u)) ++n_keep;
    }
    int vrank = block_exclusive_scan(n_keep, nullptr, s_scan);
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        if (ent[j] >= 0 && !((s_hit[ent[j] >> 5] >> (ent[j] & 31)) & 1u)) {
            if (vrank < m) a.fill_slot[vrank] = ent[j];
            ++vrank;
        }
    }
    __syncthreads();                               // fill_slot complete (same CTA)
    // ---- misses take their victims in ascending expert id; evicted ids unmapped
#pragma unroll
    for (int j = 0; j < kExpertsPerThread; ++j) {
        const int e = tid * ne + j;
        if (member[j] && slot[j] < 0) {
            const int v = a.fill_slot[miss_rank];
            const int flat = a.layer * E + e;
            const int old = a.id_of_slot[v];
            if (old >= 0) a.slot_for_id[old] = -1;
            a.slot_for_id[flat] = v;
            a.id_of_slot[v] = flat;
            a.fill_flat[miss_rank] = flat;
            slot[j] = v;
            ++miss_rank;
        }
        if (j < ne && e < E) a.slot_of[e] = member[j] ? slot[j] : -1;
        if (member[j]) atomicOr(&s_touch[slot[j] >> 5], 1u << (slot[j] & 31));
    }
    // ---- 128-row tile prefix over the group's experts
    int tiles = 0;
#pragma unroll
    for (int j = 0; j < kExpertsPerThread; ++j) {
        const int e = tid * ne + j;
        if (member[j]) tiles += (a.offsets[e + 1] - a.offsets[e] + 127) / 128;
    }
    int all_tiles = 0;
    int toff = block_exclusive_scan(tiles, &all_tiles, s_scan);   // also orders s_touch
#pragma unroll
    for (int j = 0; j < kExpertsPerThread; ++j) {
        const int e = tid * ne + j;
        if (j < ne && e < E) {
            a.mtile[e] = toff;
            if (member[j]) toff += (a.offsets[e + 1] - a.offsets[e] + 127) / 128;
        }
    }
    if (tid == 0) { a.mtile[E] = all_tiles; *a.n_fill = m; }
    __syncthreads();                               // mtile and fill_flat complete
    // ---- batches: batch j starts at fill j*m/kOdSub and at the first tile of that
    // fill's expert (fills run in ascending expert id), so its tiles are those of the
    // members from that expert up to the next batch's; batch 0 starts at tile 0
    if (tid <= kOdSub) {
        const int f = (int)((long long)tid * m / kOdSub);
        int t = all_tiles;
        if (tid == 0) t = 0;
        else if (f < m) t = a.mtile[a.fill_flat[f] - a.layer * E];
        a.sub_fill[tid] = f;
        a.sub_tile[tid] = t;
    }
    // ---- LRU order: untouched slots keep their order, touched ones follow ascending
    int n_untouched = 0;
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j)
        if (ent[j] >= 0 && !((s_touch[ent[j] >> 5] >> (ent[j] & 31)) & 1u)) ++n_untouched;
    int tot_untouched = 0;
    int r_keep = block_exclusive_scan(n_untouched, &tot_untouched, s_scan);   // every ent[] read
    int n_t = 0;
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        const int sl = tid * nc + j;
        if (j < nc && sl < C && ((s_touch[sl >> 5] >> (sl & 31)) & 1u)) ++n_t;
    }
    int r_touch = block_exclusive_scan(n_t, nullptr, s_scan);
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        if (ent[j] >= 0 && !((s_touch[ent[j] >> 5] >> (ent[j] & 31)) & 1u)) a.lru_order[r_keep++] = ent[j];
        const int sl = tid * nc + j;
        if (j < nc && sl < C && ((s_touch[sl >> 5] >> (sl & 31)) & 1u)) {
            a.lru_order[tot_untouched + r_touch++] = sl;
            a.usage[sl] = tick;
        }
    }
    if (tid == 0) a.sc->tick = tick;
}

// Fill records of one on-demand group (or of one of its batches): pinned pool ->
// victim slots, 16-byte pieces read over the host link by every thread of the grid,
// eight in flight per thread.
__global__ void __launch_bounds__(256) pf_gather_kernel(PrefillGatherArgs a) {
    const int f0 = a.sub_fill ? a.sub_fill[a.sub] : 0;
    const int f1 = a.sub_fill ? a.sub_fill[a.sub + 1] : *a.n_fill;
    if (f1 <= f0) return;
    const size_t per = a.rec_bytes / 16;
    const size_t total = (size_t)(f1 - f0) * per;
    const size_t stride = (size_t)gridDim.x * blockDim.x * 8;
    for (size_t i0 = (size_t)blockIdx.x * blockDim.x * 8 + threadIdx.x; i0 < total; i0 += stride) {
        uint4 v[8];
        size_t dst[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const size_t i = i0 + (size_t)j * blockDim.x;
            if (i < total) {
                const size_t r = f0 + i / per, off = (i % per) * 16;
                v[j] = __ldcs(reinterpret_cast<const uint4*>(a.host_pool + (size_t)a.fill_flat[r] * a.rec_bytes + off));
                dst[j] = (size_t)a.fill_slot[r] * a.rec_bytes + off;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const size_t i = i0 + (size_t)j * blockDim.x;
            if (i < total) *reinterpret_cast<uint4*>(a.slot_buf + dst[j]) = v[j];
        }
    }
}

// Whole-layer stream-in: n16 16-byte pieces from the device-mapped pinned pool to
// the buffer, read over the host link by SM loads (eight in flight per thread,
// coalesced per warp), on the cache's copy stream next to the compute stream's
// GEMMs.  SM loads reach the link's rate whichever copy engine a stream is given.
// A quarter of the SMs (one CTA each, about 1.2 MB in flight) keep the link busy;
// two CTAs on every SM kept it busy too but slowed the GEMMs beside them 2.5-fold.
__global__ void __launch_bounds__(256) pf_stream_kernel(const uint4* __restrict__ src,
                                                        uint4* __restrict__ dst, size_t n16) {
    const size_t stride = (size_t)gridDim.x * blockDim.x * 8;
    for (size_t i0 = (size_t)blockIdx.x * blockDim.x * 8 + threadIdx.x; i0 < n16; i0 += stride) {
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const size_t i = i0 + (size_t)j * blockDim.x;
            if (i < n16) v[j] = __ldcs(src + i);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const size_t i = i0 + (size_t)j * blockDim.x;
            if (i < n16) dst[i] = v[j];
        }
    }
}

// ------------------------------------------------------------------ route sort
// Chunks of 32 tokens.  Count of routes per (chunk, expert); a route with an id
// outside [0, E) or repeating an id of its own token is masked (status bit).
__global__ void pf_count_kernel(PrefillArgs a) {
    extern __shared__ uint32_t s_cnt[];            // [E]
    const int c = blockIdx.x, E = a.E, k = a.k;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    const int t0 = c * 32, t1 = min(a.T, t0 + 32);
    int bad = 0;
    for (int i = threadIdx.x; i < (t1 - t0) * k; i += blockDim.x) {
        const int r = t0 * k + i;
        const int e = a.ids[r];
        bool ok = e >= 0 && e < E;
        for (int j = 0; ok && j < i % k; ++j) ok = a.ids[r - 1 - j] != e;   // earlier in the row
        if (ok) atomicAdd(&s_cnt[e], 1u);
        else bad = 1;
    }
    if (bad) atomicOr(&a.sc->status, FT_DEV_BAD_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) a.chunk_cnt[(size_t)c * E + e] = s_cnt[e];
}

// One CTA of 1024 threads: chunk prefixes per expert (in place), expert offsets,
// m-tile prefix (128-row tiles per expert).
__global__ void __launch_bounds__(1024, 1) pf_scan_kernel(PrefillArgs a) {
    __shared__ int s_scan[33];
    const int E = a.E, n_chunks = (a.T + 31) / 32;
    const int ne = (E + 1023) / 1024;
    int tot[kExpertsPerThread], tiles[kExpertsPerThread];
    int my_tot = 0, my_tiles = 0;
#pragma unroll
    for (int j = 0; j < kExpertsPerThread; ++j) {
        tot[j] = 0;
        tiles[j] = 0;
        const int e = threadIdx.x * ne + j;
        if (j < ne && e < E) {
            int run = 0;
            for (int c0 = 0; c0 < n_chunks; c0 += 16) {   // 16 loads in flight, then the prefixes
                int v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = c0 + i < n_chunks ? a.chunk_cnt[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (c0 + i < n_chunks) a.chunk_cnt[(size_t)(c0 + i) * E + e] = run;
                    run += v[i];
                }
            }
            tot[j] = run;
            tiles[j] = (run + 127) / 128;
        }
        my_tot += tot[j];
        my_tiles += tiles[j];
    }
    int all_routes = 0, all_tiles = 0;
    int off = block_exclusive_scan(my_tot, &all_routes, s_scan);
    int toff = block_exclusive_scan(my_tiles, &all_tiles, s_scan);
#pragma unroll
    for (int j = 0; j < kExpertsPerThread; ++j) {
        const int e = threadIdx.x * ne + j;
        if (j < ne && e < E) {
            a.offsets[e] = off;
            a.mtile_prefix[e] = toff;
            off += tot[j];
            toff += tiles[j];
        }
    }
    if (threadIdx.x == 0) {
        a.offsets[E] = all_routes;
        a.mtile_prefix[E] = all_tiles;
    }
}

// CTA per chunk of 32 tokens: each valid route gets its stable position (routes of
// one expert in token order) and the quantised x row of its token.
__global__ void pf_scatter_quant_kernel(PrefillArgs a) {
    extern __shared__ uint32_t s_mask[];           // [E] token bitmask of this chunk
    const int c = blockIdx.x, E = a.E, k = a.k, H = a.H;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_mask[e] = 0;
    __syncthreads();
    const int t0 = c * 32, t1 = min(a.T, t0 + 32);
    for (int i = threadIdx.x; i < (t1 - t0) * k; i += blockDim.x) {
        const int r = t0 * k + i, e = a.ids[r];
        bool ok = e >= 0 && e < E;
        for (int j = 0; ok && j < i % k; ++j) ok = a.ids[r - 1 - j] != e;
        if (ok) atomicOr(&s_mask[e], 1u << (i / k));
    }
    __syncthreads();
    // positions
    for (int i = threadIdx.x; i < (t1 - t0) * k; i += blockDim.x) {
        const int r = t0 * k + i, e = a.ids[r];
        bool ok = e >= 0 && e < E;
        for (int j = 0; ok && j < i % k; ++j) ok = a.ids[r - 1 - j] != e;
        int pos = -1;
        if (ok) {
            const int tl = i / k;
            pos = a.offsets[e] + a.chunk_cnt[(size_t)c * E + e] + __popc(s_mask[e] & ((1u << tl) - 1u));
            a.perm[pos] = r;
        }
        a.route_pos[r] = pos;
    }
    __syncthreads();
    // quantise each token row once, write it to every route position of the token
    const int nblk = H / 16;
    for (int i = threadIdx.x; i < (t1 - t0) * nblk; i += blockDim.x) {
        const int tl = i / nblk, blk = i % nblk, t = t0 + tl;
        const __nv_bfloat16* xp = a.x + (size_t)t * H + blk * 16;
        float v[16];
        const uint4 q0 = *reinterpret_cast<const uint4*>(xp);
        const uint4 q1 = *reinterpret_cast<const uint4*>(xp + 8);
        const __nv_bfloat162* b0 = reinterpret_cast<const __nv_bfloat162*>(&q0);
        const __nv_bfloat162* b1 = reinterpret_cast<const __nv_bfloat162*>(&q1);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f0 = __bfloat1622float2(b0[j]), f1 = __bfloat1622float2(b1[j]);
            v[2 * j] = f0.x; v[2 * j + 1] = f0.y; v[8 + 2 * j] = f1.x; v[8 + 2 * j + 1] = f1.y;
        }
        uint32_t lo, hi;
        const uint8_t sc = quant_block16(v, lo, hi);
        for (int j = 0; j < k; ++j) {
            const int pos = a.route_pos[(size_t)t * k + j];
            if (pos < 0) continue;
            *reinterpret_cast<uint2*>(a.a_codes + (size_t)pos * (H / 2) + blk * 8) = make_uint2(lo, hi);
            a.a_scales[(size_t)pos * nblk + blk] = sc;
        }
    }
}

// y[t] = sum_j O[t*k + j] over the token's valid routes, in order j.
__global__ void pf_combine_kernel(PrefillArgs a) {
    const int H4 = a.H / 4;
    const size_t n = (size_t)a.T * H4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / H4), c = (int)(i % H4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < a.k; ++j) {
            const size_t r = (size_t)t * a.k + j;
            if (a.route_pos[r] < 0) continue;
            const float4 o = reinterpret_cast<const float4*>(a.O + r * a.H)[c];
            acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
        }
        reinterpret_cast<float4*>(a.y + (size_t)t * a.H)[c] = acc;
    }
}

cudaError_t launch_pf_tables(const PrefillTablesArgs& a, cudaStream_t s) {
    pf_tables_kernel<<<1, 1024, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_pf_stream(const void* src, void* dst, size_t bytes, cudaStream_t s) {
    pf_stream_kernel<<<(sm_count() + 3) / 4, 256, 0, s>>>(static_cast<const uint4*>(src),
                                                      static_cast<uint4*>(dst), bytes / 16);
    return cudaGetLastError();
}

cudaError_t launch_pf_demand_tables(const PrefillDemandArgs& a, cudaStream_t s) {
    pf_demand_tables_kernel<<<1, 1024, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_pf_gather(const PrefillGatherArgs& a, bool narrow, cudaStream_t s) {
    const int half = sm_count() / 2;
    pf_gather_kernel<<<narrow ? (half > 0 ? half : 1) : sm_count() * 4, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_pf_sort_quant(const PrefillArgs& a, cudaStream_t s) {
    const int n_chunks = (a.T + 31) / 32;
    const size_t sm = (size_t)a.E * 4;
    pf_count_kernel<<<n_chunks, 256, sm, s>>>(a);
    pf_scan_kernel<<<1, 1024, 0, s>>>(a);
    pf_scatter_quant_kernel<<<n_chunks, 256, sm, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_pf_combine(const PrefillArgs& a, cudaStream_t s) {
    const size_t n = (size_t)a.T * (a.H / 4);
    size_t grid = (n + 255) / 256;
    if (grid > (size_t)sm_count() * 8) grid = (size_t)sm_count() * 8;
    pf_combine_kernel<<<(unsigned)grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ft
