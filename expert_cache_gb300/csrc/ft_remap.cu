// Route -> slot remap of one decode layer call: dedupe, hit/miss partition, the
// Q16 miss split, LRU victim choice, table update, and the per-call work lists.
//
// [EXPLAINER §6.1] H / M / m over the deduplicated routes of the batch;
// [EXPLAINER §6.7] at most q victims from the global LRU take the chosen misses;
// [EXPLAINER §8.2] control flow as data: fixed-size arrays and device-side counts,
//   one pass over the LRU order yields the candidates and the first q are used;
// [BWRATIO "代码全链路" §3] Q16 integer split; phase 3 rewrites ids to slot / -1;
// [JUHE "生成阶段"] slot_for_id / id_of_slot / usage tables.
//
// One CTA of 1024 threads.  The LRU order is kept as a device permutation
// `lru_order` of the slots sorted by (usage, slot), free slots (usage -1) first;
// a call keeps the untouched slots in order (minus the q victims at the front)
// and appends the touched ones (hits and victims) in ascending slot order.
//
// Latency: the only dependent global loads are ids -> slot_for_id and
// lru_order -> id_of_slot (for the first B*k+1 LRU positions, where every victim
// lies); both chains are issued at the start.  Residency found in step 2 is kept in
// shared memory and updated there, so later steps never re-read the tables.
#include "ft_internal.cuh"

namespace ft {

__global__ void init_tables_kernel(int32_t* slot_for_id, int n_ids, int32_t* id_of_slot,
                                   long long* usage, int32_t* lru_order, int C,
                                   DevScalars* sc, int reset_tick) {
    const int stride = gridDim.x * blockDim.x;
    const int t0 = blockIdx.x * blockDim.x + threadIdx.x;
    for (int i = t0; i < n_ids; i += stride) slot_for_id[i] = -1;
    for (int i = t0; i < C; i += stride) {
        id_of_slot[i] = -1;
        usage[i] = -1;
        lru_order[i] = i;
    }
    if (t0 == 0) {
        if (reset_tick) {
            sc->tick = 0;
            sc->status = 0;
        }
        sc->n_units = 0;
        sc->n_fill = 0;
        sc->n_pairs = 0;
    }
}

cudaError_t launch_init_tables(int32_t* slot_for_id, int n_ids, int32_t* id_of_slot,
                               long long* usage, int32_t* lru_order, int C,
                               DevScalars* sc, bool reset_tick, cudaStream_t s) {
    int n = n_ids > C ? n_ids : C;
    int grid = (n + 255) / 256;
    if (grid > 1024) grid = 1024;
    if (grid < 1) grid = 1;
    init_tables_kernel<<<grid, 256, 0, s>>>(slot_for_id, n_ids, id_of_slot, usage,
                                            lru_order, C, sc, reset_tick ? 1 : 0);
    return cudaGetLastError();
}

__device__ __forceinline__ int q_rule_dev(int m, unsigned f) {
    if (m <= 0) return 0;
    const long long F = f;
    const long long lo = ((long long)m * F) >> 16;
    const long long c_lo = max(lo * (65536 - F), (m - lo) * F);
    const long long c_hi = max((lo + 1) * (65536 - F), (m - lo - 1) * F);
    long long fetch = c_lo <= c_hi ? lo : lo + 1;
    if (fetch < 1) fetch = 1;
    return (int)(fetch < m ? fetch : m);
}

// Exclusive prefix of popcounts over `nw` bitmap words, computed by one warp;
// writes prefix[0..nw] (prefix[nw] = total).
__device__ __forceinline__ void warp_word_prefix(const uint32_t* words, int* prefix, int nw, int lane) {
    int carry = 0;
    for (int base = 0; base < nw; base += 32) {
        const int i = base + lane;
        const int c = i < nw ? __popc(words[i]) : 0;
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (i < nw) prefix[i] = carry + incl - c;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[nw] = carry;
}

__device__ __forceinline__ int bit_rank(const uint32_t* words, const int* prefix, int i) {
    return prefix[i >> 5] + __popc(words[i >> 5] & ((1u << (i & 31)) - 1u));
}

__device__ __forceinline__ bool bit_test(const uint32_t* words, int i) {
    return (words[i >> 5] >> (i & 31)) & 1u;
}

constexpr int kPrefetchPos = kMaxRoutes + 1;   // LRU positions whose old ids are prefetched

__global__ void __launch_bounds__(kThreadsRemap, 1) remap_kernel(DecodeArgs a) {
    __shared__ uint32_t s_hitw[kMaxE / 32], s_missw[kMaxE / 32];
    __shared__ int s_hpre[kMaxE / 32 + 1], s_mpre[kMaxE / 32 + 1];
    __shared__ uint32_t s_touched[kMaxC / 32];
    __shared__ int s_tpre[kMaxC / 32 + 1];
    extern __shared__ int32_t s_dyn[];
    int32_t* s_slot = s_dyn;                     // [E] residency of present experts (after the update)
    int16_t* s_u = reinterpret_cast<int16_t*>(s_dyn + a.E);   // [E] GPU unit, -1 deferred
    __shared__ int32_t s_miss[kMaxRoutes + 1];
    __shared__ int32_t s_hit[kMaxRoutes + 1];
    __shared__ int32_t s_victim[kMaxRoutes + 1];
    __shared__ int32_t s_vold[kMaxRoutes + 1];
    __shared__ uint32_t s_tokmask[kMaxRoutes + 2];
    __shared__ int32_t s_pair0[kMaxRoutes + 2];
    __shared__ int s_scan[33];
    __shared__ int s_q, s_ndef;

    pdl_wait_and_release();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E, C = a.C, R = a.B * a.k, layer = a.layer;
    const int base_id = layer * E;
    const int nwE = (E + 31) / 32, nwC = (C + 31) / 32;

    // ---- 0. independent loads first: tick, route ids, LRU order, old ids of its head
    long long tick = 0;
    if (tid == 0) tick = a.sc->tick + 1;
    const int my_id = tid < R ? a.ids[tid] : -1;          // R <= 1023 < blockDim
    const int nc = (C + kThreadsRemap - 1) / kThreadsRemap;
    int lru_loc[kSlotsPerThread];
    int old_loc[kSlotsPerThread];
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        const int pos = tid * nc + j;
        lru_loc[j] = (j < nc && pos < C) ? a.lru_order[pos] : -1;
    }
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        const int pos = tid * nc + j;
        old_loc[j] = (lru_loc[j] >= 0 && pos < kPrefetchPos && pos <= R) ? a.id_of_slot[lru_loc[j]] : -1;
    }
    for (int i = tid; i < nwE; i += kThreadsRemap) { s_hitw[i] = 0; s_missw[i] = 0; }
    for (int i = tid; i < nwC; i += kThreadsRemap) s_touched[i] = 0;
    for (int e = tid; e < E; e += kThreadsRemap) { s_slot[e] = -2; s_u[e] = -1; }
    if (tid == 0) s_ndef = 0;
    __syncthreads();

    // ---- 1. dedupe: each present expert looks up its slot once
    const bool my_valid = tid < R && my_id >= 0 && my_id < E;
    if (tid < R && !my_valid) atomicOr(&a.sc->status, FT_DEV_BAD_ID);
    if (my_valid && atomicCAS(&s_slot[my_id], -2, -3) == -2) {   // first route of this expert
        const int s = a.slot_for_id[base_id + my_id];
        s_slot[my_id] = s;
        if (s >= 0) {
            atomicOr(&s_hitw[my_id >> 5], 1u << (my_id & 31));
            atomicOr(&s_touched[s >> 5], 1u << (s & 31));
        } else {
            atomicOr(&s_missw[my_id >> 5], 1u << (my_id & 31));
        }
    }
    __syncthreads();

    // ---- 2. ranks of hits and misses in ascending expert id; q
    if (warp == 0) warp_word_prefix(s_hitw, s_hpre, nwE, lane);
    if (warp == 1) warp_word_prefix(s_missw, s_mpre, nwE, lane);
    __syncthreads();
    const int n_hit = s_hpre[nwE], m = s_mpre[nwE];
    if (tid == 0) {
        int q = a.split_mode == FT_SPLIT_FULL_OFFLOAD ? m : q_rule_dev(m, a.f_q16);
        if (q > C - n_hit) q = C - n_hit;
        s_q = q < 0 ? 0 : q;
    }
    for (int e = tid; e < E; e += kThreadsRemap) {
        if (bit_test(s_hitw, e)) s_hit[bit_rank(s_hitw, s_hpre, e)] = e;
        else if (bit_test(s_missw, e)) s_miss[bit_rank(s_missw, s_mpre, e)] = e;
    }
    // ---- 3. victims: the first q untouched entries of the LRU order
    unsigned untouched = 0;
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        if (lru_loc[j] >= 0 && !bit_test(s_touched, lru_loc[j])) { untouched |= 1u << j; ++cnt; }
    }
    const int ut_rank0 = block_exclusive_scan(cnt, nullptr, s_scan);   // syncs: s_q visible
    const int q = s_q;
    {
        int r = ut_rank0;
#pragma unroll
        for (int j = 0; j < kSlotsPerThread; ++j) {
            if (untouched >> j & 1u) {
                if (r < q) {
                    s_victim[r] = lru_loc[j];
                    const int pos = tid * nc + j;
                    s_vold[r] = (pos < kPrefetchPos && pos <= R) ? old_loc[j] : a.id_of_slot[lru_loc[j]];
                }
                ++r;
            }
        }
    }
    __syncthreads();

    // ---- 4. fills: victim i takes miss i (ascending flat id); evicted ids unmapped
    for (int i = tid; i < q; i += kThreadsRemap) {
        const int e = s_miss[i];
        const int v = s_victim[i];
        const int old = s_vold[i];
        if (old >= 0) a.slot_for_id[old] = -1;
        a.slot_for_id[base_id + e] = v;
        a.id_of_slot[v] = base_id + e;
        s_slot[e] = v;
        s_u[e] = (int16_t)i;
        atomicOr(&s_touched[v >> 5], 1u << (v & 31));
    }
    for (int i = tid; i < n_hit; i += kThreadsRemap) s_u[s_hit[i]] = (int16_t)(q + i);
    const int n_routed = q + n_hit;
    const bool has_shared = a.shared != nullptr;
    const int n_units = n_routed + (has_shared ? 1 : 0);
    const uint32_t all_tok = a.B >= 32 ? 0xffffffffu : ((1u << a.B) - 1u);
    for (int u = tid; u < n_units; u += kThreadsRemap) s_tokmask[u] = u < n_routed ? 0u : all_tok;
    __syncthreads();

    // ---- 5. LRU order: untouched non-victims keep their order, then the touched slots
    //         ascending, stamped with this call's tick; route rewrite; token masks
    {
        int r = ut_rank0;
#pragma unroll
        for (int j = 0; j < kSlotsPerThread; ++j) {
            if (untouched >> j & 1u) {
                if (r >= q) a.lru_order[r - q] = lru_loc[j];
                ++r;
            }
        }
    }
    if (warp == 0) warp_word_prefix(s_touched, s_tpre, nwC, lane);
    if (my_valid) {
        const int s = s_slot[my_id];
        const int b = tid / a.k;
        if (s >= 0) atomicOr(&s_tokmask[s_u[my_id]], 1u << b);
        else atomicAdd(&s_ndef, 1);
        a.deferred[tid] = s >= 0 ? -1 : base_id + my_id;
        if (a.route_slot) a.route_slot[tid] = s;
    } else if (tid < R) {
        a.deferred[tid] = -1;
        if (a.route_slot) a.route_slot[tid] = -1;
    }
    if (tid == 0) a.sc->tick = tick;
    __shared__ long long s_tick;
    if (tid == 0) s_tick = tick;
    __syncthreads();
    {
        const int T = n_hit + q;
        const long long tk = s_tick;
        for (int w = tid; w < nwC; w += kThreadsRemap) {
            uint32_t bits = s_touched[w];
            int rank = s_tpre[w];
            while (bits) {
                const int s = w * 32 + __ffs(bits) - 1;
                a.lru_order[C - T + rank] = s;
                a.usage[s] = tk;
                ++rank;
                bits &= bits - 1;
            }
        }
    }

    // ---- 6. (unit, token) pairs
    const int ntok = tid < n_units ? __popc(s_tokmask[tid]) : 0;
    int n_pairs = 0;
    const int p0 = block_exclusive_scan(ntok, &n_pairs, s_scan);
    if (tid < n_units) {
        const int u = tid;
        s_pair0[u] = p0;
        Unit un;
        if (u < q) {
            const int f = base_id + s_miss[u];
            un.src = a.host_pool + (size_t)f * a.rec_bytes;
            un.dst = a.slot_buf + (size_t)s_victim[u] * a.rec_bytes;
        } else if (u < n_routed) {
            un.src = a.slot_buf + (size_t)s_slot[s_hit[u - q]] * a.rec_bytes;
            un.dst = nullptr;
        } else {
            un.src = a.shared + (size_t)layer * a.rec_bytes;
            un.dst = nullptr;
        }
        un.pair0 = p0;
        un.n_tok = ntok;
        a.units[u] = un;
        uint32_t msk = s_tokmask[u];
        int p = p0;
        while (msk) {
            const int b = __ffs(msk) - 1;
            a.pair_tok[p++] = b;
            msk &= msk - 1;
        }
    }
    __syncthreads();
    if (tid < R) {
        int pr = -1;
        if (my_valid) {
            const int u = s_u[my_id];
            if (u >= 0) {
                const int b = tid / a.k;
                pr = s_pair0[u] + __popc(s_tokmask[u] & ((1u << b) - 1u));
            }
        }
        a.route_pair[tid] = pr;
    }
    const int tiles2 = a.H / kDownRowsPerItem;
    for (int i = tid; i < tiles2; i += kThreadsRemap) a.tile_done[i] = 0;
    if (tid == 0) {
        DevScalars* sc = a.sc;
        const int def_total = s_ndef;
        sc->n_units = n_units;
        sc->n_fill = q;
        sc->n_hit = n_hit;
        sc->n_pairs = n_pairs;
        sc->shared_pair0 = has_shared ? s_pair0[n_routed] : -1;
        sc->work1 = 0;
        sc->work2 = 0;
        sc->counters[0] = n_hit;
        sc->counters[1] = m;
        sc->counters[2] = q;
        sc->counters[3] = def_total;
        if (a.counters) {
            a.counters[0] = n_hit;
            a.counters[1] = m;
            a.counters[2] = q;
            a.counters[3] = def_total;
        }
    }
}

size_t remap_smem(int E) { return (size_t)E * 6 + 16; }

cudaError_t launch_remap(const DecodeArgs& a, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(remap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)remap_smem(kMaxE));
        attr = true;
    }
    return launch_pdl(remap_kernel, dim3(1), dim3(kThreadsRemap), remap_smem(a.E), s, a);
}

}  // namespace ft
