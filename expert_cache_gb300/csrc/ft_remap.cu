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

__global__ void __launch_bounds__(kThreadsRemap, 1) remap_kernel(DecodeArgs a) {
    __shared__ uint32_t s_present[kMaxE / 32];
    __shared__ uint32_t s_touched[kMaxC / 32];
    __shared__ int32_t s_u_of_e[kMaxE];
    __shared__ int32_t s_miss[kMaxRoutes + 1];
    __shared__ int32_t s_hit[kMaxRoutes + 1];
    __shared__ int32_t s_victim[kMaxRoutes + 1];
    __shared__ uint32_t s_tokmask[kMaxRoutes + 2];
    __shared__ int32_t s_pair0[kMaxRoutes + 2];
    __shared__ int s_scan[33];
    __shared__ int s_n_hit, s_m, s_q;
    __shared__ long long s_tick;

    const int tid = threadIdx.x;
    const int E = a.E, C = a.C, R = a.B * a.k, layer = a.layer;
    const int base_id = layer * E;

    if (tid == 0) {
        s_tick = a.sc->tick + 1;
        a.sc->tick = s_tick;
    }
    for (int i = tid; i < (E + 31) / 32; i += kThreadsRemap) s_present[i] = 0;
    for (int i = tid; i < (C + 31) / 32; i += kThreadsRemap) s_touched[i] = 0;
    for (int i = tid; i < E; i += kThreadsRemap) s_u_of_e[i] = -1;
    __syncthreads();

    // 1. routes -> present set (dedupe across the batch)
    int bad = 0;
    for (int r = tid; r < R; r += kThreadsRemap) {
        const int e = a.ids[r];
        if (e >= 0 && e < E) atomicOr(&s_present[e >> 5], 1u << (e & 31));
        else bad = 1;
    }
    if (bad) atomicOr(&a.sc->status, FT_DEV_BAD_ID);
    __syncthreads();

    // 2. hit / miss per present expert, ranks in ascending expert id
    const int ne = (E + kThreadsRemap - 1) / kThreadsRemap;
    int slot_of[kExpertsPerThread];
    unsigned kind = 0;  // 2 bits per expert: 1 hit, 2 miss
    int packed = 0;     // (hits << 16) | misses
#pragma unroll
    for (int j = 0; j < kExpertsPerThread; ++j) {
        slot_of[j] = -1;
        const int e = tid * ne + j;
        if (j < ne && e < E && (s_present[e >> 5] >> (e & 31) & 1u)) {
            const int s = a.slot_for_id[base_id + e];
            slot_of[j] = s;
            if (s >= 0) { kind |= 1u << (2 * j); packed += 1 << 16; }
            else        { kind |= 2u << (2 * j); packed += 1; }
        }
    }
    int tot = 0;
    const int rank0 = block_exclusive_scan(packed, &tot, s_scan);
    {
        int hr = rank0 >> 16, mr = rank0 & 0xFFFF;
#pragma unroll
        for (int j = 0; j < kExpertsPerThread; ++j) {
            const unsigned kj = (kind >> (2 * j)) & 3u;
            const int e = tid * ne + j;
            if (kj == 1u) {
                s_hit[hr++] = e;
                atomicOr(&s_touched[slot_of[j] >> 5], 1u << (slot_of[j] & 31));
            } else if (kj == 2u) {
                s_miss[mr++] = e;
            }
        }
    }
    if (tid == 0) {
        const int n_hit = tot >> 16, m = tot & 0xFFFF;
        int q = a.split_mode == FT_SPLIT_FULL_OFFLOAD ? m : q_rule_dev(m, a.f_q16);
        if (q > C - n_hit) q = C - n_hit;
        if (q < 0) q = 0;
        s_n_hit = n_hit; s_m = m; s_q = q;
    }
    __syncthreads();
    const int n_hit = s_n_hit, m = s_m, q = s_q;

    // 3. victims: the first q untouched entries of the LRU order
    const int nc = (C + kThreadsRemap - 1) / kThreadsRemap;
    int lru_loc[kSlotsPerThread];
    unsigned untouched = 0;
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        const int pos = tid * nc + j;
        lru_loc[j] = -1;
        if (j < nc && pos < C) {
            const int s = a.lru_order[pos];
            lru_loc[j] = s;
            if (!(s_touched[s >> 5] >> (s & 31) & 1u)) { untouched |= 1u << j; ++cnt; }
        }
    }
    const int ut_rank0 = block_exclusive_scan(cnt, nullptr, s_scan);
    {
        int r = ut_rank0;
#pragma unroll
        for (int j = 0; j < kSlotsPerThread; ++j) {
            if (untouched >> j & 1u) {
                if (r < q) s_victim[r] = lru_loc[j];
                ++r;
            }
        }
    }
    __syncthreads();

    // 4. fills: victim i takes miss i (ascending flat id); evicted ids are unmapped
    for (int i = tid; i < q; i += kThreadsRemap) {
        const int f = base_id + s_miss[i];
        const int v = s_victim[i];
        const int old = a.id_of_slot[v];
        if (old >= 0) a.slot_for_id[old] = -1;
        a.slot_for_id[f] = v;
        a.id_of_slot[v] = f;
        atomicOr(&s_touched[v >> 5], 1u << (v & 31));
    }
    __syncthreads();

    // 5. new LRU order: untouched non-victims keep their order ...
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
    // ... then every touched slot, ascending, stamped with this call's tick
    const int T = n_hit + q;
    int tcnt = 0;
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        const int s = tid * nc + j;
        if (j < nc && s < C && (s_touched[s >> 5] >> (s & 31) & 1u)) ++tcnt;
    }
    int tr = block_exclusive_scan(tcnt, nullptr, s_scan);
    const long long tick = s_tick;
#pragma unroll
    for (int j = 0; j < kSlotsPerThread; ++j) {
        const int s = tid * nc + j;
        if (j < nc && s < C && (s_touched[s >> 5] >> (s & 31) & 1u)) {
            a.lru_order[C - T + tr] = s;
            a.usage[s] = tick;
            ++tr;
        }
    }

    // 6. GPU units: fills first (link-bound work starts first), then hits, then shared
    for (int i = tid; i < q; i += kThreadsRemap) s_u_of_e[s_miss[i]] = i;
    for (int i = tid; i < n_hit; i += kThreadsRemap) s_u_of_e[s_hit[i]] = q + i;
    const int n_routed = q + n_hit;
    const bool has_shared = a.shared != nullptr;
    const int n_units = n_routed + (has_shared ? 1 : 0);
    const uint32_t all_tok = a.B >= 32 ? 0xffffffffu : ((1u << a.B) - 1u);
    for (int u = tid; u < n_units; u += kThreadsRemap) s_tokmask[u] = u < n_routed ? 0u : all_tok;
    __syncthreads();

    // 7. route rewrite: slot or -1, deferred flat id for the host share
    int n_def = 0;
    for (int r = tid; r < R; r += kThreadsRemap) {
        const int e = a.ids[r];
        int rs = -1, df = -1;
        if (e >= 0 && e < E) {
            const int f = base_id + e;
            rs = a.slot_for_id[f];
            if (rs < 0) { df = f; ++n_def; }
            else atomicOr(&s_tokmask[s_u_of_e[e]], 1u << (r / a.k));
        }
        a.deferred[r] = df;
        if (a.route_slot) a.route_slot[r] = rs;
    }
    int def_total = 0;
    block_exclusive_scan(n_def, &def_total, s_scan);   // also orders the atomics above

    // 8. (unit, token) pairs
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
            const int s = a.slot_for_id[base_id + s_hit[u - q]];
            un.src = a.slot_buf + (size_t)s * a.rec_bytes;
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
    for (int r = tid; r < R; r += kThreadsRemap) {
        const int e = a.ids[r];
        int pr = -1;
        if (e >= 0 && e < E) {
            const int u = s_u_of_e[e];
            if (u >= 0) {
                const int b = r / a.k;
                pr = s_pair0[u] + __popc(s_tokmask[u] & ((1u << b) - 1u));
            }
        }
        a.route_pair[r] = pr;
    }
    const int tiles2 = a.H / kDownRowsPerItem;
    for (int i = tid; i < tiles2; i += kThreadsRemap) a.tile_done[i] = 0;
    if (tid == 0) {
        DevScalars* sc = a.sc;
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

cudaError_t launch_remap(const DecodeArgs& a, cudaStream_t s) {
    remap_kernel<<<1, kThreadsRemap, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ft
