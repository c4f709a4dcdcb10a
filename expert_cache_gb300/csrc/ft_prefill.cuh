// Internal declarations of the prefill path.
#pragma once
#include "ft_internal.cuh"

namespace ft {

struct PrefillTablesArgs {
    int32_t* slot_for_id;
    int32_t* id_of_slot;
    long long* usage;
    int32_t* lru_order;
    DevScalars* sc;
    int C, E;
    int la, ba;            // layer loaded into buffer ba
    int lb, bb;            // layer prefetched into buffer bb (lb < 0: none)
};

struct PrefillArgs {
    DevScalars* sc;
    int T, k, E, H, I;
    const __nv_bfloat16* x;     // [T, H]
    const int32_t* ids;         // [T, k]
    const float* w;             // [T, k]
    float* y;                   // [T, H]
    int32_t* chunk_cnt;         // [ceil(T/32), E]
    int32_t* offsets;           // [E + 1] first sorted row of each expert
    int32_t* mtile_prefix;      // [E + 1] 128-row tiles before each expert
    int32_t* perm;              // [T*k] sorted row -> route
    int32_t* route_pos;         // [T*k] route -> sorted row (-1: masked)
    uint8_t* a_codes;           // [T*k, H/2]  quantised x, sorted rows
    uint8_t* a_scales;          // [T*k, H/16]
    uint8_t* h_codes;           // [T*k, I/2]  quantised h, sorted rows
    uint8_t* h_scales;          // [T*k, I/16]
    float* O;                   // [T*k, H]    gated expert outputs, route rows
    uint8_t* debug_h;           // optional: [T*k, I/2] codes then [T*k, I/16] scales, route rows
};

// On-demand prefill, one group of the layer's routed union (experts with at least
// one route, ascending) of at most C experts: group g holds union ranks
// [g*C, g*C + C).  The tables are updated like a decode call that fills every miss.
struct PrefillDemandArgs {
    int32_t* slot_for_id;
    int32_t* id_of_slot;
    long long* usage;
    int32_t* lru_order;
    DevScalars* sc;
    int C, E, layer, group;
    const int32_t* offsets;     // [E + 1] sorted-row offsets (from the route sort)
    int32_t* slot_of;           // [E] out: slot of each expert of the group, else -1
    int32_t* mtile;             // [E + 1] out: 128-row tile prefix over the group's experts
    int32_t* fill_flat;         // [E] out: flat id of fill i (ascending)
    int32_t* fill_slot;         // [E] out: victim slot of fill i
    int32_t* n_fill;            // out: number of fills
    // out: the group in kOdSub batches by expert id, each starting at a fill: batch j
    // holds fills [sub_fill[j], sub_fill[j+1]) and 128-row tiles [sub_tile[j], sub_tile[j+1])
    int32_t* sub_fill;          // [kOdSub + 1]
    int32_t* sub_tile;          // [kOdSub + 1]
};

struct PrefillGatherArgs {
    const uint8_t* host_pool;   // device-mapped pinned pool
    uint8_t* slot_buf;
    size_t rec_bytes;
    const int32_t* fill_flat;
    const int32_t* fill_slot;
    const int32_t* n_fill;
    const int32_t* sub_fill;    // when not null: fills [sub_fill[sub], sub_fill[sub + 1]) only
    int sub;
};

cudaError_t launch_pf_tables(const PrefillTablesArgs& a, cudaStream_t s);
// bytes (a multiple of 16, both ends 16-byte aligned) from src (device-mapped pinned
// host memory) to dst (device).
cudaError_t launch_pf_stream(const void* src, void* dst, size_t bytes, cudaStream_t s);
cudaError_t launch_pf_demand_tables(const PrefillDemandArgs& a, cudaStream_t s);
// narrow: half of the SMs (one CTA each), beside the GEMMs of the previous batch
cudaError_t launch_pf_gather(const PrefillGatherArgs& a, bool narrow, cudaStream_t s);
cudaError_t launch_pf_sort_quant(const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_pf_combine(const PrefillArgs& a, cudaStream_t s);

}  // namespace ft
