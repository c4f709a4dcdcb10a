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

cudaError_t launch_pf_tables(const PrefillTablesArgs& a, cudaStream_t s);
cudaError_t launch_pf_sort_quant(const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_pf_combine(const PrefillArgs& a, cudaStream_t s);

}  // namespace ft
