// Internal declarations of the tcgen05 FP4 grouped GEMM used by prefill.
#pragma once
#include <cuda.h>
#include "ft_internal.cuh"

namespace ft {

struct UmmaArgs {
    int kind;                   // 1: gate/up + SwiGLU + h quantisation; 2: down + gate
    int E, K;                   // experts, reduction length in elements (multiple of 256)
    int n_tiles_n;              // 256-column tiles per expert
    int R_max, R_total;         // rows of the sorted buffers, valid routes T*k
    int I, H;
    int slot0;                  // slot of expert 0 of the layer (buffer base) ...
    const int32_t* slot_of;     // ... or, when not null, the slot of each expert
    const uint8_t* slot_buf;
    size_t rec_bytes;
    size_t off_b_scales;        // record offset of the B scales (W_gu or W_d)
    int mx;                     // 1: B scales are E8M0 per 32 (MXFP4 records)
    size_t off_tscale;          // record offset of the B tensor scale
    const uint8_t* a_scales;    // [R_max, K/16]
    const int32_t* offsets;     // [E + 1]
    const int32_t* mtile_prefix;// [E + 1]
    const int32_t* mrange;      // when not null: only m-tiles [mrange[0], mrange[1])
    const int32_t* perm;        // sorted row -> route
    const float* w;             // gates by route
    uint8_t* h_codes;           // kind 1 outputs (sorted rows)
    uint8_t* h_scales;
    uint8_t* debug_h;           // kind 1: optional route-order copy of h
    float* O;                   // kind 2 output (route rows)
    int* status;
};

bool make_map_2d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows);
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
                 uint64_t rec_bytes, uint32_t box_rows);
size_t umma_smem_bytes();
cudaError_t launch_umma(const CUtensorMap& a, const CUtensorMap& b, const UmmaArgs& g, int grid,
                        cudaStream_t s);

}  // namespace ft
