// Table (re)initialisation: every slot free, every id unmapped, the LRU order the
// identity (free slots in ascending slot order).  Used at creation and by resize.
// [EXPLAINER §7.2-7.3] a cold cache; a resize rebuilds at a safe point.
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
    if (t0 == 0 && reset_tick) {
        sc->tick = 0;
        sc->status = 0;
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

}  // namespace ft
