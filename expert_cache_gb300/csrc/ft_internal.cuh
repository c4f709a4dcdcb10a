// Internal declarations of the expert-cache library (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>
#include <utility>

#include <nvtx3/nvToolsExt.h>

#include "../../include/ft.h"
#include "ft_record.h"
#include "ft_host.h"

namespace ft {

// ----------------------------------------------------------------- limits
constexpr int kMaxDevices = 64;           // per-device host-side caches (attributes, SM count)
constexpr int kThreadsRemap = 1024;
constexpr int kMaxE = 4096;            // experts per layer
constexpr int kMaxC = 16384;           // slots
constexpr int kMaxRoutes = 1023;       // B_max * k_max
constexpr int kMaxB = 32;
constexpr int kMaxH = 8192;            // hidden size (decode stages 4 tokens of x in smem)
constexpr int kMaxI = 4096;            // intermediate size (4 tokens of h in smem)
constexpr int kMaxK = 32;
constexpr int kSlotsPerThread = kMaxC / kThreadsRemap;     // 16
constexpr int kExpertsPerThread = kMaxE / kThreadsRemap;   // 4

// Decode layer kernel tiling.
constexpr int kDecThreads = 256;       // 8 warps
constexpr int kTokGroup = 4;           // tokens accumulated per pass
constexpr int kOdSub = 8;              // on-demand prefill: gather / GEMM batches per group

// Work items of the decode kernel: a gate/up item holds decode_pairs(H) (gate row,
// up row) pairs and a down item decode_rows(I) output rows, each at most 32 KB of
// codes; both powers of two (so they divide I and H).
#ifdef __CUDACC__
__host__ __device__
#endif
inline int decode_pairs(int H) {
    int p = 16;
    while (p > 1 && p * H > 32768) p >>= 1;
    return p;
}
#ifdef __CUDACC__
__host__ __device__
#endif
inline int decode_rows(int I) {
    int r = 64;
    while (r > 8 && r * (I / 2) > 32768) r >>= 1;
    return r;
}

// ----------------------------------------------------------------- record
// (RecordLayout, scale_block, record_layout: ft_record.h)

// ----------------------------------------------------------------- device state
// Scalars kept in the workspace (device).
struct DevScalars {
    long long tick;        // one tick per decode / prefill layer call
    int status;            // FT_DEV_* bits
    int counters[4];       // last decode call: n_hit, m, q, deferred routes
    int pad[3];
};

// Offsets of the workspace regions (bytes, 256-aligned).
struct WsLayout {
    size_t slot_for_id, id_of_slot, usage, lru_order, scalars;
    size_t sync, h, yflag, h_end;   // decode grid state; tagged words (h_end: end)
    // prefill region (present when T_max > 0)
    size_t pf_chunk_cnt, pf_offsets, pf_mtile, pf_perm, pf_route_pos;
    size_t pf_a_codes, pf_a_scales, pf_h_codes, pf_h_scales, pf_o;
    // on-demand prefill: per-group expert -> slot, tile prefix and fill list
    size_t pf_slot_of, pf_gmtile, pf_fill_flat, pf_fill_slot, pf_nfill, pf_sub;
    size_t total;
};

WsLayout ws_layout(const ft_cache_desc& d);

// Grid state of the decode kernel (zero-initialised; see ft_decode.cu):
// [epoch: 64-bit, words 0-1][read_done][unused]
constexpr int kSyncWords = 4;

// Arguments of one decode call, passed by value to the decode kernel.
struct DecodeArgs {
    int32_t* slot_for_id;
    int32_t* id_of_slot;
    long long* usage;
    int32_t* lru_order;
    DevScalars* sc;
    unsigned long long* h; // [pairs, I] tagged values (tag << 32 | fp32 bits)
    unsigned long long* yflag;  // [H / decode_rows(I)] y row tile zeroed (tag)
    unsigned* sync;        // kSyncWords words of grid state, 8-byte aligned
    unsigned long long* scrub;  // the whole h / o region of this call's scratch ...
    size_t scrub_words;         // ... in 8-byte words (periodic tag scrub)
    const uint8_t* host_pool;   // device-mapped address of the pinned pool
    uint8_t* slot_buf;
    const uint8_t* shared;      // device, or nullptr
    size_t rec_bytes;
    size_t off_gu_scales, off_d_codes, off_d_scales, off_s_gu, off_s_d;
    int L, E, H, I, C, layer, B, k;
    int R_cap;             // B_max * k_max: sizes of the per-call arrays
    int mx;                // 1: MXFP4 records (E8M0 scale per 32), 0: NVFP4 (E4M3 per 16)
    int split_mode;
    unsigned f_q16;
    const __nv_bfloat16* x;
    const int32_t* ids;
    const float* w;
    float* y;
    int32_t* deferred;
    int32_t* route_slot;
    int32_t* counters;
    unsigned long long* trace;  // stats ring header (count), or nullptr
    unsigned trace_cap;         // records after the 16-byte header
    uint8_t* mb;                // host branch mailbox (device-mapped), or nullptr
    unsigned mb_x, mb_def, mb_w;  // its x, deferred-id and gate regions (byte offsets)
};

// Kernel launchers (each returns the launch error).
cudaError_t launch_init_tables(int32_t* slot_for_id, int n_ids, int32_t* id_of_slot,
                               long long* usage, int32_t* lru_order, int C,
                               DevScalars* sc, bool reset_tick, cudaStream_t s);
// Grid of the decode kernel for a cache shape (every CTA resident at once), and the
// launch; both take the cache's B_max * k_max as R_cap.
int decode_grid(int H, int I, int E, int R_cap);
cudaError_t check_bounded_waits(unsigned* expired);
cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t s);
// After a decode call with a host branch: when the call had host routes (*n_def > 0),
// wait (bounded) for the branch's partial and add it into y (fp32 [B, H]); sets
// FT_DEV_TIMEOUT in *status when the wait runs out.
cudaError_t launch_host_join(uint8_t* mb, unsigned mb_y, float* y, int n, const int* n_def, int* status,
                             cudaStream_t s);
cudaError_t launch_quantize(const float* w_gu, const float* w_d, int n, int H, int I,
                            uint8_t* records, size_t rec_bytes, cudaStream_t s);
cudaError_t launch_quantize_mx(const float* w_gu, const float* w_d, int n, int H, int I,
                               uint8_t* records, size_t rec_bytes, cudaStream_t s);

int sm_count();

// NVTX range around a host API call: named spans on a profiler's timeline (host side;
// nothing happens when no tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// ----------------------------------------------------------------- device helpers
#ifdef __CUDACC__

// Exclusive prefix sum over the whole block (blockDim.x a multiple of 32, <= 1024).
// All threads must call it.  `buf` is 33 ints of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* buf) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) buf[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int s = lane < nw ? buf[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += t;
        }
        buf[lane] = s;
    }
    __syncthreads();
    const int base = wid ? buf[wid - 1] : 0;
    if (total) *total = buf[nw - 1];
    __syncthreads();
    return base + incl - v;
}

// Programmatic dependent launch: wait until the previous kernel of the stream has
// completed and its writes are visible (returns at once when this kernel was not
// launched as a dependent), then allow the next kernel to be scheduled; it waits in
// turn for this one.
__device__ __forceinline__ void pdl_wait_and_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#endif  // __CUDACC__

// Launch with programmatic stream serialisation (see pdl_wait_and_release).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace ft

struct ft_cache {
    ft_cache_desc d;
    ft::RecordLayout rec;
    ft::WsLayout ws;
    int C;                          // current slot count
    const uint8_t* host_pool_dev;   // device-mapped pool address
    uint8_t* slot_buf;
    uint8_t* workspace;
    cudaStream_t copy_stream;
    cudaEvent_t copy_done[2];       // prefill buffer loaded
    cudaEvent_t compute_done[2];    // prefill buffer no longer read
    int buffer_layer[2];            // layer last streamed into each prefill buffer (-1 none)
    bool copy_pending;
    cudaEvent_t entry_ev;           // work enqueued before a prefill call
    cudaEvent_t od_ev[ft::kOdSub + 1];  // on-demand prefill: group tables done, batches gathered
    CUtensorMap map_a1, map_b1;     // GEMM1: quantised x rows; W_gu codes of the slots
    CUtensorMap map_a2, map_b2;     // GEMM2: quantised h rows; W_d codes of the slots
    bool maps_ok;
    int grid_decode;
    void* trace;                    // per-call stats ring (device) or nullptr
    int trace_cap;
    ft_host_branch* host;           // attached host branch, or nullptr
    uint8_t* mb_dev;                // its mailbox (device-mapped)
    ft::MailboxLayout ml;
    // profiling
    unsigned prof;          // bit i set: time launches of kind i
    static constexpr int kProfEvents = 65536;
    cudaEvent_t prof_ev[kProfEvents];
    int prof_kind[kProfEvents / 2];
    int prof_n;
    double prof_ms[FT_PROF_KINDS];
    long long prof_launches[FT_PROF_KINDS];
    char err[256];
};

namespace ft {
// CUDA-event timing of a launch of `kind` on stream s while profiling that kind is
// on: prof_begin returns the event pair index (or -1), prof_end closes it.
int prof_begin(ft_cache* c, int kind, cudaStream_t s);
void prof_end(ft_cache* c, int i, cudaStream_t s);
// Arguments of a decode call on cache c except the per-call scratch (h, o, sync).
DecodeArgs decode_args(ft_cache* c, int layer, const void* x, const int32_t* ids, const float* w,
                       int B, int k, float* y, int32_t* deferred, int32_t* route_slot,
                       int32_t* counters);
}  // namespace ft
