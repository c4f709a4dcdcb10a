// ft_moe_decode_static: the decode layer call with its per-call scratch in a
// file-scope device array instead of the caller's workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they set up or run decode -- code running under a framework that owns every
// device allocation through its own pool and forbids raw cudaMalloc, or a serving
// loop that must never enter the CUDA allocator (an allocation can synchronise the
// device and stall the token pipeline).  Such a caller still owns the cache (its
// tables live in the workspace given to ft_cache_create) and passes inputs and
// outputs; only the per-call scratch (GPU unit list, route/token pair maps, the h
// activations, the per-pair expert outputs and the row-tile counters) comes from
// the static array below.
//
// The array is a module-scope __device__ object: every GPU that loads this
// library holds kStaticScratchBytes of it until the process exits.  In host code
// its name is only a host-side stand-in, so the device address is looked up once
// per device with cudaGetSymbolAddress, on the first call made on that device
// (make that first call before any stream capture).  All calls share the array
// and it keeps the last call's contents: the row-tile counters that must start at
// zero are cleared by the remap kernel of every call, everything else is written
// before it is read.  Calls that overlap on the GPU (two streams, two caches) race
// on the array and must be serialised by the caller.
#include <cstdio>
#include <mutex>

#include "ft_internal.cuh"

namespace ft {

constexpr size_t kStaticScratchBytes = (size_t)8 << 20;   // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

static uint8_t* g_scratch_dev[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (nullptr on failure).
static uint8_t* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_dev[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_dev[dev] = static_cast<uint8_t*>(p);
    }
    return g_scratch_dev[dev];
}

static size_t up256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace ft

using namespace ft;

extern "C" ft_status ft_moe_decode_static(ft_cache* c, int32_t layer, const void* x,
                                          const int32_t* topk_ids, const float* topk_w,
                                          int32_t B, int32_t k, float* y, int32_t* deferred,
                                          int32_t* route_slot, int32_t* counters, void* stream) {
    if (!c) return FT_ERR_ARG;
    auto fail = [&](ft_status s, const char* m) { snprintf(c->err, sizeof(c->err), "%s", m); return s; };
    if (layer < 0 || layer >= c->d.L) return fail(FT_ERR_ARG, "layer out of range");
    if (B < 1 || B > c->d.B_max) return fail(FT_ERR_ARG, "B outside [1, B_max]");
    if (k < 1 || k > c->d.k_max) return fail(FT_ERR_ARG, "k outside [1, k_max]");
    if (!x || !topk_ids || !topk_w || !y || !deferred) return fail(FT_ERR_ARG, "NULL argument");
    if (((uintptr_t)x) % 16) return fail(FT_ERR_ARG, "x must be 16-byte aligned");

    // per-call scratch carve-up (same regions as the workspace's per-call part)
    const size_t R = (size_t)B * k, P = R + B;
    size_t off = 0;
    const size_t o_units = off;  off = up256(off + (R + 1) * sizeof(Unit));
    const size_t o_rpair = off;  off = up256(off + R * 4);
    const size_t o_ptok = off;   off = up256(off + P * 4);
    const size_t o_h = off;      off = up256(off + P * (size_t)c->d.I * 4);
    const size_t o_o = off;      off = up256(off + P * (size_t)c->d.H * 4);
    const size_t o_tile = off;   off = up256(off + (size_t)(c->d.H / kDownRowsPerItem + 1) * 4);
    if (off > kStaticScratchBytes)
        return fail(FT_ERR_ARG, "B, k, H and I need more than the 8 MiB static scratch");
    uint8_t* scr = scratch_address();
    if (!scr) return fail(FT_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (c->copy_pending) {
        cudaStreamWaitEvent(s, c->copy_done[0], 0);
        cudaStreamWaitEvent(s, c->copy_done[1], 0);
        c->copy_pending = false;
    }
    c->buffer_layer[0] = c->buffer_layer[1] = -1;

    uint8_t* ws = c->workspace;
    DecodeArgs a;
    a.slot_for_id = reinterpret_cast<int32_t*>(ws + c->ws.slot_for_id);
    a.id_of_slot = reinterpret_cast<int32_t*>(ws + c->ws.id_of_slot);
    a.usage = reinterpret_cast<long long*>(ws + c->ws.usage);
    a.lru_order = reinterpret_cast<int32_t*>(ws + c->ws.lru_order);
    a.sc = reinterpret_cast<DevScalars*>(ws + c->ws.scalars);
    a.units = reinterpret_cast<Unit*>(scr + o_units);
    a.route_pair = reinterpret_cast<int32_t*>(scr + o_rpair);
    a.pair_tok = reinterpret_cast<int32_t*>(scr + o_ptok);
    a.h = reinterpret_cast<float*>(scr + o_h);
    a.o = reinterpret_cast<float*>(scr + o_o);
    a.tile_done = reinterpret_cast<unsigned*>(scr + o_tile);
    a.host_pool = c->host_pool_dev;
    a.slot_buf = c->slot_buf;
    a.shared = static_cast<const uint8_t*>(c->d.shared_experts);
    a.rec_bytes = c->rec.bytes;
    a.off_gu_scales = c->rec.gu_scales;
    a.off_d_codes = c->rec.d_codes;
    a.off_d_scales = c->rec.d_scales;
    a.off_s_gu = c->rec.s_gu;
    a.off_s_d = c->rec.s_d;
    a.L = c->d.L; a.E = c->d.E; a.H = c->d.H; a.I = c->d.I; a.C = c->C;
    a.layer = layer; a.B = B; a.k = k;
    a.split_mode = c->d.split.mode;
    a.f_q16 = c->d.split.f_q16;
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.ids = topk_ids;
    a.w = topk_w;
    a.y = y;
    a.deferred = deferred;
    a.route_slot = route_slot;
    a.counters = counters;

    cudaError_t e = launch_remap(a, s);
    if (e == cudaSuccess) e = launch_gate_up(a, c->grid_gemv, s);
    if (e == cudaSuccess) e = launch_down(a, c->grid_gemv, s);
    if (e != cudaSuccess) {
        snprintf(c->err, sizeof(c->err), "static decode launch: %s", cudaGetErrorString(e));
        return FT_ERR_CUDA;
    }
    return FT_OK;
}
