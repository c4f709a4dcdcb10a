// ft_moe_decode_static: the decode layer call with its per-call scratch in a
// file-scope device array instead of the caller's workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they set up or run decode -- code running under a framework that owns every
// device allocation through its own pool and forbids raw cudaMalloc, or a serving
// loop that must never enter the CUDA allocator (an allocation can synchronise the
// device and stall the token pipeline).  Such a caller still owns the cache (its
// tables live in the workspace given to ft_cache_create) and passes inputs and
// outputs; only the per-call scratch (the h activations, the per-tile
// flags and the grid state of the decode kernel) comes from the static array below.
//
// The array is a module-scope __device__ object: every GPU that loads this
// library holds kStaticScratchBytes of it until the process exits.  In host code
// its name is only a host-side stand-in, so the device address is looked up once
// per device with cudaGetSymbolAddress, on the first call made on that device
// (make that first call before any stream capture).  All calls share the array
// and it keeps the last call's contents: the decode kernel's grid state (a call
// epoch shared by every cache that uses the array, and a counter that each call
// returns to zero) starts zero-initialised when the module loads, and the h words
// and the flags carry the epoch of the call that wrote them, so stale words are
// never taken for fresh ones.  Calls that overlap on the GPU (two streams, two caches)
// race on the array and must be serialised by the caller.
#include <cstdio>
#include <mutex>

#include "ft_internal.cuh"

namespace ft {

constexpr size_t kStaticScratchBytes = (size_t)8 << 20;   // 8 MiB

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
    NvtxRange range("ft_moe_decode_static");
    if (!c) return FT_ERR_ARG;
    auto fail = [&](ft_status s, const char* m) { snprintf(c->err, sizeof(c->err), "%s", m); return s; };
    if (layer < 0 || layer >= c->d.L) return fail(FT_ERR_ARG, "layer out of range");
    if (B < 1 || B > c->d.B_max) return fail(FT_ERR_ARG, "B outside [1, B_max]");
    if (k < 1 || k > c->d.k_max) return fail(FT_ERR_ARG, "k outside [1, k_max]");
    if (!x || !topk_ids || !topk_w || !y || !deferred) return fail(FT_ERR_ARG, "NULL argument");
    if (((uintptr_t)x) % 16) return fail(FT_ERR_ARG, "x must be 16-byte aligned");

    // per-call scratch carve-up: grid state first (same place for every cache
    // shape), then the tagged h words and flags
    const size_t P = (size_t)B * k + B;
    size_t off = 0;
    const size_t o_sync = off;   off = up256(off + kSyncWords * 4);
    const size_t o_h = off;      off = up256(off + P * (size_t)c->d.I * 8);
    const size_t o_yf = off;     off = up256(off + (size_t)(c->d.H / decode_rows(c->d.I)) * 8);
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

    DecodeArgs a = decode_args(c, layer, x, topk_ids, topk_w, B, k, y, deferred, route_slot,
                               counters);
    a.h = reinterpret_cast<unsigned long long*>(scr + o_h);
    a.sync = reinterpret_cast<unsigned*>(scr + o_sync);
    a.yflag = reinterpret_cast<unsigned long long*>(scr + o_yf);
    a.scrub = reinterpret_cast<unsigned long long*>(scr + o_h);
    a.scrub_words = (kStaticScratchBytes - o_h) / 8;
    const int p = prof_begin(c, 0, s);
    cudaError_t e = launch_decode(a, c->grid_decode, s);
    prof_end(c, p, s);
    if (e == cudaSuccess && c->host)
        e = launch_host_join(c->mb_dev, (unsigned)c->ml.y, y, B * c->d.H, &a.sc->counters[3], &a.sc->status, s);
    if (e != cudaSuccess) {
        snprintf(c->err, sizeof(c->err), "static decode launch: %s", cudaGetErrorString(e));
        return FT_ERR_CUDA;
    }
    return FT_OK;
}
