// One routed-MoE decode layer call as ONE kernel: route -> slot decision, LRU
// victims, load-through fills, NVFP4 SwiGLU gate/up, down, the gated combine and
// the table update.
//
// [EXPLAINER §6.1] H / M / m over the deduplicated routes of the batch;
// [EXPLAINER §6.7] at most q victims from the global LRU take the chosen misses;
// [EXPLAINER §6.8] one fused expert batch: hits and fills computed together;
// [EXPLAINER §8.2] control flow as data: fixed-size arrays, device-side counts;
// [EXPLAINER §1.1] y = sum_e p_e Expert_{l,e}(x);
// [BWRATIO "代码全链路" §2-3] Q16 integer split; ids of GPU routes become slots, the
//   rest -1 (here such routes are skipped, not computed at weight 0);
// [JUHE "生成阶段"] slot_for_id / id_of_slot / usage tables;
// [JUHE "为什么可以直接相加？"] y_gpu + y_cpu is the exact layer output.
//
// Grid: G CTAs of 256 threads, all resident at once (G = SMs x occupancy).  CTAs
// 0..G-2 compute, CTA G-1 writes the tables.
//
//  1. Decision.  Every CTA reads the same table entries (ids -> slot_for_id, the
//     head of the LRU order) and derives the same decision in shared memory:
//     hits, misses, q, victims, the GPU units (fills ascending by expert id, then
//     hits ascending, then the shared expert), each unit's tokens and (unit, token)
//     pairs.  Up to 32 routes one warp decides with warp intrinsics while the
//     other warps stage x; larger batches use the whole CTA.
//  2. Gate/up items (unit, P row pairs; P * H/2 <= 16 KB per matrix) go to CTAs
//     0, 1, ... in order.  The item's rows are staged in shared memory first by bulk
//     copies issued by one thread: from HBM for hits and the shared expert, from the
//     device-mapped pinned pool over the host link for fills (one link read per
//     byte, one request per run); a fill's rows are then bulk-stored from shared
//     memory into its victim slot, which makes the fill resident.  Warp w then computes
//     pairs w, w + 8, ... in rolled loops (the per-item code stays small enough
//     for the instruction cache).  Meanwhile warps 1..7 of compute CTA z zero y's
//     R-row tile z (mod the compute CTAs) and raise the tile's flag (release).
//  3. Down items (unit, R output rows; R * I/2 <= 32 KB) go to CTAs G-2, G-3, ... so
//     the fills' down items land on CTAs without gate/up work and fetch their W_d
//     rows at once; a CTA's first down item of a hit unit is staged under its
//     gate/up work.  A CTA first acquires the flags of its down items' y tiles;
//     each item waits for its unit's h and adds w * s_d W_d h into y (fp32 adds at
//     the L2; w = the token's routing weight to that expert, 1 for the shared
//     expert).  That is the gated combine y[b] = sum_j w[b,j] o_(b,j) + shared,
//     summed in arrival order; y is complete when the grid ends.
//  4. CTA G-1 writes the per-call outputs, waits until every compute CTA has read
//     the tables, then applies the update: fills mapped, evicted ids unmapped,
//     touched slots stamped with the tick, LRU order rebuilt (untouched slots keep
//     their order, touched ones follow in ascending slot order).
//
// The LRU order is a permutation `lru_order` of the slots sorted by (usage, slot),
// free slots (usage -1) first; the q victims are the first q entries that no hit
// of this call holds, all within its first B*k positions.
//
// Exchange inside the grid: h values travel as single 64-bit words (call tag << 32
// | fp32 bits), stored and loaded with relaxed gpu-scope accesses.  A down item reads
// its unit's h words directly, re-polling any word that does not carry the call's tag
// yet (its gate/up item has not stored it); loads go out 8 at a time.  A per-item
// flag to wait on first cost a round trip more.  No fence or counter sits between those
// producers and consumers; the y tile flags (zeroed data in other words) are the one
// release / acquire pair.  The tag is the
// low half of a 64-bit call epoch kept in the scratch (never 0); every 2^31 calls
// the commit CTA zeroes the scratch words this call does not use, so no word is
// older than 2^31 calls and a stale tag can never equal the current one.  The
// only counter, read_done, is reset by the commit CTA.  Every wait is bounded:
// past one second FT_DEV_TIMEOUT is set and the CTA goes on.
//
// Arithmetic: E2M1 codes become f16 exactly (cvt.rn.f16x2.e2m1x2); x (bf16) is
// staged as f16 after an exact power-of-two prescale that keeps |x| < 2^15; code*x
// products are exact and accumulate in fp32 (fma.rn.f32.f16); each 16-element block
// partial is scaled by its E4M3 scale in fp32; the fp32 tensor scale and the
// prescale are applied at the end.  h stays fp32; the down GEMV is fp32 FMA.
#include <algorithm>
#include <mutex>

#include "ft_internal.cuh"

namespace ft {

namespace {

constexpr int kThreads = kDecThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kTok = kTokGroup;
constexpr int kMaxPerThread = 4;       // routes / head positions / units per thread
constexpr unsigned long long kWaitNs = 1000000000ull;
constexpr unsigned kWaitIters = 1u << 25;

static_assert((kMaxRoutes + 1) <= kThreads * kMaxPerThread, "routes per thread");
static_assert(kMaxB <= 32, "token masks are 32-bit");

// ------------------------------------------------------------------ memory helpers

// Expert weights stream through L2 once per call: they are read and written with
// an evict-first policy so that the tables, the exchange words and the kernel's
// own code stay resident in L2 across calls.
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint4 ldg16_l1(const void* p) {        // read-only, kept in L1
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long tagged(float v, unsigned tag) {
    return ((unsigned long long)tag << 32) | __float_as_uint(v);
}
// Release store / acquire load of a tagged word (a flag that orders other data).
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// y += v (fp32 add performed at the L2; the order of the adds to one word is free).
__device__ __forceinline__ void red_add_f32(float* p, float v) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" :: "l"(p), "f"(v) : "memory");
}
// The same for two adjacent words (p 8-byte aligned): one request.
__device__ __forceinline__ void red_add_v2_f32(float* p, float v0, float v1) {
    asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1, %2};" :: "l"(p), "f"(v0), "f"(v1) : "memory");
}

// One thread waits until *p >= target; false when the bound ran out.
__device__ __forceinline__ bool wait_geq(const unsigned* p, unsigned target) {
    if (ld_acquire(p) >= target) return true;
    const unsigned long long t0 = gtime();
    for (unsigned it = 0; it < kWaitIters; ++it) {
        __nanosleep(64);
        if (ld_acquire(p) >= target) return true;
        if ((it & 63u) == 63u && gtime() - t0 > kWaitNs) break;
    }
    return false;
}

// One thread waits until the tagged word *p carries `tag` (acquire); false when the
// bound ran out.
__device__ __forceinline__ bool wait_tag_acquire(const unsigned long long* p, unsigned tag) {
    if ((unsigned)(ld_acquire_u64(p) >> 32) == tag) return true;
    const unsigned long long t0 = gtime();
    for (unsigned it = 0; it < kWaitIters; ++it) {
        __nanosleep(64);
        if ((unsigned)(ld_acquire_u64(p) >> 32) == tag) return true;
        if ((it & 63u) == 63u && gtime() - t0 > kWaitNs) break;
    }
    return false;
}

// The N tagged words addr(0..N-1) (nullptr: no word), once each carries `tag`: every
// load of a round is in flight at once and only the stale words are reloaded
// (bounded wait).
template <int N = 8, typename AddrF>
__device__ __forceinline__ void fetch_tagged(AddrF addr, unsigned tag, float* out, int* timeout) {
    const unsigned long long ready = (unsigned long long)tag << 32;
    unsigned long long raw[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const unsigned long long* p = addr(i);
        raw[i] = p ? ld_relaxed_u64(p) : ready;
    }
    bool ok = true;
#pragma unroll
    for (int i = 0; i < N; ++i) ok &= (unsigned)(raw[i] >> 32) == tag;
    if (!ok) {
        const unsigned long long t0 = gtime();
        for (unsigned it = 0; it < kWaitIters && !ok; ++it) {
            __nanosleep(64);
#pragma unroll
            for (int i = 0; i < N; ++i)
                if ((unsigned)(raw[i] >> 32) != tag) raw[i] = ld_relaxed_u64(addr(i));
            ok = true;
#pragma unroll
            for (int i = 0; i < N; ++i) ok &= (unsigned)(raw[i] >> 32) == tag;
            if (!ok && (it & 63u) == 63u && gtime() - t0 > kWaitNs) break;
        }
        if (!ok) *timeout = 1;
    }
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __uint_as_float((unsigned)raw[i]);
}

// ------------------------------------------------------------------ arithmetic helpers

// 8 E2M1 codes (one 32-bit word, element 0 in the lowest nibble) -> 4 f16x2.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t* o) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

// Two unsigned E4M3 scale bytes (first scale in the low byte) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_float2(unsigned short v) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    __half2 hh = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(hh);
}

// acc += sum over 8 elements of code * x (f16 operands, exact products, fp32 sums).
__device__ __forceinline__ float dot8_f16(const uint32_t* c, uint4 x, float acc) {
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %5;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %0, a1, b1, %0;\n\t"
        "mov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %6;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %0, a1, b1, %0;\n\t"
        "mov.b32 {a0, a1}, %3;\n\tmov.b32 {b0, b1}, %7;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %0, a1, b1, %0;\n\t"
        "mov.b32 {a0, a1}, %4;\n\tmov.b32 {b0, b1}, %8;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc)
        : "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w));
    return acc;
}

// E8M0 scale byte -> fp32 2^(c - 127) (c = 0: the subnormal 2^-127).
__device__ __forceinline__ float e8m0_value(uint32_t c) {
    return __uint_as_float(c ? c << 23 : 0x00400000u);
}

// Scales of the two 16-element halves of 32-element chunk ch of a staged scale row:
// NVFP4 two E4M3 bytes, MXFP4 one E8M0 byte for both.
__device__ __forceinline__ float2 chunk_scales(const uint8_t* srow_p, int ch, int mx) {
    if (mx) {
        const float s = e8m0_value(srow_p[ch]);
        return make_float2(s, s);
    }
    return e4m3x2_to_float2(*reinterpret_cast<const unsigned short*>(srow_p + 2 * ch));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// f16 x staging: element e lives in 16-byte piece c = e/8; piece c is stored at
// c ^ ((c >> 3) & 3) so that the 32 lanes reading pieces 4*lane + t hit 8 distinct
// bank groups per quarter warp.
__device__ __forceinline__ int xswz(int c) { return c ^ ((c >> 3) & 3); }
// fp32 h staging: piece c = e/4 stored at c ^ ((c >> 3) & 7).
__device__ __forceinline__ int hswz(int c) { return c ^ ((c >> 3) & 7); }

// ------------------------------------------------------------------ decision helpers

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

// ------------------------------------------------------------------ async copies

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(ok) : "r"(smem_u32(b)), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait for phase `parity` of an mbarrier; false when the bound ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
    if (mbar_try(b, parity)) return true;
    const unsigned long long t0 = gtime();
    for (unsigned it = 0; it < kWaitIters; ++it) {
        if (mbar_try(b, parity)) return true;
        if ((it & 255u) == 255u && gtime() - t0 > kWaitNs) break;
    }
    return false;
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// global memory into shared memory, completing on mbarrier `b`; L2 evict-first.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
                 "[%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(b)), "l"(evict_first_policy())
                 : "memory");
}

// ------------------------------------------------------------------ shared memory

struct SmemStatic {
    uint32_t hitw[kMaxE / 32], missw[kMaxE / 32];
    int hpre[kMaxE / 32 + 1], mpre[kMaxE / 32 + 1];
    uint32_t touched[kMaxC / 32];
    int tpre[kMaxC / 32 + 1];
    int scan[33];
    float xmul[kTok];
    float uw[kMaxB];            // routing weights of the current down item's tokens
    float red[kTok][kWarps];
    // the decision's scalars
    int n_hit, m, q, n_routed, n_units, n_pairs, n_def, bad;
    int timeout;
    unsigned tag;
    unsigned long long epoch;   // this call's epoch (tag = its low half)
    long long tick;
    uint64_t bar_w, bar_d;      // completion of the staged gate/up and down weights
};

// Dynamic shared memory carve-up (byte offsets), identical on host and device.
// stage, wc and ws are contiguous: in a CTA's down items (after all of its gate/up
// items) the range holds h of up to kTok pairs.
struct DynLayout {
    unsigned stage;            // x (f16, kTok rows); later h (fp32, kTok rows)
    unsigned wc, ws;           // gate/up item: codes [2P rows][H/2], scales [2P rows][H/16]
    unsigned dc, ds;           // down item: codes [R rows][I/2], scales [R rows][I/16]
    unsigned slot, unit, ue, us, umask, upair0, rpair, runit, vold, total;
};

__host__ __device__ inline unsigned up16(unsigned x) { return (x + 15u) & ~15u; }

__host__ __device__ inline DynLayout dyn_layout(int H, int I, int E, int R_cap) {
    DynLayout d;
    unsigned off = 0;
    const unsigned P = (unsigned)decode_pairs(H), R = (unsigned)decode_rows(I);
    d.stage = off;  off = up16(off + (unsigned)kTok * H * 2);
    d.wc = off;     off = up16(off + 2 * P * (unsigned)H / 2);
    d.ws = off;     off = up16(off + 2 * P * (unsigned)H / 16);
    if (off - d.stage < (unsigned)kTok * I * 4) off = d.stage + up16((unsigned)kTok * I * 4);
    d.dc = off;     off = up16(off + R * (unsigned)I / 2);
    d.ds = off;     off = up16(off + R * (unsigned)I / 16);
    d.slot = off;   off = up16(off + (unsigned)E * 4);
    d.unit = off;   off = up16(off + (unsigned)E * 2);
    d.ue = off;     off = up16(off + (unsigned)(R_cap + 1) * 4);
    d.us = off;     off = up16(off + (unsigned)(R_cap + 1) * 4);
    d.umask = off;  off = up16(off + (unsigned)(R_cap + 1) * 4);
    d.upair0 = off; off = up16(off + (unsigned)(R_cap + 2) * 4);
    d.rpair = off;  off = up16(off + (unsigned)R_cap * 4);
    d.runit = off;  off = up16(off + (unsigned)R_cap * 4);
    d.vold = off;   off = up16(off + (unsigned)R_cap * 4);
    d.total = off;
    return d;
}

// The decision in shared memory.
struct Decision {
    int32_t* u_e;       // [units] expert id (shared: -1)
    int32_t* u_s;       // [units] slot (fills: the victim; shared: -1)
    uint32_t* u_mask;   // [units] tokens routed to the unit
    int32_t* u_pair0;   // [units + 1] first (unit, token) pair; [units] = pairs
    int32_t* r_pair;    // [R] pair of each route, -1 when not on the GPU
    int32_t* r_unit;    // [R] unit of each route, -1 host share, -2 masked id
};

// ------------------------------------------------------------------ x staging

// Stage tokens toks[0..n) of x (bf16 [B, H]) into rows 0..n-1 of xs as f16, each
// row prescaled by an exact power of two that keeps |x| < 2^15; S.xmul[t] undoes
// it.  Block-wide; every thread calls it.
__device__ void stage_x(const DecodeArgs& a, SmemStatic& S, uint4* xs, const int* toks, int n) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pieces = a.H / 8;
    float amax[kTok];
#pragma unroll
    for (int t = 0; t < kTok; ++t) amax[t] = 0.f;
    for (int p = tid; p < pieces; p += kThreads) {
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
            if (t < n) {
                const uint4 v = *reinterpret_cast<const uint4*>(a.x + (size_t)toks[t] * a.H + p * 8);
                const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __bfloat1622float2(b2[j]);
                    amax[t] = fmaxf(amax[t], fmaxf(fabsf(f.x), fabsf(f.y)));
                }
                xs[t * pieces + xswz(p)] = v;          // raw bf16 for now
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kTok; ++t) {
        float m = amax[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) S.red[t][warp] = m;
    }
    __syncthreads();
    if (tid < kTok) {
        float m = 0.f;
        for (int w = 0; w < kWarps; ++w) m = fmaxf(m, S.red[tid][w]);
        int k = 0;
        if (m >= 32768.f) k = ilogbf(m) - 14;
        S.xmul[tid] = ldexpf(1.f, k);
    }
    __syncthreads();
    for (int p = tid; p < pieces; p += kThreads) {      // each thread converts its own pieces
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
            if (t < n) {
                const float dn = 1.f / S.xmul[t];       // exact power of two
                const uint4 v = xs[t * pieces + xswz(p)];
                const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v);
                uint4 o;
                uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __bfloat1622float2(b2[j]);
                    __half2 hv = __floats2half2_rn(f.x * dn, f.y * dn);
                    ow[j] = *reinterpret_cast<uint32_t*>(&hv);
                }
                xs[t * pieces + xswz(p)] = o;
            }
        }
    }
    __syncthreads();
}

// Stage all B <= kTok tokens of x into rows 0..B-1 with warps 1..7 only (warp 0
// is deciding meanwhile): each warp loads the whole token row once, reduces its
// amax itself (no block barrier needed before the caller's next one) and converts
// the pieces j == w (mod 7) of the ones it holds.
__device__ void stage_x_warps(const DecodeArgs& a, SmemStatic& S, uint4* xs) {
    const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) - 1;   // 0..6
    const int pieces = a.H / 8;
    const int nj = (pieces + 31) / 32;
    for (int t = 0; t < a.B; ++t) {
        const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H);
        float m = 0.f;
        for (int j0 = 0; j0 < nj; j0 += 8) {           // 8 loads in flight per lane
            uint4 v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int p = (j0 + jj) * 32 + lane;
                v[jj] = (j0 + jj < nj && p < pieces) ? ldg16_l1(xr + p) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v[jj]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __bfloat1622float2(b2[q]);
                    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        int k = 0;
        if (m >= 32768.f) k = ilogbf(m) - 14;
        const float xm = ldexpf(1.f, k);
        const float dn = 1.f / xm;                       // exact power of two
        if (w == 0 && lane == 0) S.xmul[t] = xm;
        for (int j = w; j < nj; j += 7) {               // L1 holds the row by now
            const int p = j * 32 + lane;
            if (p >= pieces) continue;
            const uint4 v = ldg16_l1(xr + p);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v);
            uint4 o;
            uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __bfloat1622float2(b2[q]);
                __half2 hv = __floats2half2_rn(f.x * dn, f.y * dn);
                ow[q] = *reinterpret_cast<uint32_t*>(&hv);
            }
            xs[t * pieces + xswz(p)] = o;
        }
    }
}

// Tokens of a unit: the set bits of its mask; group g0 holds its tokens g0 .. g0+kTok-1
// (toks[t] = token of pair g0 + t, for t < the returned count).
__device__ __forceinline__ int group_tokens(uint32_t mask, int g0, int* toks) {
    const int n = min(kTok, __popc(mask) - g0);
#pragma unroll
    for (int t = 0; t < kTok; ++t) toks[t] = t < n ? (int)__fns(mask, 0, g0 + t + 1) : 0;
    return n;
}

struct UnitRef {
    const uint8_t* src;   // record to read: pinned pool (fill), slot (hit), shared
    uint8_t* dst;         // victim slot written on the way (fill), else nullptr
};

// Every item is staged the same way: thread 0 issues bulk copies (`cp.async.bulk`,
// the tensor memory accelerator) of the item's runs into shared memory, completing on
// an mbarrier the item's threads wait on.  For hits and the shared expert the source
// is HBM; for fills it is the device-mapped pinned pool, read over the host link in
// one request per run (no per-thread round trips), and once the bytes have landed
// thread 0 bulk-stores them from shared memory into the victim slot (the write-through
// that makes the fill resident).  Before a CTA restages a buffer it waits until its
// earlier bulk stores have read it; before the CTA exits, until they are complete.

// Bulk store of n bytes (a multiple of 16, both ends 16-byte aligned), shared -> global,
// in the calling thread's bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(dst), "r"(smem_u32(src)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's bulk stores have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until this thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Arms `bar` for `bytes` of bulk copies (thread 0).
__device__ __forceinline__ void arm_bulk(uint64_t* bar, uint32_t bytes) {
    if (threadIdx.x == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_tx(bar, bytes);
    }
}

// ------------------------------------------------------------------ gate / up item

// Where gate/up item `tile` lives in a record: rows P*tile .. +P-1 of gate and of up,
// codes and scales.
struct GuRuns {
    size_t cg, cu, sg, su;      // record offsets: gate codes, up codes, gate scales, up scales
    uint32_t nc, ns;            // bytes of one matrix's codes / scales in the item
};
__device__ __forceinline__ GuRuns gu_runs(const DecodeArgs& a, int tile) {
    const int H = a.H, I = a.I, P = decode_pairs(H), sb = a.mx ? 32 : 16;
    GuRuns r;
    r.cg = (size_t)(tile * P) * (H / 2);
    r.cu = (size_t)(I + tile * P) * (H / 2);
    r.sg = a.off_gu_scales + (size_t)(tile * P) * (H / sb);
    r.su = a.off_gu_scales + (size_t)(I + tile * P) * (H / sb);
    r.nc = (uint32_t)P * (H / 2);
    r.ns = (uint32_t)P * (H / sb);
    return r;
}

// Weights of gate/up item `tile` into wc / ws (gate rows first), bulk copies on `bar`.
__device__ __forceinline__ void stage_gate_up(const DecodeArgs& a, UnitRef ur, int tile, uint8_t* wc,
                                              uint8_t* ws, uint64_t* bar) {
    const GuRuns r = gu_runs(a, tile);
    if (threadIdx.x == 0) {
        bulk_wait_read();                              // wc / ws no longer read by stores
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_tx(bar, 2 * (r.nc + r.ns));
        bulk_g2s(wc, ur.src + r.cg, r.nc, bar);
        bulk_g2s(wc + r.nc, ur.src + r.cu, r.nc, bar);
        bulk_g2s(ws, ur.src + r.sg, r.ns, bar);
        bulk_g2s(ws + r.ns, ur.src + r.su, r.ns, bar);
    }
}

// A fill's staged gate/up item into its victim slot (thread 0, after the item landed).
__device__ __forceinline__ void store_gate_up(const DecodeArgs& a, UnitRef ur, int tile, const uint8_t* wc,
                                              const uint8_t* ws) {
    const GuRuns r = gu_runs(a, tile);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    bulk_s2g(ur.dst + r.cg, wc, r.nc);
    bulk_s2g(ur.dst + r.cu, wc + r.nc, r.nc);
    bulk_s2g(ur.dst + r.sg, ws, r.ns);
    bulk_s2g(ur.dst + r.su, ws + r.ns, r.ns);
    bulk_commit();
}

// h = silu(g) * u of the item's row pairs for NT tokens (x rows xrow[]), from the
// staged weights.  Warp w takes pairs w, w + 8, ...; lane l chunk l + 32m of a row.
template <int NT>
__device__ void gate_up_rows(const DecodeArgs& a, const SmemStatic& S, const uint4* xs, const uint8_t* wc,
                             const uint8_t* ws, int tile, int pair0, const int* xrow, float s_gu) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, P = decode_pairs(H);
    const int nch = H / 32, pieces = H / 8, rb = H / 2, srow = H / (a.mx ? 32 : 16);
#pragma unroll 1
    for (int p = warp; p < P; p += kWarps) {
        float ag[NT], au[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) { ag[t] = 0.f; au[t] = 0.f; }
        const uint8_t* cgp = wc + (size_t)p * rb;
        const uint8_t* cup = wc + (size_t)(P + p) * rb;
        const uint8_t* sgp = ws + (size_t)p * srow;
        const uint8_t* sup = ws + (size_t)(P + p) * srow;
#pragma unroll 1
        for (int ch = lane; ch < nch; ch += 32) {
            const uint4 wg = *reinterpret_cast<const uint4*>(cgp + ch * 16);
            const uint4 wu = *reinterpret_cast<const uint4*>(cup + ch * 16);
            const float2 fg = chunk_scales(sgp, ch, a.mx);
            const float2 fu = chunk_scales(sup, ch, a.mx);
            const uint32_t gw[4] = {wg.x, wg.y, wg.z, wg.w};
            const uint32_t uw[4] = {wu.x, wu.y, wu.z, wu.w};
            float pg[2][NT], pu[2][NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) { pg[0][t] = pg[1][t] = pu[0][t] = pu[1][t] = 0.f; }
#pragma unroll
            for (int pi = 0; pi < 4; ++pi) {          // 8-element pieces; block = pi / 2
                uint32_t dg[4], du[4];
                e2m1x8_to_f16x2(gw[pi], dg);
                e2m1x8_to_f16x2(uw[pi], du);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const uint4 xv = xs[xrow[t] * pieces + xswz(4 * ch + pi)];
                    pg[pi >> 1][t] = dot8_f16(dg, xv, pg[pi >> 1][t]);
                    pu[pi >> 1][t] = dot8_f16(du, xv, pu[pi >> 1][t]);
                }
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                ag[t] = fmaf(pg[0][t], fg.x, ag[t]);
                ag[t] = fmaf(pg[1][t], fg.y, ag[t]);
                au[t] = fmaf(pu[0][t], fu.x, au[t]);
                au[t] = fmaf(pu[1][t], fu.y, au[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float gsum = warp_sum(ag[t]);
            const float usum = warp_sum(au[t]);
            if (lane == 0) {
                const float xm = S.xmul[xrow[t]];
                const float g = gsum * s_gu * xm;
                const float uu = usum * s_gu * xm;
                const float hv = g / (1.f + expf(-g)) * uu;
                st_relaxed_u64(a.h + (size_t)(pair0 + t) * I + tile * P + p, tagged(hv, S.tag));
            }
        }
    }
}

// The gate/up rows of one token at H = 2048 (P = 16 pairs, 64 chunks of 32 elements per
// row): warp w takes pairs w and w + 8, lane l chunks l and l + 32 of each row, with
// the lane's 64 x values read from shared memory once.  Per row the same sums as
// gate_up_rows; the four per-lane row partials (gate and up of both pairs) meet in one
// butterfly over the warp (6 shuffles instead of 4 x 5, the same additions in the same
// order as a warp sum), after which lanes 0 and 16 hold gate and up of their pair.
__device__ void gate_up_rows_t1_h2048(const DecodeArgs& a, const SmemStatic& S, const uint4* xs,
                                      const uint8_t* wc, const uint8_t* ws, int tile, int pair0, int xr,
                                      float s_gu) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int P = 16, rb = 1024, pieces = 256;
    const int srow = 2048 / (a.mx ? 32 : 16);
    uint4 xv[2][4];
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
        for (int pi = 0; pi < 4; ++pi) xv[c2][pi] = xs[xr * pieces + xswz(4 * (lane + 32 * c2) + pi)];
    float r[4];
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        const int p = warp + 8 * pp;
        const uint8_t* cgp = wc + (size_t)p * rb;
        const uint8_t* cup = wc + (size_t)(P + p) * rb;
        const uint8_t* sgp = ws + (size_t)p * srow;
        const uint8_t* sup = ws + (size_t)(P + p) * srow;
        float ag = 0.f, au = 0.f;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            const int ch = lane + 32 * c2;
            const uint4 wg = *reinterpret_cast<const uint4*>(cgp + ch * 16);
            const uint4 wu = *reinterpret_cast<const uint4*>(cup + ch * 16);
            const float2 fg = chunk_scales(sgp, ch, a.mx);
            const float2 fu = chunk_scales(sup, ch, a.mx);
            const uint32_t gw[4] = {wg.x, wg.y, wg.z, wg.w};
            const uint32_t uw[4] = {wu.x, wu.y, wu.z, wu.w};
            float pg[2] = {0.f, 0.f}, pu[2] = {0.f, 0.f};
#pragma unroll
            for (int pi = 0; pi < 4; ++pi) {
                uint32_t dg[4], du[4];
                e2m1x8_to_f16x2(gw[pi], dg);
                e2m1x8_to_f16x2(uw[pi], du);
                pg[pi >> 1] = dot8_f16(dg, xv[c2][pi], pg[pi >> 1]);
                pu[pi >> 1] = dot8_f16(du, xv[c2][pi], pu[pi >> 1]);
            }
            ag = fmaf(pg[0], fg.x, ag);
            ag = fmaf(pg[1], fg.y, ag);
            au = fmaf(pu[0], fu.x, au);
            au = fmaf(pu[1], fu.y, au);
        }
        r[2 * pp] = ag;
        r[2 * pp + 1] = au;
    }
    const bool b16 = (lane & 16) != 0, b8 = (lane & 8) != 0;
    float a0 = b16 ? r[2] : r[0], a1 = b16 ? r[3] : r[1];
    const float s0 = b16 ? r[0] : r[2], s1 = b16 ? r[1] : r[3];
    a0 += __shfl_xor_sync(0xffffffffu, s0, 16);
    a1 += __shfl_xor_sync(0xffffffffu, s1, 16);
    float c = b8 ? a1 : a0;
    c += __shfl_xor_sync(0xffffffffu, b8 ? a0 : a1, 8);
    c += __shfl_xor_sync(0xffffffffu, c, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    const float up = __shfl_xor_sync(0xffffffffu, c, 8);
    if ((lane & 15) == 0) {                               // lanes 0, 16: gate in c, up in `up`
        const int p = warp + 8 * (lane >> 4);
        const float xm = S.xmul[xr];
        const float g = c * s_gu * xm;
        const float uu = up * s_gu * xm;
        const float hv = g / (1.f + expf(-g)) * uu;
        st_relaxed_u64(a.h + (size_t)pair0 * a.I + tile * P + p, tagged(hv, S.tag));
    }
}

// One gate/up item: every token group of the unit, on the staged weights.
// (The caller has staged the item's weights with stage_gate_up.)
__device__ void gate_up_item(const DecodeArgs& a, SmemStatic& S, uint4* xs, uint8_t* wc, uint8_t* ws,
                             uint32_t& par_w, UnitRef ur, int tile, int pair0, uint32_t tokmask,
                             bool staged_all) {
    const bool fill = ur.dst != nullptr;
    const float s_gu = *reinterpret_cast<const float*>(ur.src + a.off_s_gu);
    const bool landed = mbar_wait(&S.bar_w, par_w);
    if (!landed) S.timeout = 1;
    par_w ^= 1u;
    if (fill && landed && threadIdx.x == 0) store_gate_up(a, ur, tile, wc, ws);
    const int ntok = __popc(tokmask);
    for (int g0 = 0; g0 < ntok; g0 += kTok) {
        int toks[kTok];
        const int ntg = group_tokens(tokmask, g0, toks);
        int xrow[kTok];
        if (staged_all) {
#pragma unroll
            for (int t = 0; t < kTok; ++t) xrow[t] = t < ntg ? toks[t] : 0;
        } else {
            stage_x(a, S, xs, toks, ntg);                 // ends with a barrier
#pragma unroll
            for (int t = 0; t < kTok; ++t) xrow[t] = t;
        }
        __syncthreads();                                  // staged weights (fills) and x visible
        switch (ntg) {
            case 1:
                if (a.H == 2048) gate_up_rows_t1_h2048(a, S, xs, wc, ws, tile, pair0 + g0, xrow[0], s_gu);
                else gate_up_rows<1>(a, S, xs, wc, ws, tile, pair0 + g0, xrow, s_gu);
                break;
            case 2: gate_up_rows<2>(a, S, xs, wc, ws, tile, pair0 + g0, xrow, s_gu); break;
            case 3: gate_up_rows<3>(a, S, xs, wc, ws, tile, pair0 + g0, xrow, s_gu); break;
            default: gate_up_rows<4>(a, S, xs, wc, ws, tile, pair0 + g0, xrow, s_gu); break;
        }
        __syncthreads();                                  // xs is restaged by the next group
    }
}

// Where unit u's record is read from, and written to (fills only).
__device__ __forceinline__ UnitRef unit_ref_of(const DecodeArgs& a, const Decision& D, int q, int n_routed,
                                               int u) {
    UnitRef ur;
    if (u < q) {
        ur.src = a.host_pool + (size_t)(a.layer * a.E + D.u_e[u]) * a.rec_bytes;
        ur.dst = a.slot_buf + (size_t)D.u_s[u] * a.rec_bytes;
    } else if (u < n_routed) {
        ur.src = a.slot_buf + (size_t)D.u_s[u] * a.rec_bytes;
        ur.dst = nullptr;
    } else {
        ur.src = a.shared + (size_t)a.layer * a.rec_bytes;
        ur.dst = nullptr;
    }
    return ur;
}

// ------------------------------------------------------------------ down item

// Where down item `rt` lives in a record: rows R*rt .. +R-1 of W_d, codes and scales.
struct DownRuns {
    size_t co, so;
    uint32_t nc, ns;
};
__device__ __forceinline__ DownRuns down_runs(const DecodeArgs& a, int rt) {
    const int I = a.I, R = decode_rows(I), sb = a.mx ? 32 : 16;
    DownRuns r;
    r.co = a.off_d_codes + (size_t)(rt * R) * (I / 2);
    r.so = a.off_d_scales + (size_t)(rt * R) * (I / sb);
    r.nc = (uint32_t)R * (I / 2);
    r.ns = (uint32_t)R * (I / sb);
    return r;
}

// Weights of down item `rt` into dc / ds, bulk copies on `bar`.  A fill's item 0 also
// copies the record's two tensor-scale words into the victim slot.
__device__ __forceinline__ void stage_down(const DecodeArgs& a, UnitRef ur, int rt, uint8_t* dc,
                                           uint8_t* ds, uint64_t* bar) {
    const DownRuns r = down_runs(a, rt);
    if (threadIdx.x == 0) {
        bulk_wait_read();                              // dc / ds no longer read by stores
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_tx(bar, r.nc + r.ns);
        bulk_g2s(dc, ur.src + r.co, r.nc, bar);
        bulk_g2s(ds, ur.src + r.so, r.ns, bar);
    }
    if (ur.dst != nullptr && rt == 0 && threadIdx.x < 2)   // tensor scales s_gu, s_d
        reinterpret_cast<float*>(ur.dst + a.off_s_gu)[threadIdx.x] =
            reinterpret_cast<const float*>(ur.src + a.off_s_gu)[threadIdx.x];
}

// A fill's staged down item into its victim slot (thread 0, after the item landed).
__device__ __forceinline__ void store_down(const DecodeArgs& a, UnitRef ur, int rt, const uint8_t* dc,
                                           const uint8_t* ds) {
    const DownRuns r = down_runs(a, rt);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    bulk_s2g(ur.dst + r.co, dc, r.nc);
    bulk_s2g(ur.dst + r.so, ds, r.ns);
    bulk_commit();
}

// o = s_d * W_d h for the item's rows and NT tokens (the set bits g0 .. g0+NT-1 of
// the unit's token mask, routing weights S.uw[g0 + t]), from the staged weights,
// added into y: y[token, row] += weight * o.
// Warp w takes rows R/8 * w .. +R/8-1; a row is read by lpr lanes (the power of
// two >= its 16-byte chunks, at most 32), so one instruction covers 32/lpr rows.
template <int NT>
__device__ void down_rows(const DecodeArgs& a, const SmemStatic& S, const float* hs, const uint8_t* dc,
                          const uint8_t* ds, int rt, uint32_t tokmask, int g0, float s_d) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, R = decode_rows(I);
    const int nch = I / 32, rb = I / 2, srow = I / (a.mx ? 32 : 16), hpieces = I / 4;
    int lpr = 1;
    while (lpr < nch && lpr < 32) lpr <<= 1;
    const int rpi = 32 / lpr, sub = lane / lpr, li = lane % lpr;
    const int rows_w = R / kWarps;
    const int groups = (rows_w + rpi - 1) / rpi;
    const float4* hs4 = reinterpret_cast<const float4*>(hs);
#pragma unroll 1
    for (int g = 0; g < groups; ++g) {
        const int rw = g * rpi + sub;                     // row within the warp's rows
        const bool rok = rw < rows_w;
        const int rl = warp * rows_w + rw;                // row within the item
        float acc[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] = 0.f;
#pragma unroll 1
        for (int ch = li; rok && ch < nch; ch += lpr) {
            const uint4 w4 = *reinterpret_cast<const uint4*>(dc + (size_t)rl * rb + ch * 16);
            const float2 f = chunk_scales(ds + rl * srow, ch, a.mx);
            const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                float p0[NT], p1[NT];
#pragma unroll
                for (int t = 0; t < NT; ++t) { p0[t] = 0.f; p1[t] = 0.f; }
#pragma unroll
                for (int wq = 0; wq < 2; ++wq) {
                    uint32_t d[4];
                    e2m1x8_to_f16x2(ww[blk * 2 + wq], d);
                    const int piece = 8 * ch + blk * 4 + wq * 2;
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const float4 ha = hs4[t * hpieces + hswz(piece)];
                        const float4 hb = hs4[t * hpieces + hswz(piece + 1)];
                        const float hv[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&d[j]));
                            p0[t] = fmaf(f2.x, hv[2 * j], p0[t]);
                            p1[t] = fmaf(f2.y, hv[2 * j + 1], p1[t]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < NT; ++t) acc[t] = fmaf(p0[t] + p1[t], blk ? f.y : f.x, acc[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float v = acc[t];
            for (int o = lpr >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (li == 0 && rok) {
                const int tok = (int)__fns(tokmask, 0, g0 + t + 1);
                red_add_f32(a.y + (size_t)tok * H + rt * R + rl, S.uw[g0 + t] * (v * s_d));
            }
        }
    }
}

// The down rows of one token at I = 512 (R = 64 rows per item, 16 chunks of 32 elements
// per row): lane (sub, li) of warp w owns chunk li of rows w*8 + 2g + sub, g = 0..3.
// The chunk's 32 h values are read into registers once; per row the chunk's partial
// sums blocks as down_rows does; the four partials of a lane then meet across the 16
// lanes of its half-warp in one butterfly (5 shuffles instead of 4 x 4), after which
// lane li = 4g' of each half holds row 2g' + sub, and each pair of adjacent rows is
// added into y with one vector add (two scalar adds when y is not 8-byte aligned).
__device__ void down_rows_t1_i512(const DecodeArgs& a, const SmemStatic& S, const float* hs, const uint8_t* dc,
                                  const uint8_t* ds, int rt, uint32_t tokmask, int g0, float s_d) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane >> 4, li = lane & 15;
    const int srow = 512 / (a.mx ? 32 : 16);
    const float4* hs4 = reinterpret_cast<const float4*>(hs);
    float hv[32];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const float4 v = hs4[hswz(8 * li + p)];
        hv[4 * p] = v.x;
        hv[4 * p + 1] = v.y;
        hv[4 * p + 2] = v.z;
        hv[4 * p + 3] = v.w;
    }
    float res[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int rl = warp * 8 + 2 * g + sub;
        const uint4 w4 = *reinterpret_cast<const uint4*>(dc + (size_t)rl * 256 + li * 16);
        const float2 f = chunk_scales(ds + rl * srow, li, a.mx);
        const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
        float acc = 0.f;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            float p0 = 0.f, p1 = 0.f;
#pragma unroll
            for (int wq = 0; wq < 2; ++wq) {
                uint32_t d[4];
                e2m1x8_to_f16x2(ww[blk * 2 + wq], d);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 c2 = __half22float2(*reinterpret_cast<const __half2*>(&d[j]));
                    const int e = blk * 16 + wq * 8 + 2 * j;
                    p0 = fmaf(c2.x, hv[e], p0);
                    p1 = fmaf(c2.y, hv[e + 1], p1);
                }
            }
            acc = fmaf(p0 + p1, blk ? f.y : f.x, acc);
        }
        res[g] = acc;
    }
    const bool b8 = (li & 8) != 0, b4 = (li & 4) != 0;
    float a0 = b8 ? res[2] : res[0], a1 = b8 ? res[3] : res[1];
    const float s0 = b8 ? res[0] : res[2], s1 = b8 ? res[1] : res[3];
    a0 += __shfl_xor_sync(0xffffffffu, s0, 8);
    a1 += __shfl_xor_sync(0xffffffffu, s1, 8);
    float c = b4 ? a1 : a0;
    c += __shfl_xor_sync(0xffffffffu, b4 ? a0 : a1, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    const float c_odd = __shfl_xor_sync(0xffffffffu, c, 16);    // row 2g' + 1 (the other half)
    if (sub == 0 && (li & 3) == 0) {
        const int gq = 2 * (li >> 3) + ((li >> 2) & 1);
        const int tok = (int)__fns(tokmask, 0, g0 + 1);
        const float wsc = S.uw[g0] * s_d;
        float* yp = a.y + (size_t)tok * a.H + rt * 64 + warp * 8 + 2 * gq;
        if ((reinterpret_cast<uintptr_t>(yp) & 7) == 0) {
            red_add_v2_f32(yp, wsc * c, wsc * c_odd);
        } else {
            red_add_f32(yp, wsc * c);
            red_add_f32(yp + 1, wsc * c_odd);
        }
    }
}

// One down item: stage the weights (unless prefetched), wait for the unit's h,
// then every token group, added into y.  A token's weight for a routed unit is the
// sum of its routing weights to that expert (one route, unless the token lists the
// expert twice); for the shared expert it is 1.
__device__ void down_item(const DecodeArgs& a, SmemStatic& S, const Decision& D, float* hs, uint8_t* dc,
                          uint8_t* ds, uint32_t& par_d, bool prefetched, UnitRef ur, int u, bool shared_unit,
                          int rt, int pair0, uint32_t tokmask) {
    const int I = a.I;
    const bool fill = ur.dst != nullptr;
    const unsigned tag = S.tag;
    const float s_d = *reinterpret_cast<const float*>(ur.src + a.off_s_d);
    if (!prefetched) stage_down(a, ur, rt, dc, ds, &S.bar_d);
    if ((int)threadIdx.x < __popc(tokmask)) {          // (published by the barrier below)
        const int b = (int)__fns(tokmask, 0, threadIdx.x + 1);
        float wsum = 1.f;
        if (!shared_unit) {
            wsum = 0.f;
            for (int j = 0; j < a.k; ++j)
                if (D.r_unit[b * a.k + j] == u) wsum += a.w[b * a.k + j];
        }
        S.uw[threadIdx.x] = wsum;
    }
    int timeout = 0;
    __syncthreads();
    const bool landed = mbar_wait(&S.bar_d, par_d);
    if (!landed) timeout = 1;
    par_d ^= 1u;
    if (fill && landed && threadIdx.x == 0) store_down(a, ur, rt, dc, ds);
    const int ntok = __popc(tokmask);
    for (int g0 = 0; g0 < ntok; g0 += kTok) {
        const int ntg = min(kTok, ntok - g0);
        // the unit's h: every word carries the call's tag, so a word not yet written by
        // its gate/up item (an older tag) is polled until it is
        const int ne = ntg * I;
        for (int e0 = threadIdx.x; e0 < ne; e0 += 8 * kThreads) {
            float v[8];
            const unsigned long long* hb = a.h + (size_t)(pair0 + g0) * I + e0;
            fetch_tagged<8>([&](int i) { return e0 + i * kThreads < ne ? hb + i * kThreads : nullptr; },
                          tag, v, &timeout);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + i * kThreads;
                if (e < ne) {
                    const int t = e / I, ii = e - t * I;
                    hs[t * I + hswz(ii >> 2) * 4 + (ii & 3)] = v[i];
                }
            }
        }
        __syncthreads();                                   // h (and the fills' weights) visible
        switch (ntg) {
            case 1:
                if (I == 512) down_rows_t1_i512(a, S, hs, dc, ds, rt, tokmask, g0, s_d);
                else down_rows<1>(a, S, hs, dc, ds, rt, tokmask, g0, s_d);
                break;
            case 2: down_rows<2>(a, S, hs, dc, ds, rt, tokmask, g0, s_d); break;
            case 3: down_rows<3>(a, S, hs, dc, ds, rt, tokmask, g0, s_d); break;
            default: down_rows<4>(a, S, hs, dc, ds, rt, tokmask, g0, s_d); break;
        }
        __syncthreads();                                   // hs is restaged by the next group
    }
    if (timeout) S.timeout = 1;
}

// Early staging of a CTA's first down item (a hit unit: bulk copies only); out of
// line, it runs once per CTA.
__device__ __noinline__ void prefetch_down(const DecodeArgs& a, const Decision& D, int q, int n_routed,
                                           int u, int rt, uint8_t* dc, uint8_t* ds, uint64_t* bar) {
    stage_down(a, unit_ref_of(a, D, q, n_routed, u), rt, dc, ds, bar);
}

// ------------------------------------------------------------------ decision

// Fast path, up to 32 routes: warp 0 alone, on the layer's slot_for_id row staged in
// shared memory.  Lane r holds route r (id); lane p < min(C, R) holds LRU position p
// (head).  Ranks in ascending expert id come from bitmaps over the experts (S.hitw,
// S.missw) and the hit test of the LRU head from a bitmap over the slots
// (S.touched); all three are zero on entry.
__device__ void decide_warp(const DecodeArgs& a, SmemStatic& S, const Decision& D,
                            const int32_t* srow, int id, int head) {
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int R = a.B * a.k, E = a.E, C = a.C, k = a.k;
    const int nhead = min(C, R);
    const bool valid = lane < R && id >= 0 && id < E;
    // routes of one expert form a group; its lowest lane leads it
    const unsigned grp = __match_any_sync(FULL, valid ? (unsigned)id : (0x80000000u | (unsigned)lane));
    const int leader = __ffs(grp) - 1;
    const bool lead = valid && leader == lane;
    const int slot = lead ? srow[id] : -1;
    const unsigned hitm = __ballot_sync(FULL, lead && slot >= 0);
    const unsigned missm = __ballot_sync(FULL, lead && slot < 0);
    const int n_hit = __popc(hitm), m = __popc(missm);
    int q = a.split_mode == FT_SPLIT_FULL_OFFLOAD ? m : q_rule_dev(m, a.f_q16);
    if (q > C - n_hit) q = C - n_hit;
    if (q < 0) q = 0;
    if (lead) {
        atomicOr(slot >= 0 ? &S.hitw[id >> 5] : &S.missw[id >> 5], 1u << (id & 31));
        if (slot >= 0) atomicOr(&S.touched[slot >> 5], 1u << (slot & 31));
    }
    __syncwarp();
    // rank among the hits (misses) = set bits of the expert bitmap below id
    int rank = 0;
    if (lead) {
        const uint32_t* bits = slot >= 0 ? S.hitw : S.missw;
        for (int w = 0; w < (id >> 5); ++w) rank += __popc(bits[w]);
        rank += __popc(bits[id >> 5] & ((1u << (id & 31)) - 1u));
    }
    const bool touched = head >= 0 && ((S.touched[head >> 5] >> (head & 31)) & 1u);
    const unsigned untm = __ballot_sync(FULL, lane < nhead && !touched);
    const int vrank = __popc(untm & ((1u << lane) - 1u));
    int unit = -1;
    if (lead) unit = slot >= 0 ? q + rank : (rank < q ? rank : -1);
    unsigned tm = 0;
    for (unsigned g = grp; g; g &= g - 1) tm |= 1u << ((__ffs(g) - 1) / k);
    // (unit, token) pairs: lane u scans the token counts of unit u (units < 32 + shared)
    const int n_routed = q + n_hit;
    const bool has_shared = a.shared != nullptr;
    const int n_units = n_routed + (has_shared ? 1 : 0);
    int* ucnt = S.scan;
    if (unit >= 0) ucnt[unit] = __popc(tm);
    __syncwarp();
    const int c = lane < n_routed ? ucnt[lane] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += t;
    }
    const int routed_pairs = __shfl_sync(FULL, incl, 31);
    const int n_pairs = routed_pairs + (has_shared ? a.B : 0);
    if (lane < n_routed) D.u_pair0[lane] = incl - c;
    if (lane == 0) {
        if (has_shared) D.u_pair0[n_routed] = routed_pairs;
        D.u_pair0[n_units] = n_pairs;
    }
    if (unit >= 0) {
        D.u_e[unit] = id;
        D.u_mask[unit] = tm;
        if (slot >= 0) D.u_s[unit] = slot;
    }
    if (lane < nhead && !touched && vrank < q) D.u_s[vrank] = head;
    if (lane == 0 && has_shared) {
        D.u_e[n_routed] = -1;
        D.u_s[n_routed] = -1;
        D.u_mask[n_routed] = a.B >= 32 ? 0xffffffffu : ((1u << a.B) - 1u);
    }
    __syncwarp();
    const int lunit = __shfl_sync(FULL, unit, leader);
    const unsigned ltm = __shfl_sync(FULL, tm, leader);
    if (lane < R) {
        const int b = lane / k;
        D.r_unit[lane] = valid ? lunit : -2;
        D.r_pair[lane] = (valid && lunit >= 0) ? D.u_pair0[lunit] + __popc(ltm & ((1u << b) - 1u)) : -1;
    }
    const unsigned badm = __ballot_sync(FULL, lane < R && !valid);
    const unsigned defm = __ballot_sync(FULL, valid && lunit < 0);
    if (lane == 0) {
        S.n_hit = n_hit; S.m = m; S.q = q; S.n_routed = n_routed; S.n_units = n_units;
        S.n_pairs = n_pairs; S.n_def = __popc(defm); S.bad = badm != 0;
    }
}

// General path: the whole CTA, any R up to kMaxRoutes.  s_slot / s_unit are [E]
// scratch; the head positions are read contiguously per thread for the scan.
__device__ void decide_block(const DecodeArgs& a, SmemStatic& S, const Decision& D,
                             int32_t* s_slot, int16_t* s_unit) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E, C = a.C, B = a.B, k = a.k, R = B * k;
    const int base_id = a.layer * E;
    const int nwE = (E + 31) / 32, nwC = (C + 31) / 32;
    const int nhead = min(C, R);
    const int hp = (nhead + kThreads - 1) / kThreads;
    int my_id[kMaxPerThread], my_head[kMaxPerThread];
#pragma unroll
    for (int j = 0; j < kMaxPerThread; ++j) {
        const int r = tid + kThreads * j;
        my_id[j] = r < R ? a.ids[r] : -1;
        const int pos = tid * hp + j;
        my_head[j] = (j < hp && pos < nhead) ? a.lru_order[pos] : -1;
    }
    for (int i = tid; i < nwE; i += kThreads) { S.hitw[i] = 0; S.missw[i] = 0; }
    for (int i = tid; i < nwC; i += kThreads) S.touched[i] = 0;
    for (int e = tid; e < E; e += kThreads) { s_slot[e] = -2; s_unit[e] = -1; }
    if (tid == 0) { S.n_def = 0; S.bad = 0; }
    __syncthreads();

    // dedupe: each present expert looks up its slot once
#pragma unroll
    for (int j = 0; j < kMaxPerThread; ++j) {
        const int r = tid + kThreads * j;
        if (r >= R) continue;
        const int id = my_id[j];
        if (id < 0 || id >= E) { S.bad = 1; continue; }
        if (atomicCAS(&s_slot[id], -2, -3) == -2) {
            const int s = a.slot_for_id[base_id + id];
            s_slot[id] = s;
            if (s >= 0) {
                atomicOr(&S.hitw[id >> 5], 1u << (id & 31));
                atomicOr(&S.touched[s >> 5], 1u << (s & 31));
            } else {
                atomicOr(&S.missw[id >> 5], 1u << (id & 31));
            }
        }
    }
    __syncthreads();

    // ranks of hits and misses in ascending expert id; q
    if (warp == 0) warp_word_prefix(S.hitw, S.hpre, nwE, lane);
    if (warp == 1) warp_word_prefix(S.missw, S.mpre, nwE, lane);
    __syncthreads();
    const int n_hit = S.hpre[nwE], m = S.mpre[nwE];
    int q = a.split_mode == FT_SPLIT_FULL_OFFLOAD ? m : q_rule_dev(m, a.f_q16);
    if (q > C - n_hit) q = C - n_hit;
    if (q < 0) q = 0;
    const int n_routed = q + n_hit;
    const bool has_shared = a.shared != nullptr;
    const int n_units = n_routed + (has_shared ? 1 : 0);
    const uint32_t all_tok = B >= 32 ? 0xffffffffu : ((1u << B) - 1u);

    // units (fills = the first q misses, then hits) and victims
    for (int e = tid; e < E; e += kThreads) {
        if (bit_test(S.hitw, e)) {
            const int u = q + bit_rank(S.hitw, S.hpre, e);
            D.u_e[u] = e;
            D.u_s[u] = s_slot[e];
            s_unit[e] = (int16_t)u;
        } else if (bit_test(S.missw, e)) {
            const int rk = bit_rank(S.missw, S.mpre, e);
            if (rk < q) {
                D.u_e[rk] = e;
                s_unit[e] = (int16_t)rk;
            }
        }
    }
    for (int u = tid; u < n_units; u += kThreads) D.u_mask[u] = u < n_routed ? 0u : all_tok;
    unsigned untouched = 0;
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kMaxPerThread; ++j) {
        if (my_head[j] >= 0 && !bit_test(S.touched, my_head[j])) { untouched |= 1u << j; ++cnt; }
    }
    const int ut_rank0 = block_exclusive_scan(cnt, nullptr, S.scan);
    {
        int rk = ut_rank0;
#pragma unroll
        for (int j = 0; j < kMaxPerThread; ++j) {
            if (untouched >> j & 1u) {
                if (rk < q) D.u_s[rk] = my_head[j];
                ++rk;
            }
        }
    }
    if (tid == 0 && has_shared) { D.u_e[n_routed] = -1; D.u_s[n_routed] = -1; }
    __syncthreads();

    // token masks of the units; deferred routes
#pragma unroll
    for (int j = 0; j < kMaxPerThread; ++j) {
        const int r = tid + kThreads * j;
        if (r >= R) continue;
        const int id = my_id[j];
        if (id < 0 || id >= E) continue;
        const int u = s_unit[id];
        if (u >= 0) atomicOr(&D.u_mask[u], 1u << (r / k));
        else atomicAdd(&S.n_def, 1);
    }
    __syncthreads();

    // (unit, token) pairs: unit u owns pairs u_pair0[u] .. + popc(mask)
    {
        const int up = (n_units + kThreads - 1) / kThreads;
        int c2 = 0;
#pragma unroll
        for (int j = 0; j < kMaxPerThread; ++j) {
            const int u = tid * up + j;
            if (j < up && u < n_units) c2 += __popc(D.u_mask[u]);
        }
        int n_pairs = 0;
        int p = block_exclusive_scan(c2, &n_pairs, S.scan);
#pragma unroll
        for (int j = 0; j < kMaxPerThread; ++j) {
            const int u = tid * up + j;
            if (j < up && u < n_units) { D.u_pair0[u] = p; p += __popc(D.u_mask[u]); }
        }
        if (tid == 0) {
            D.u_pair0[n_units] = n_pairs;
            S.n_hit = n_hit; S.m = m; S.q = q; S.n_routed = n_routed; S.n_units = n_units;
            S.n_pairs = n_pairs;
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kMaxPerThread; ++j) {
        const int r = tid + kThreads * j;
        if (r >= R) continue;
        const int id = my_id[j];
        int pr = -1, un = -2;
        if (id >= 0 && id < E) {
            un = s_unit[id];
            if (un >= 0) {
                const int b = r / k;
                pr = D.u_pair0[un] + __popc(D.u_mask[un] & ((1u << b) - 1u));
            }
        }
        D.r_pair[r] = pr;
        D.r_unit[r] = un;
    }
}

}  // namespace

// ------------------------------------------------------------------ the kernel

__global__ void __launch_bounds__(kThreads, 2) decode_layer_kernel(DecodeArgs a) {
    __shared__ SmemStatic S;
    extern __shared__ __align__(128) uint8_t dsm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        mbar_init(&S.bar_w, 1);
        mbar_init(&S.bar_d, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait_and_release();

    const bool commit_cta = blockIdx.x == gridDim.x - 1;
    const int n_compute = gridDim.x - 1;
    const int E = a.E, C = a.C, B = a.B, k = a.k, R = B * k;
    const int base_id = a.layer * E;
    const DynLayout L = dyn_layout(a.H, a.I, E, a.R_cap);
    Decision D;
    D.u_e = reinterpret_cast<int32_t*>(dsm + L.ue);
    D.u_s = reinterpret_cast<int32_t*>(dsm + L.us);
    D.u_mask = reinterpret_cast<uint32_t*>(dsm + L.umask);
    D.u_pair0 = reinterpret_cast<int32_t*>(dsm + L.upair0);
    D.r_pair = reinterpret_cast<int32_t*>(dsm + L.rpair);
    D.r_unit = reinterpret_cast<int32_t*>(dsm + L.runit);
    uint4* xs = reinterpret_cast<uint4*>(dsm + L.stage);
    unsigned long long* epoch_p = reinterpret_cast<unsigned long long*>(a.sync);
    unsigned* read_done = a.sync + 2;

    if (tid == kThreads - 32) {   // the last warp (not the deciding one) reads the call's tick
        S.tick = a.sc->tick + 1;
        unsigned long long e = *epoch_p + 1;
        if ((unsigned)e == 0u) ++e;                      // tag 0 marks scrubbed words
        S.epoch = e;
        S.tag = (unsigned)e;
        S.timeout = 0;
    }
    // ---- 1. decision (and, for B <= kTok, x staged by the other warps meanwhile)
    const bool staged_all = B <= kTok;
    if (R <= 32) {
        // one round trip: the route ids and the LRU head (warp 0) and the layer's
        // slot_for_id row (every thread, into shared memory)
        int32_t* srow = reinterpret_cast<int32_t*>(dsm + L.slot);
        int my_id = -1, my_head = -1;
        if (warp == 0) {
            my_id = lane < R ? a.ids[lane] : -1;
            my_head = lane < min(C, R) ? a.lru_order[lane] : -1;
        }
        for (int e = tid; e < E; e += kThreads) srow[e] = a.slot_for_id[base_id + e];
        for (int w = tid; w < (E + 31) / 32; w += kThreads) { S.hitw[w] = 0; S.missw[w] = 0; }
        for (int w = tid; w < (C + 31) / 32; w += kThreads) S.touched[w] = 0;
        __syncthreads();
        if (warp == 0) decide_warp(a, S, D, srow, my_id, my_head);
        else if (staged_all && !commit_cta) stage_x_warps(a, S, xs);
    } else {
        decide_block(a, S, D, reinterpret_cast<int32_t*>(dsm + L.slot),
                     reinterpret_cast<int16_t*>(dsm + L.unit));
        if (staged_all && !commit_cta) {
            __syncthreads();
            int toks[kTok];
#pragma unroll
            for (int t = 0; t < kTok; ++t) toks[t] = t;
            stage_x(a, S, xs, toks, B);
        }
    }
    __syncthreads();
    // every table entry this CTA reads has been consumed
    if (tid == 0 && !commit_cta) atomicAdd(read_done, 1u);
    const int q = S.q, n_hit = S.n_hit, n_routed = S.n_routed, n_units = S.n_units;

    if (commit_cta) {
        const long long tick = S.tick;
        const int nwC = (C + 31) / 32;
        int32_t* v_old = reinterpret_cast<int32_t*>(dsm + L.vold);
        // ---- per-call outputs
        for (int r = tid; r < R; r += kThreads) {
            const int u = D.r_unit[r];
            a.deferred[r] = u == -1 ? base_id + a.ids[r] : -1;
            if (a.route_slot) a.route_slot[r] = u >= 0 ? D.u_s[u] : -1;
        }
        if (tid == 0) {
            const int nd = S.n_def;
            a.sc->counters[0] = n_hit;
            a.sc->counters[1] = S.m;
            a.sc->counters[2] = q;
            a.sc->counters[3] = nd;
            if (a.counters) {
                a.counters[0] = n_hit;
                a.counters[1] = S.m;
                a.counters[2] = q;
                a.counters[3] = nd;
            }
            if (S.bad) atomicOr(&a.sc->status, FT_DEV_BAD_ID);
            if (a.trace) {   // per-call stats ring: 16-byte header, then the records
                const unsigned long long i = atomicAdd(a.trace, 1ull);
                ft_trace_rec* rec = reinterpret_cast<ft_trace_rec*>(a.trace + 2) + (i % a.trace_cap);
                rec->tick = S.tick;
                rec->layer = a.layer;
                rec->n_hit = n_hit;
                rec->m = S.m;
                rec->q = q;
                rec->n_def_routes = nd;
                rec->n_units = n_units;
                rec->t_commit_ns = (long long)gtime();
            }
        }
        // ---- a call with host routes hands them to the host branch: deferred ids,
        // gates and x into its mailbox (device-mapped pinned memory), then the task flag
        // with a system-scope release after every writer's fence; done is cleared first,
        // so the join kernel of this call waits for this call's partial.  A call without
        // host routes touches no host memory (the join reads the count from the
        // workspace).
        if (a.mb && S.n_def > 0) {
            MailboxHeader* hd = reinterpret_cast<MailboxHeader*>(a.mb);
            int32_t* mdef = reinterpret_cast<int32_t*>(a.mb + a.mb_def);
            float* mw = reinterpret_cast<float*>(a.mb + a.mb_w);
            for (int r = tid; r < R; r += kThreads) {
                mdef[r] = D.r_unit[r] == -1 ? base_id + a.ids[r] : -1;
                mw[r] = a.w[r];
            }
            const uint4* xs = reinterpret_cast<const uint4*>(a.x);
            uint4* xd = reinterpret_cast<uint4*>(a.mb + a.mb_x);
            for (int i = tid; i < B * a.H / 8; i += kThreads) xd[i] = xs[i];
            if (tid == 0) {
                hd->layer = a.layer;
                hd->B = B;
                hd->k = k;
                hd->n_def = S.n_def;
                hd->published += 1;
                asm volatile("st.relaxed.sys.global.u32 [%0], 0;" :: "l"(&hd->done) : "memory");
            }
            __threadfence_system();
            __syncthreads();
            if (tid == 0) asm volatile("st.release.sys.global.u32 [%0], 1;" :: "l"(&hd->task) : "memory");
        }
        for (int i = tid; i < q; i += kThreads) v_old[i] = a.id_of_slot[D.u_s[i]];
        // touched slots: the hits' and the victims'
        for (int w = tid; w < nwC; w += kThreads) S.touched[w] = 0;
        __syncthreads();
        for (int u = tid; u < n_routed; u += kThreads)
            atomicOr(&S.touched[D.u_s[u] >> 5], 1u << (D.u_s[u] & 31));
        // ---- wait until no compute CTA will read the tables (or the epoch) again
        if (tid == 0) {
            if (!wait_geq(read_done, (unsigned)n_compute)) atomicOr(&a.sc->status, FT_DEV_TIMEOUT);
            *read_done = 0;
            a.sc->tick = tick;
            *epoch_p = S.epoch;
            __threadfence();
        }
        __syncthreads();
        // ---- fills: victim i takes miss i; evicted ids unmapped
        for (int i = tid; i < q; i += kThreads) {
            const int v = D.u_s[i];
            const int old = v_old[i];
            if (old >= 0) a.slot_for_id[old] = -1;
            a.slot_for_id[base_id + D.u_e[i]] = v;
            a.id_of_slot[v] = base_id + D.u_e[i];
        }
        // ---- LRU order: untouched slots keep their order, touched ones follow
        const int T = n_routed;
        int dst = 0;
        for (int pos0 = 0; pos0 < C; pos0 += kThreads * 4) {
            int ent[4];
            unsigned keep = 0;
            int kc = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int pos = pos0 + tid * 4 + j;
                ent[j] = pos < C ? a.lru_order[pos] : -1;
                if (ent[j] >= 0 && !bit_test(S.touched, ent[j])) { keep |= 1u << j; ++kc; }
            }
            int tot = 0;
            int o = block_exclusive_scan(kc, &tot, S.scan);   // every load above is done
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (keep >> j & 1u) a.lru_order[dst + o++] = ent[j];
            dst += tot;
        }
        if (warp == 0) warp_word_prefix(S.touched, S.tpre, nwC, lane);
        __syncthreads();
        for (int w = tid; w < nwC; w += kThreads) {
            uint32_t bits = S.touched[w];
            int rank = S.tpre[w];
            while (bits) {
                const int s = w * 32 + __ffs(bits) - 1;
                a.lru_order[C - T + rank] = s;
                a.usage[s] = tick;
                ++rank;
                bits &= bits - 1;
            }
        }
        // ---- every 2^31 calls: zero the scratch words this call does not use
        if ((S.tag & 0x7fffffffu) == 1u) {
            const unsigned long long* h_end = a.h + (size_t)S.n_pairs * a.I;
            const unsigned long long* yf_end = a.yflag + (n_units > 0 ? a.H / decode_rows(a.I) : 0);
            for (size_t i = tid; i < a.scrub_words; i += kThreads) {
                unsigned long long* w = a.scrub + i;
                const bool used = (w >= a.h && w < h_end) || (w >= a.yflag && w < yf_end);
                if (!used) *w = 0ull;
            }
        }
        if (tid == 0 && S.timeout) atomicOr(&a.sc->status, FT_DEV_TIMEOUT);
        return;
    }

    // ---- compute CTAs
    if (n_units == 0) {   // every route is on the host share or masked: the GPU partial is 0
        for (int i = blockIdx.x * kThreads + tid; i < B * a.H; i += n_compute * kThreads) a.y[i] = 0.f;
        return;
    }
    const int T1 = a.I / decode_pairs(a.H);              // gate/up items per unit
    const int T2 = a.H / decode_rows(a.I);               // down items per unit (= row tiles)
    const int n1 = n_units * T1, n2 = n_units * T2;
    // ---- y row tiles z == this CTA (mod n_compute): zeroed, then flagged (release)
    // for the down items that add into them.  Warps 1..7 only: warp 0 issues the
    // first weight copies meanwhile.
    if (warp > 0) {
        const int RW = decode_rows(a.I);
        for (int z = blockIdx.x; z < T2; z += n_compute)
            for (int i = tid - 32; i < B * RW; i += kThreads - 32)
                a.y[(size_t)(i / RW) * a.H + z * RW + i % RW] = 0.f;
        asm volatile("bar.sync 1, %0;" :: "r"(kThreads - 32) : "memory");
        if (tid == 32)
            for (int z = blockIdx.x; z < T2; z += n_compute) st_release_u64(a.yflag + z, tagged(0.f, S.tag));
    }
    uint8_t* wc = dsm + L.wc;
    uint8_t* ws = dsm + L.ws;
    uint8_t* dc = dsm + L.dc;
    uint8_t* ds = dsm + L.ds;
    uint32_t par_w = 0, par_d = 0;
    // a first down item of a hit unit has its weights staged early, right after the
    // CTA's first gate/up weights (which come first on the critical path)
    const int p_first = n_compute - 1 - (int)blockIdx.x;
    const bool prefetch = p_first < n2 && p_first / T2 >= q;
    bool prefetch_due = prefetch;
    for (int i = blockIdx.x; i < n1; i += n_compute) {
        const int u = i / T1, tile = i % T1;
        const UnitRef ur = unit_ref_of(a, D, q, n_routed, u);
        stage_gate_up(a, ur, tile, wc, ws, &S.bar_w);
        if (prefetch_due) {
            prefetch_down(a, D, q, n_routed, p_first / T2, p_first % T2, dc, ds, &S.bar_d);
            prefetch_due = false;
        }
        gate_up_item(a, S, xs, wc, ws, par_w, ur, tile, D.u_pair0[u], D.u_mask[u], staged_all);
    }
    if (prefetch_due) prefetch_down(a, D, q, n_routed, p_first / T2, p_first % T2, dc, ds, &S.bar_d);
    // the down items stage h in the range of x and of the gate/up weights: a fill's bulk
    // stores must have read wc / ws first (the down item's barrier orders the other
    // threads after this wait)
    if (tid == 0) bulk_wait_read();
    // the y tiles of this CTA's down items are zeroed (acquire: the adds come after)
    if (warp == 0) {
        int timeout = 0;
        for (int p = p_first + lane * n_compute; p < n2; p += 32 * n_compute)
            if (!wait_tag_acquire(a.yflag + p % T2, S.tag)) timeout = 1;
        if (timeout) S.timeout = 1;
    }
    float* hs = reinterpret_cast<float*>(dsm + L.stage);
    for (int p = p_first; p < n2; p += n_compute) {
        const int u = p / T2, rt = p % T2;
        down_item(a, S, D, hs, dc, ds, par_d, prefetch && p == p_first, unit_ref_of(a, D, q, n_routed, u), u,
                  u >= n_routed, rt, D.u_pair0[u], D.u_mask[u]);
    }
    if (tid == 0) bulk_wait_all();                 // the fills' slot writes are complete
    if (tid == 0 && S.timeout) atomicOr(&a.sc->status, FT_DEV_TIMEOUT);
}

// ------------------------------------------------------------------ host side

static size_t decode_smem(int H, int I, int E, int R_cap) {
    return dyn_layout(H, I, E, R_cap).total;
}

int decode_grid(int H, int I, int E, int R_cap) {
    // the attribute is per kernel and device: keep it at the largest size any cache on
    // the device needs
    static std::mutex mu;
    static size_t attr_bytes[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 0;
    }
    const size_t sm = decode_smem(H, I, E, R_cap);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (sm > attr_bytes[dev]) {
            if (cudaFuncSetAttribute(decode_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sm) != cudaSuccess) {
                cudaGetLastError();
                return 0;
            }
            attr_bytes[dev] = sm;
        }
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_layer_kernel, kThreads, sm) !=
            cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        return 0;
    }
    return sm_count() * per_sm;
}

// The CTAs of one launch wait on each other's flags, so all of them must be resident
// at once: the launch is cooperative (the driver starts it only when the whole grid
// fits, and fails it otherwise) as well as a programmatic dependent of the previous
// kernel on the stream.
cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t s) {
    if (grid < 2) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = decode_smem(a.H, a.I, a.E, a.R_cap);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, decode_layer_kernel, a);
}

// ------------------------------------------------------------------ host share join

// y += the host branch's partial of the call just decoded (mailbox in device-mapped
// pinned memory), once the branch raised `done` (system-scope acquire; bounded wait of
// one second, then FT_DEV_TIMEOUT and no add).  No host routes (*n_def, the call's
// count in the workspace, is 0): nothing to wait for.  Launched as a programmatic
// dependent of the decode kernel: it is scheduled while the decode kernel runs, lets
// the next kernel on the stream be scheduled at once (that kernel waits for this one
// to complete), and starts its work when the decode kernel has completed.
__global__ void host_join_kernel(uint8_t* mb, unsigned mb_y, float* y, int n, const int* n_def, int* status) {
    __shared__ int go;
    MailboxHeader* hd = reinterpret_cast<MailboxHeader*>(mb);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) {
        int g = 0;
        if (*n_def > 0) {
            unsigned v;
            asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(&hd->done) : "memory");
            if (v != 1u) {
                const unsigned long long t0 = gtime();
                for (unsigned it = 0; it < kWaitIters && v != 1u; ++it) {
                    __nanosleep(128);
                    asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(&hd->done) : "memory");
                    if ((it & 63u) == 63u && gtime() - t0 > kWaitNs) break;
                }
            }
            if (v == 1u) g = 1;
            else if (blockIdx.x == 0) atomicOr(status, FT_DEV_TIMEOUT);
        }
        go = g;
    }
    __syncthreads();
    if (!go) return;
    const float* yh = reinterpret_cast<const float*>(mb + mb_y);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) y[i] += __ldcv(yh + i);
}

cudaError_t launch_host_join(uint8_t* mb, unsigned mb_y, float* y, int n, const int* n_def, int* status,
                             cudaStream_t s) {
    const int grid = std::min((n + 255) / 256, 64);
    return launch_pdl(host_join_kernel, dim3(grid), dim3(256), 0, s, mb, mb_y, y, n, n_def, status);
}

// ------------------------------------------------------------------ bounded waits check

// One thread runs each bounded wait of the decode kernel against a condition that
// nothing will satisfy: a counter nobody raises (wait_geq), a word whose tag nobody
// writes (wait_tag_acquire, fetch_tagged) and an mbarrier nobody arrives on
// (mbar_wait).  Bit i of *expired is set when wait i gave up.
__global__ void wait_check_kernel(const unsigned* counter, const unsigned long long* words,
                                  unsigned* expired) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    unsigned bits = 0;
    if (!wait_geq(counter, 1u)) bits |= 1u;
    if (!wait_tag_acquire(words, 7u)) bits |= 2u;
    int timeout = 0;
    float v[8];
    fetch_tagged<8>([&](int i) { return words + i; }, 7u, v, &timeout);
    if (timeout) bits |= 4u;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!mbar_wait(&bar, 0)) bits |= 8u;
    *expired = bits;
}

cudaError_t check_bounded_waits(unsigned* expired) {
    // scratch: [0] counter (0), [1] result, bytes 32..95 eight words with tag 0
    unsigned* d = nullptr;
    cudaError_t e = cudaMalloc(&d, 256);
    if (e != cudaSuccess) return e;
    e = cudaMemset(d, 0, 256);
    if (e == cudaSuccess) {
        wait_check_kernel<<<1, 32>>>(d, reinterpret_cast<const unsigned long long*>(d + 8), d + 1);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpy(expired, d + 1, sizeof(unsigned), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e;
}

}  // namespace ft
