// NVFP4 SwiGLU expert GEMV of one decode layer call, over the GPU units the remap
// kernel listed (fills, hits, shared expert), and the gated combine.
//
// [EXPLAINER §1.1] y = sum_e p_e Expert_{l,e}(x);  [EXPLAINER §6.8] one fused
// expert batch copy and the grouped execution of hits and fills;  [BWRATIO "代码全链路"
// §2] GPU-side weights of CPU routes are zero -- here such routes are skipped
// instead of computed at weight 0;  [JUHE "为什么可以直接相加？"] exact merge.
//
// Kernel 1 (gate_up): persistent CTAs pull work items from a device counter:
//   fill gate/up tiles first (their rows are read from the pinned host pool over
//   the host link and written into the victim slot on the way: one link read per
//   byte), then the plain copies of the fills' W_d part, then the hit and shared
//   tiles (HBM).  A tile is 16 (gate row, up row) pairs; each warp computes both
//   rows of a pair against the same x chunk and emits h = silu(g) * u.
// Kernel 2 (down): work item = (unit, 64 output rows); o = W_d h per (unit, token)
//   pair.  The CTA that completes the last unit of a row tile (device counter,
//   no waiting) sums y[b] = sum_j w[b,j] o_(b,j) in order j, then + shared.
//
// Arithmetic: E2M1 codes become f16 exactly (cvt.rn.f16x2.e2m1x2); x (bf16) is
// staged as f16 after an exact power-of-two prescale that keeps |x| < 2^15; code*x
// products are exact and accumulate in fp32 (fma.rn.f32.f16); each 16-element block
// partial is scaled by its E4M3 scale in fp32; the fp32 tensor scale and the
// prescale are applied at the end.  h stays fp32; the down GEMV is fp32 FMA.
#include "ft_internal.cuh"

namespace ft {

namespace {

__device__ __forceinline__ uint4 ldg16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned short ldg2(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void stg16(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void stg2(void* p, unsigned short v) {
    asm volatile("st.global.u16 [%0], %1;" :: "l"(p), "h"(v) : "memory");
}

// 8 E2M1 codes (one 32-bit word, element 0 in the lowest nibble) -> 4 f16x2.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&o)[4]) {
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

__device__ __forceinline__ float ldcg_f(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

}  // namespace

// ------------------------------------------------------------------ gate / up

__global__ void __launch_bounds__(kGemvThreads) gate_up_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_wait_and_release();
    uint4* xs = reinterpret_cast<uint4*>(smem);          // [kTokGroup][H/8] pieces
    __shared__ unsigned s_item;
    __shared__ int s_tok[kTokGroup];
    __shared__ int s_ntok, s_need;
    __shared__ float s_xmul[kTokGroup];
    __shared__ float s_red[kTokGroup][kGemvThreads / 32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, I = a.I;
    const int n_units = a.sc->n_units, q = a.sc->n_fill;
    const int tiles = I / kRowPairsPerItem;
    const size_t dsz = a.rec_bytes - a.off_d_codes;
    const unsigned dchunks = (unsigned)((dsz + kCopyChunk - 1) / kCopyChunk);
    const unsigned n_fill_items = (unsigned)q * tiles;
    const unsigned n_copy = (unsigned)q * dchunks;
    const unsigned n_items = n_fill_items + n_copy + (unsigned)(n_units - q) * tiles;
    const int pieces = H / 8;
    const int nch = H / 32;
    if (tid == 0) s_ntok = -1;

    for (;;) {
        __syncthreads();
        if (tid == 0) s_item = atomicAdd(&a.sc->work1, 1u);
        __syncthreads();
        const unsigned item = s_item;
        if (item >= n_items) break;

        if (item >= n_fill_items && item < n_fill_items + n_copy) {
            // plain copy of a fill's W_d part (+ tensor scales, padding)
            const unsigned f = (item - n_fill_items) / dchunks;
            const unsigned c = (item - n_fill_items) % dchunks;
            const Unit un = a.units[f];
            const size_t beg = a.off_d_codes + (size_t)c * kCopyChunk;
            size_t end = beg + kCopyChunk;
            if (end > a.rec_bytes) end = a.rec_bytes;
            for (size_t o = beg + (size_t)tid * 16; o < end; o += (size_t)kGemvThreads * 16)
                stg16(un.dst + o, ldg16(un.src + o));
            continue;
        }
        const unsigned ui = item < n_fill_items ? item / tiles
                                                : q + (item - n_fill_items - n_copy) / tiles;
        const int tile = item < n_fill_items ? item % tiles
                                             : (item - n_fill_items - n_copy) % tiles;
        const Unit un = a.units[ui];
        const float s_gu = *reinterpret_cast<const float*>(un.src + a.off_s_gu);

        for (int tg = 0; tg < un.n_tok; tg += kTokGroup) {
            const int ntg = min(kTokGroup, un.n_tok - tg);
            // ---- stage x of this token group (skipped when already staged)
            if (tid == 0) {
                int need = s_ntok != ntg;
                for (int t = 0; t < ntg; ++t) {
                    const int b = a.pair_tok[un.pair0 + tg + t];
                    need |= (t < s_ntok) ? (s_tok[t] != b) : 1;
                    s_tok[t] = b;
                }
                s_ntok = ntg;
                s_need = need;
            }
            __syncthreads();
            if (s_need) {
                float amax[kTokGroup];
#pragma unroll
                for (int t = 0; t < kTokGroup; ++t) amax[t] = 0.f;
                for (int p = tid; p < pieces; p += kGemvThreads) {
#pragma unroll
                    for (int t = 0; t < kTokGroup; ++t) {
                        if (t < ntg) {
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                a.x + (size_t)s_tok[t] * H + p * 8);
                            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float2 f = __bfloat1622float2(b2[j]);
                                amax[t] = fmaxf(amax[t], fmaxf(fabsf(f.x), fabsf(f.y)));
                            }
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < kTokGroup; ++t) {
                    float m = amax[t];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if (lane == 0) s_red[t][warp] = m;
                }
                __syncthreads();
                if (tid < kTokGroup) {
                    float m = 0.f;
                    for (int w = 0; w < kGemvThreads / 32; ++w) m = fmaxf(m, s_red[tid][w]);
                    // keep |x| * 2^-k below 2^15 so the f16 copy cannot overflow
                    int k = 0;
                    if (m >= 32768.f) k = ilogbf(m) - 14;
                    s_xmul[tid] = ldexpf(1.f, k);
                }
                __syncthreads();
                for (int p = tid; p < pieces; p += kGemvThreads) {
#pragma unroll
                    for (int t = 0; t < kTokGroup; ++t) {
                        if (t < ntg) {
                            const float dn = 1.f / s_xmul[t];   // exact power of two
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                a.x + (size_t)s_tok[t] * H + p * 8);
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

            // ---- rows
            for (int rp = warp; rp < kRowPairsPerItem; rp += kGemvThreads / 32) {
                const int i = tile * kRowPairsPerItem + rp;
                const size_t g_off = (size_t)i * (H / 2);
                const size_t u_off = (size_t)(I + i) * (H / 2);
                const size_t gs_off = a.off_gu_scales + (size_t)i * (H / 16);
                const size_t us_off = a.off_gu_scales + (size_t)(I + i) * (H / 16);
                float ag[kTokGroup], au[kTokGroup];
#pragma unroll
                for (int t = 0; t < kTokGroup; ++t) { ag[t] = 0.f; au[t] = 0.f; }
                const bool write = un.dst != nullptr && tg == 0;
                for (int ch = lane; ch < nch; ch += 32) {
                    const uint4 cg = ldg16(un.src + g_off + ch * 16);
                    const uint4 cu = ldg16(un.src + u_off + ch * 16);
                    const unsigned short sg = ldg2(un.src + gs_off + ch * 2);
                    const unsigned short su = ldg2(un.src + us_off + ch * 2);
                    if (write) {
                        stg16(un.dst + g_off + ch * 16, cg);
                        stg16(un.dst + u_off + ch * 16, cu);
                        stg2(un.dst + gs_off + ch * 2, sg);
                        stg2(un.dst + us_off + ch * 2, su);
                    }
                    const float2 fg = e4m3x2_to_float2(sg);
                    const float2 fu = e4m3x2_to_float2(su);
                    uint32_t dg[16], du[16];
                    e2m1x8_to_f16x2(cg.x, *reinterpret_cast<uint32_t(*)[4]>(dg + 0));
                    e2m1x8_to_f16x2(cg.y, *reinterpret_cast<uint32_t(*)[4]>(dg + 4));
                    e2m1x8_to_f16x2(cg.z, *reinterpret_cast<uint32_t(*)[4]>(dg + 8));
                    e2m1x8_to_f16x2(cg.w, *reinterpret_cast<uint32_t(*)[4]>(dg + 12));
                    e2m1x8_to_f16x2(cu.x, *reinterpret_cast<uint32_t(*)[4]>(du + 0));
                    e2m1x8_to_f16x2(cu.y, *reinterpret_cast<uint32_t(*)[4]>(du + 4));
                    e2m1x8_to_f16x2(cu.z, *reinterpret_cast<uint32_t(*)[4]>(du + 8));
                    e2m1x8_to_f16x2(cu.w, *reinterpret_cast<uint32_t(*)[4]>(du + 12));
#pragma unroll
                    for (int t = 0; t < kTokGroup; ++t) {
                        if (t < ntg) {
                            const uint4* xt = xs + t * pieces;
                            const uint4 x0 = xt[xswz(4 * ch + 0)];
                            const uint4 x1 = xt[xswz(4 * ch + 1)];
                            const uint4 x2 = xt[xswz(4 * ch + 2)];
                            const uint4 x3 = xt[xswz(4 * ch + 3)];
                            float g0 = dot8_f16(dg + 0, x0, 0.f);
                            g0 = dot8_f16(dg + 4, x1, g0);
                            float g1 = dot8_f16(dg + 8, x2, 0.f);
                            g1 = dot8_f16(dg + 12, x3, g1);
                            float u0 = dot8_f16(du + 0, x0, 0.f);
                            u0 = dot8_f16(du + 4, x1, u0);
                            float u1 = dot8_f16(du + 8, x2, 0.f);
                            u1 = dot8_f16(du + 12, x3, u1);
                            ag[t] = fmaf(g0, fg.x, ag[t]);
                            ag[t] = fmaf(g1, fg.y, ag[t]);
                            au[t] = fmaf(u0, fu.x, au[t]);
                            au[t] = fmaf(u1, fu.y, au[t]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < kTokGroup; ++t) {
                    if (t < ntg) {
                        const float gsum = warp_sum(ag[t]);
                        const float usum = warp_sum(au[t]);
                        if (lane == 0) {
                            const float g = gsum * s_gu * s_xmul[t];
                            const float uu = usum * s_gu * s_xmul[t];
                            const float hv = g / (1.f + expf(-g)) * uu;
                            a.h[(size_t)(un.pair0 + tg + t) * I + i] = hv;
                        }
                    }
                }
            }
            __syncthreads();
        }
    }
}

// ------------------------------------------------------------------ down + combine

__global__ void __launch_bounds__(kGemvThreads) down_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_wait_and_release();
    float4* hs = reinterpret_cast<float4*>(smem);         // [kTokGroup][I/4] pieces
    __shared__ unsigned s_item;
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, I = a.I, B = a.B, k = a.k;
    const int n_units = a.sc->n_units;
    const int tiles2 = H / kDownRowsPerItem;
    const unsigned n_items = (unsigned)n_units * tiles2;
    const int hpieces = I / 4;
    const int nch = I / 32;
    int lpr = 1;                                 // lanes per row: a power of two
    while (lpr * 2 <= nch && lpr * 2 <= 32) lpr *= 2;
    const int groups = 32 / lpr;
    const int grp = lane / lpr, li = lane % lpr;

    if (n_units == 0) {   // every route is on the host share: the GPU partial is 0
        for (int i = blockIdx.x * kGemvThreads + tid; i < B * H; i += gridDim.x * kGemvThreads)
            a.y[i] = 0.f;
        return;
    }

    for (;;) {
        __syncthreads();
        if (tid == 0) s_item = atomicAdd(&a.sc->work2, 1u);
        __syncthreads();
        const unsigned item = s_item;
        if (item >= n_items) break;
        const int ui = item / tiles2, rt = item % tiles2;
        const Unit un = a.units[ui];
        const uint8_t* rec = un.dst ? un.dst : un.src;   // fills were copied by kernel 1
        const float s_d = *reinterpret_cast<const float*>(rec + a.off_s_d);

        for (int tg = 0; tg < un.n_tok; tg += kTokGroup) {
            const int ntg = min(kTokGroup, un.n_tok - tg);
            for (int p = tid; p < hpieces; p += kGemvThreads) {
#pragma unroll
                for (int t = 0; t < kTokGroup; ++t)
                    if (t < ntg)
                        hs[t * hpieces + hswz(p)] = *reinterpret_cast<const float4*>(
                            a.h + (size_t)(un.pair0 + tg + t) * I + p * 4);
            }
            __syncthreads();
            const int r_base = rt * kDownRowsPerItem + warp * (kDownRowsPerItem / 8);
            // Every lane runs the same number of passes (warp shuffles below need the
            // full warp); lanes whose row pair lies past the warp's 4 pairs idle.
            constexpr int kPairsPerWarp = kDownRowsPerItem / 16;
            for (int rp0 = 0; rp0 < kPairsPerWarp; rp0 += groups) {
                const int rp = rp0 + grp;
                const bool act = rp < kPairsPerWarp;
                const int r0 = r_base + 2 * (act ? rp : 0), r1 = r0 + 1;
                const size_t c0 = a.off_d_codes + (size_t)r0 * (I / 2);
                const size_t c1 = a.off_d_codes + (size_t)r1 * (I / 2);
                const size_t s0 = a.off_d_scales + (size_t)r0 * (I / 16);
                const size_t s1 = a.off_d_scales + (size_t)r1 * (I / 16);
                float acc0[kTokGroup], acc1[kTokGroup];
#pragma unroll
                for (int t = 0; t < kTokGroup; ++t) { acc0[t] = 0.f; acc1[t] = 0.f; }
                for (int ch = li; act && ch < nch; ch += lpr) {
                    const uint4 w0 = ldg16(rec + c0 + ch * 16);
                    const uint4 w1 = ldg16(rec + c1 + ch * 16);
                    const float2 f0 = e4m3x2_to_float2(ldg2(rec + s0 + ch * 2));
                    const float2 f1 = e4m3x2_to_float2(ldg2(rec + s1 + ch * 2));
                    const uint32_t ww0[4] = {w0.x, w0.y, w0.z, w0.w};
                    const uint32_t ww1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        float p0[kTokGroup], p1[kTokGroup];
#pragma unroll
                        for (int t = 0; t < kTokGroup; ++t) { p0[t] = 0.f; p1[t] = 0.f; }
#pragma unroll
                        for (int wq = 0; wq < 2; ++wq) {
                            uint32_t d0[4], d1[4];
                            e2m1x8_to_f16x2(ww0[blk * 2 + wq], d0);
                            e2m1x8_to_f16x2(ww1[blk * 2 + wq], d1);
                            float v0[8], v1[8];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&d0[j]));
                                const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&d1[j]));
                                v0[2 * j] = a0.x; v0[2 * j + 1] = a0.y;
                                v1[2 * j] = a1.x; v1[2 * j + 1] = a1.y;
                            }
                            const int piece = 8 * ch + blk * 4 + wq * 2;
#pragma unroll
                            for (int t = 0; t < kTokGroup; ++t) {
                                if (t < ntg) {
                                    const float4 ha = hs[t * hpieces + hswz(piece)];
                                    const float4 hb = hs[t * hpieces + hswz(piece + 1)];
                                    const float hv[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
#pragma unroll
                                    for (int j = 0; j < 8; ++j) {
                                        p0[t] = fmaf(v0[j], hv[j], p0[t]);
                                        p1[t] = fmaf(v1[j], hv[j], p1[t]);
                                    }
                                }
                            }
                        }
                        const float sc0 = blk ? f0.y : f0.x, sc1 = blk ? f1.y : f1.x;
#pragma unroll
                        for (int t = 0; t < kTokGroup; ++t) {
                            acc0[t] = fmaf(p0[t], sc0, acc0[t]);
                            acc1[t] = fmaf(p1[t], sc1, acc1[t]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < kTokGroup; ++t) {
                    if (t < ntg) {
                        float v0 = acc0[t], v1 = acc1[t];
                        for (int o = lpr >> 1; o > 0; o >>= 1) {
                            v0 += __shfl_xor_sync(0xffffffffu, v0, o);
                            v1 += __shfl_xor_sync(0xffffffffu, v1, o);
                        }
                        if (act && li == 0) {
                            float* orow = a.o + (size_t)(un.pair0 + tg + t) * H;
                            orow[r0] = v0 * s_d;
                            orow[r1] = v1 * s_d;
                        }
                    }
                }
            }
            __syncthreads();
        }

        // tile completion; the CTA finishing the last unit of this row tile combines
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = atomicAdd(&a.tile_done[rt], 1u) == (unsigned)(n_units - 1);
        __syncthreads();
        if (s_last) {
            __threadfence();
            const int sp0 = a.sc->shared_pair0;
            for (int idx = tid; idx < B * kDownRowsPerItem; idx += kGemvThreads) {
                const int b = idx / kDownRowsPerItem;
                const int r = rt * kDownRowsPerItem + idx % kDownRowsPerItem;
                float v = 0.f;
                for (int j = 0; j < k; ++j) {
                    const int p = a.route_pair[b * k + j];
                    if (p >= 0) v = fmaf(a.w[b * k + j], ldcg_f(a.o + (size_t)p * H + r), v);
                }
                if (sp0 >= 0) v += ldcg_f(a.o + (size_t)(sp0 + b) * H + r);
                a.y[(size_t)b * H + r] = v;
            }
        }
    }
}

static size_t gate_up_smem(int H) { return (size_t)kTokGroup * H * 2; }
static size_t down_smem(int I) { return (size_t)kTokGroup * I * 4; }

cudaError_t launch_gate_up(const DecodeArgs& a, int grid, cudaStream_t s) {
    const size_t sm = gate_up_smem(a.H);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(gate_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
        cudaFuncSetAttribute(down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
        attr_set = true;
    }
    return launch_pdl(gate_up_kernel, dim3(grid), dim3(kGemvThreads), sm, s, a);
}

cudaError_t launch_down(const DecodeArgs& a, int grid, cudaStream_t s) {
    return launch_pdl(down_kernel, dim3(grid), dim3(kGemvThreads), down_smem(a.I), s, a);
}

int gemv_occupancy(int H, int I) {
    cudaFuncSetAttribute(gate_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    cudaFuncSetAttribute(down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    int b1 = 1, b2 = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, gate_up_kernel, kGemvThreads, gate_up_smem(H));
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b2, down_kernel, kGemvThreads, down_smem(I));
    int b = b1 < b2 ? b1 : b2;
    return b < 1 ? 1 : b;
}

}  // namespace ft
