// Grouped block-scaled FP4 GEMMs of prefill on the 5th-generation tensor cores
// (tcgen05, kind::mxf4nvf4, E2M1 operands with UE4M3 scales per 16 along K).
//
// [EXPLAINER §4.2] prefill computes layer l from one full-layer buffer while the
// next layer streams into the other; this is the compute side.  Routes are sorted
// by expert; each expert's rows form one group.  Tile = 128 sorted rows x 256
// output columns; K is staged 256 elements (128 bytes per row) at a time.
//   GEMM1: A = quantised x rows, B = W_gu of the expert; the 256 columns are 128
//          gate rows and the matching 128 up rows, so the epilogue computes
//          h = silu(g * s_gu) * (u * s_gu) and quantises h to NVFP4 (unit tensor
//          scale, E4M3 per 16) in place of the accumulator.
//   GEMM2: A = quantised h rows, B = W_d; the epilogue scales by s_d and the route's
//          gate and writes the row of O belonging to the route.
//
// Warp roles (192 threads): warp 0 loads A/B tiles with TMA (SWIZZLE_128B) and the
// scale factors with plain loads into 512-byte 32x4-interleaved atoms; warp 1 (one
// lane) copies the atoms to tensor memory (tcgen05.cp 32x128b.warpx4) and issues
// four 128x256x64 MMAs per stage, accumulating in TMEM; warps 2-5 read the
// accumulator (tcgen05.ld) and run the epilogue.  Every mbarrier wait is bounded:
// on expiry the CTA records FT_DEV_TIMEOUT, drains its own copies and frees TMEM.
#include <cuda.h>
#include <atomic>
#include <cstdio>
#include <mutex>

#include "ft_prefill.cuh"
#include "ft_quant.cuh"
#include "ft_umma.cuh"

namespace ft {

namespace {

constexpr int kBM = 128, kBN = 256, kBKB = 128;          // BK = 256 fp4 = 128 bytes
constexpr int kStages = 4;
constexpr int kSA = kBM * kBKB;                           // 16 KB
constexpr int kSB = kBN * kBKB;                           // 32 KB
constexpr int kSFA = 4 * 512;                             // 4 k-blocks x 128 rows x 4 scales
constexpr int kSFB = 8 * 512;                             // 4 k-blocks x 256 rows x 4 scales
constexpr int kStageBytes = kSA + kSB + kSFA + kSFB;      // 54 KB (multiple of 1024)
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kSfCol0 = 256;                              // accumulator uses columns 0..255
constexpr int kSfStageCols = 48;                          // 16 (A) + 32 (B) per stage
constexpr long kWaitLimit = 1L << 26;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* b, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(b)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(b)) : "memory");
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

// Bounded wait; false once the limit is hit or another role gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
    for (long it = 0; it < kWaitLimit; ++it) {
        if (mbar_try(b, parity)) return true;
        if ((it & 1023) == 1023 && *abort_flag) return false;
    }
    *abort_flag = 1;
    return false;
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                 "[%0], [%1, {%2, %3}], [%4];"
                 :: "r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                 "[%0], [%1, {%2, %3, %4}], [%5];"
                 :: "r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)) : "memory");
}

// K-major operand tile, 128-byte rows, 128B swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Scale-factor atom: 32 rows x 16 bytes, no swizzle, 8-row groups 128 B apart.
__device__ __forceinline__ uint64_t desc_atom(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(128 >> 4) << 16) |
           ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor: E2M1 x E2M1, UE4M3 scales, K-major A and B, M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ void tmem_ld16(uint32_t addr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// An E8M0 scale (2^(c - 127)) as the UE4M3 byte of the same value: exact for
// 2^-9 .. 2^8 (subnormal codes 1, 2, 4 below 2^-6); outside, the nearest end of that
// range and *bad set.
__device__ __forceinline__ uint32_t e8m0_to_ue4m3(uint32_t c, int* bad) {
    const int k = (int)c - 127;
    const int kc = min(max(k, -9), 8);
    *bad |= k != kc;
    return kc >= -6 ? (uint32_t)(kc + 7) << 3 : 1u << (kc + 9);
}

struct TileInfo {
    int e, m0, rows, nt;
};

__device__ __forceinline__ TileInfo tile_info(const UmmaArgs& g, int tile) {
    TileInfo t;
    const int mt = tile / g.n_tiles_n;
    t.nt = tile % g.n_tiles_n;
    int lo = 0, hi = g.E;                    // largest e with mtile_prefix[e] <= mt
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (g.mtile_prefix[mid] <= mt) lo = mid; else hi = mid;
    }
    t.e = lo;
    t.m0 = g.offsets[lo] + (mt - g.mtile_prefix[lo]) * kBM;
    t.rows = min(kBM, g.offsets[lo + 1] - t.m0);
    return t;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
umma_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const UmmaArgs g) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], acc_full, acc_empty;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tiles of m-tiles [m_lo, m_hi) (all of them unless a range is given), n fastest
    const int m_lo = g.mrange ? g.mrange[0] : 0;
    const int m_hi = g.mrange ? g.mrange[1] : g.mtile_prefix[g.E];
    const int total = max(m_hi - m_lo, 0) * g.n_tiles_n;
    const int tile0 = m_lo * g.n_tiles_n;
    const int kstages = g.K / 256;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], 33);          // expect_tx arrival + 32 scale-factor lanes
            mbar_init(&empty_bar[s], 1);          // tcgen05.commit
        }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_empty, 128);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&tmem_base)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int it = 0;
        bool ok = true;
        int scale_bad = 0;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            const TileInfo ti = tile_info(g, tile0 + tile);
            const int slot = g.slot_of ? g.slot_of[ti.e] : g.slot0 + ti.e;
            const uint8_t* rec = g.slot_buf + (size_t)slot * g.rec_bytes;
            for (int ks = 0; ks < kstages; ++ks, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                if (!mbar_wait(&empty_bar[s], ph ^ 1u, &abort_flag)) { ok = false; break; }
                uint8_t* st = smem + s * kStageBytes;
                if (lane == 0) {
                    mbar_arrive_tx(&full_bar[s], kSA + kSB);
                    tma_2d(st, &tmA, ks * kBKB, ti.m0, &full_bar[s]);
                    if (g.kind == 1) {
                        tma_3d(st + kSA, &tmB, ks * kBKB, ti.nt * 128, slot, &full_bar[s]);
                        tma_3d(st + kSA + kSB / 2, &tmB, ks * kBKB, g.I + ti.nt * 128, slot, &full_bar[s]);
                    } else {
                        tma_3d(st + kSA, &tmB, ks * kBKB, ti.nt * kBN, slot, &full_bar[s]);
                    }
                }
                uint8_t* sfa = st + kSA + kSB;
                uint8_t* sfb = sfa + kSFA;
                const int srow = g.K / 16;       // scale bytes per row (activations, NVFP4 B)
                // every scale load of the stage goes out first (4 A rows and 8 B rows per
                // lane in flight), then the 512-byte atoms are written
                uint4 av[kBM / 32], bv[kBN / 32];
#pragma unroll
                for (int j = 0; j < kBM / 32; ++j) {
                    const int row = ti.m0 + lane + 32 * j;
                    av[j] = row < g.R_max
                                ? __ldg(reinterpret_cast<const uint4*>(g.a_scales + (size_t)row * srow + ks * 16))
                                : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int j = 0; j < kBN / 32; ++j) {
                    const int n = lane + 32 * j;
                    const int brow = g.kind == 1 ? (n < 128 ? ti.nt * 128 + n : g.I + ti.nt * 128 + (n - 128))
                                                 : ti.nt * kBN + n;
                    if (!g.mx) {
                        bv[j] = __ldg(reinterpret_cast<const uint4*>(rec + g.off_b_scales + (size_t)brow * srow +
                                                                     ks * 16));
                    } else {                      // 8 E8M0 scales of 32 elements
                        const uint2 v = __ldg(reinterpret_cast<const uint2*>(rec + g.off_b_scales +
                                                                             (size_t)brow * (g.K / 32) + ks * 8));
                        bv[j] = make_uint4(v.x, v.y, 0, 0);
                    }
                }
#pragma unroll
                for (int j = 0; j < kBM / 32; ++j) {
                    const int r = lane + 32 * j;
                    const uint32_t w4[4] = {av[j].x, av[j].y, av[j].z, av[j].w};
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb)
                        *reinterpret_cast<uint32_t*>(sfa + kb * 512 + (r & 31) * 16 + (r >> 5) * 4) = w4[kb];
                }
#pragma unroll
                for (int j = 0; j < kBN / 32; ++j) {
                    const int n = lane + 32 * j;
                    uint32_t w4[4];
                    if (!g.mx) {
                        w4[0] = bv[j].x; w4[1] = bv[j].y; w4[2] = bv[j].z; w4[3] = bv[j].w;
                    } else {                      // -> 16 UE4M3 scales of 16 (each twice)
#pragma unroll
                        for (int kb = 0; kb < 4; ++kb) {
                            const uint32_t word = kb < 2 ? bv[j].x : bv[j].y;
                            const uint32_t s0 = e8m0_to_ue4m3((word >> (16 * (kb & 1))) & 0xFF, &scale_bad);
                            const uint32_t s1 = e8m0_to_ue4m3((word >> (16 * (kb & 1) + 8)) & 0xFF, &scale_bad);
                            w4[kb] = s0 | (s0 << 8) | (s1 << 16) | (s1 << 24);
                        }
                    }
                    const int half = n >> 7, r = n & 127;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb)
                        *reinterpret_cast<uint32_t*>(sfb + (2 * kb + half) * 512 + (r & 31) * 16 + (r >> 5) * 4) = w4[kb];
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(&full_bar[s]);
            }
        }
        if (scale_bad) atomicOr(g.status, FT_DEV_SCALE_RANGE);
        if (!ok) {
            // drain: wait (bounded) for this CTA's TMA copies still in flight
            for (int j = 1; j <= kStages && it - j >= 0; ++j) {
                const int i2 = it - j, s = i2 % kStages;
                const uint32_t ph = (uint32_t)(i2 / kStages) & 1u;
                for (long w = 0; w < (1L << 20) && !mbar_try(&full_bar[s], ph); ++w) {}
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int it = 0, tl = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++tl) {
                if (!mbar_wait(&acc_empty, ((uint32_t)tl & 1u) ^ 1u, &abort_flag)) { ok = false; break; }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                for (int ks = 0; ks < kstages; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_wait(&full_bar[s], ph, &abort_flag)) { ok = false; break; }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    uint8_t* st = smem + s * kStageBytes;
                    const uint32_t a0 = smem_u32(st), b0 = smem_u32(st + kSA);
                    const uint32_t sfa = smem_u32(st + kSA + kSB), sfb = sfa + kSFA;
                    const uint32_t sf_col = tmem + kSfCol0 + s * kSfStageCols;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) {
                        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;"
                                     :: "r"(sf_col + 4 * kb), "l"(desc_atom(sfa + kb * 512)) : "memory");
                        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;"
                                     :: "r"(sf_col + 16 + 8 * kb), "l"(desc_atom(sfb + (2 * kb) * 512)) : "memory");
                        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;"
                                     :: "r"(sf_col + 20 + 8 * kb), "l"(desc_atom(sfb + (2 * kb + 1) * 512)) : "memory");
                    }
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) {
                        const uint32_t acc = (ks | kb) != 0;
                        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                                     "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
                                     "[%0], %1, %2, %3, [%4], [%5], p;\n\t}"
                                     :: "r"(tmem), "l"(desc_sw128(a0 + 32 * kb)), "l"(desc_sw128(b0 + 32 * kb)),
                                        "r"(kIdesc), "r"(sf_col + 4 * kb), "r"(sf_col + 16 + 8 * kb), "r"(acc)
                                     : "memory");
                    }
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                                 :: "r"(smem_u32(&empty_bar[s])) : "memory");
                }
                if (!ok) break;
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                             :: "r"(smem_u32(&acc_full)) : "memory");
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                          // TMEM lane quadrant of this warp
        const int r = q * 32 + lane;                     // tile row of this thread
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        int tl = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++tl) {
            const TileInfo ti = tile_info(g, tile0 + tile);
            if (!mbar_wait(&acc_full, (uint32_t)tl & 1u, &abort_flag)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const bool valid = r < ti.rows;
            const int p = ti.m0 + r;
            const int route = valid ? g.perm[p] : 0;
            const uint8_t* rec = g.slot_buf + (size_t)(g.slot_of ? g.slot_of[ti.e] : g.slot0 + ti.e) * g.rec_bytes;
            const float ts = *reinterpret_cast<const float*>(rec + g.off_tscale);
            if (g.kind == 1) {
                for (int c = 0; c < 128; c += 16) {
                    float gv[16], uv[16], hv[16];
                    tmem_ld16(lane_addr + c, gv);
                    tmem_ld16(lane_addr + 128 + c, uv);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float gg = gv[j] * ts, uu = uv[j] * ts;
                        hv[j] = gg / (1.f + expf(-gg)) * uu;
                    }
                    uint32_t lo, hi;
                    const uint8_t sc = quant_block16(hv, lo, hi);
                    if (valid) {
                        const int col = ti.nt * 128 + c;
                        *reinterpret_cast<uint2*>(g.h_codes + (size_t)p * (g.I / 2) + col / 2) = make_uint2(lo, hi);
                        g.h_scales[(size_t)p * (g.I / 16) + col / 16] = sc;
                        if (g.debug_h) {
                            *reinterpret_cast<uint2*>(g.debug_h + (size_t)route * (g.I / 2) + col / 2) = make_uint2(lo, hi);
                            g.debug_h[(size_t)g.R_total * (g.I / 2) + (size_t)route * (g.I / 16) + col / 16] = sc;
                        }
                    }
                }
            } else {
                const float mul = valid ? ts * g.w[route] : 0.f;
                float* orow = g.O + (size_t)route * g.H + ti.nt * kBN;
                for (int c = 0; c < kBN; c += 16) {
                    float v[16];
                    tmem_ld16(lane_addr + c, v);
                    if (valid) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4*>(orow + c + j) =
                                make_float4(v[j] * mul, v[j + 1] * mul, v[j + 2] * mul, v[j + 3] * mul);
                    }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(&acc_empty);
        }
    }

    __syncthreads();
    if (abort_flag && threadIdx.x == 0) atomicOr(g.status, FT_DEV_TIMEOUT);
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled encode_fn() {
    static PFN_encodeTiled fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_encodeTiled>(p);
    }
    return fn;
}

// 2D uint8 map [rows, row_bytes], box 128 x 128 bytes, 128B swizzle.
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows) {
    PFN_encodeTiled f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {128, 128};
    const cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D uint8 map [slots, rows, row_bytes] with slot stride rec_bytes, box 128 bytes x box_rows x 1.
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
                 uint64_t rec_bytes, uint32_t box_rows) {
    PFN_encodeTiled f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[3] = {row_bytes, rows, slots};
    const cuuint64_t strides[2] = {row_bytes, rec_bytes};
    const cuuint32_t box[3] = {128, box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t umma_smem_bytes() { return (size_t)kStages * kStageBytes + 1024; }

cudaError_t launch_umma(const CUtensorMap& a, const CUtensorMap& b, const UmmaArgs& g, int grid,
                        cudaStream_t s) {
    // the shared-memory attribute is per device; set it once on each
    static std::atomic<bool> attr[kMaxDevices];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr[dev].load(std::memory_order_relaxed)) {
            e = cudaFuncSetAttribute(umma_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)umma_smem_bytes());
            if (e != cudaSuccess) return e;
            attr[dev].store(true, std::memory_order_release);
        }
    }
    umma_gemm_kernel<<<grid, kThreads, umma_smem_bytes(), s>>>(a, b, g);
    return cudaGetLastError();
}

}  // namespace ft
