// The host share of decode: a persistent pool of worker threads, each pinned to one
// CPU core, that computes the routes a decode call leaves to the host straight from
// the pinned pool, and the mailbox dispatcher that takes those calls from the decode
// kernel while the GPU computes its own share.
//
// [EXPLAINER §8.3] a persistent C++ worker pool pinned to physical cores; the CPU
//   expert kernel is SIMD and dequantises inside the kernel, never into a full
//   precision copy of the expert;
// [EXPLAINER §6.2, §6.9] the host computes the set C of misses; each route is
//   computed once, so y = y_gpu + y_cpu;
// [BWRATIO "代码全链路" §2] the host side receives -1 for every route the GPU
//   keeps, and the two partials are added.
//
// Arithmetic (the same on every host): x (bf16) is rounded to f16 after a per-token
// power-of-two prescale that keeps |x| < 2^15 (exact for bf16 values in the f16 normal
// range); E2M1 codes and block scales (E4M3, or E8M0 for MXFP4 records) are exact in
// f16 / fp32; a row is a sum over 16-element groups: lane j of a group accumulates
// elements j, 4+j, 8+j, 12+j with fused multiply-adds of exact products starting from
// zero, the group partial is (l0 + l1) + (l2 + l3) and enters the row sum through one
// fused multiply-add with the group's scale.  On aarch64 the gate/up rows use the f16
// widening multiply-add (FMLAL) and the down rows fp32 NEON; elsewhere the same
// operations run one element at a time.  Then g, u = row * s_gu * prescale,
// h = silu(g) * u, o = (W_d h) * s_d, y[b] += w * o with the units in ascending flat id.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include <pthread.h>
#include <sched.h>

#if defined(__aarch64__)
#include <arm_neon.h>
#endif
#if defined(__aarch64__) && defined(__ARM_FEATURE_FP16_FML)
#define FT_HOST_FMLAL 1
#endif

#include "../../include/ft.h"
#include "ft_host.h"
#include "ft_record.h"

namespace ft {
namespace {

// The value of each E2M1 code (sign in bit 3), and the high byte of its f16 encoding
// (every E2M1 value has a zero low byte in f16).
constexpr float kE2M1[16] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f,
                             -0.f, -0.5f, -1.f, -1.5f, -2.f, -3.f, -4.f, -6.f};
alignas(16) constexpr uint8_t kE2M1f16hi[16] = {0x00, 0x38, 0x3C, 0x3E, 0x40, 0x42, 0x44, 0x46,
                                                0x80, 0xB8, 0xBC, 0xBE, 0xC0, 0xC2, 0xC4, 0xC6};

// The value of each E4M3 code (sign bit 7, exponent bits 6..3 with bias 7, mantissa
// bits 2..0; exponent 0 is subnormal; 0x7F / 0xFF are NaN) and of each E8M0 code
// (2^(c - 127); 0xFF is NaN).
struct ScaleTables {
    float e4m3[256];
    float e8m0[256];
    ScaleTables() {
        for (int c = 0; c < 256; ++c) {
            const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
            float v = e == 0 ? std::ldexp((float)m / 8.f, -6) : std::ldexp(1.f + (float)m / 8.f, e - 7);
            if ((c & 127) == 127) v = NAN;
            e4m3[c] = s ? -v : v;
            e8m0[c] = c == 255 ? NAN : std::ldexp(1.f, c - 127);
        }
    }
};
const ScaleTables& tables() {
    static const ScaleTables t;
    return t;
}

// f16 encoding of a float, round to nearest even (the sign kept; values past the f16
// range become infinity, values below half the smallest subnormal zero).
uint16_t f16_bits(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    const uint32_t sign = (u >> 16) & 0x8000u;
    const uint32_t a = u & 0x7FFFFFFFu;
    if (a >= 0x7F800000u) return (uint16_t)(sign | 0x7C00u | (a > 0x7F800000u ? 0x200u : 0u));
    const int e = (int)(a >> 23) - 127;                       // unbiased exponent
    if (e > 15) return (uint16_t)(sign | 0x7C00u);
    uint32_t mant, base;
    int shift;                                                 // low bits dropped
    if (e >= -14) {                                            // normal: 10 of 23 bits kept
        mant = a & 0x7FFFFFu;
        base = (uint32_t)(e + 15) << 10;
        shift = 13;
    } else {                                                   // subnormal: units of 2^-24
        mant = (a & 0x7FFFFFu) | 0x800000u;
        base = 0;
        shift = -e - 1;
        if (shift > 24) return (uint16_t)sign;
    }
    const uint32_t q = mant >> shift;
    const uint32_t rem = mant & ((1u << shift) - 1u), half = 1u << (shift - 1);
    uint32_t r = base + q;
    if (rem > half || (rem == half && (q & 1u))) r += 1;       // a carry moves into the exponent
    return (uint16_t)(sign | r);
}

float f16_value(uint16_t h) {
    const uint32_t e = (h >> 10) & 31, m = h & 1023;
    float v = e == 0 ? std::ldexp((float)m, -24) : std::ldexp((float)(m | 1024), (int)e - 25);
    if (e == 31) v = m ? NAN : INFINITY;
    return (h & 0x8000) ? -v : v;
}

inline float group_sum(const float* a) { return (a[0] + a[1]) + (a[2] + a[3]); }

// out[t] = sum over the K elements of one row of code * v[t][k] * scale, for NT
// vectors of fp32 values (the down rows; also the gate/up rows where FMLAL is absent).
template <int NT>
void row_dot(const uint8_t* codes, const uint8_t* scales, int K, bool mx, const float* const* v, float* out) {
    const float* sct = mx ? tables().e8m0 : tables().e4m3;
    float row[NT];
    for (int t = 0; t < NT; ++t) row[t] = 0.f;
    const int ng = K / 16;
#if defined(__aarch64__)
    const uint8x16_t tab = vld1q_u8(kE2M1f16hi);
    const uint8x8_t m15 = vdup_n_u8(15);
    const uint8x16_t zero = vdupq_n_u8(0);
    for (int gi = 0; gi < ng; ++gi) {
        const float sc = sct[scales[mx ? gi >> 1 : gi]];
        const uint8x8_t b = vld1_u8(codes + 8 * gi);
        const uint8x8x2_t z = vzip_u8(vand_u8(b, m15), vshr_n_u8(b, 4));
        const uint8x16_t hi = vqtbl1q_u8(tab, vcombine_u8(z.val[0], z.val[1]));
        const float16x8_t h0 = vreinterpretq_f16_u8(vzip1q_u8(zero, hi));
        const float16x8_t h1 = vreinterpretq_f16_u8(vzip2q_u8(zero, hi));
        const float32x4_t c0 = vcvt_f32_f16(vget_low_f16(h0)), c1 = vcvt_high_f32_f16(h0);
        const float32x4_t c2 = vcvt_f32_f16(vget_low_f16(h1)), c3 = vcvt_high_f32_f16(h1);
        for (int t = 0; t < NT; ++t) {
            const float* xv = v[t] + 16 * gi;
            float32x4_t a = vfmaq_f32(vdupq_n_f32(0.f), c0, vld1q_f32(xv));
            a = vfmaq_f32(a, c1, vld1q_f32(xv + 4));
            a = vfmaq_f32(a, c2, vld1q_f32(xv + 8));
            a = vfmaq_f32(a, c3, vld1q_f32(xv + 12));
            const float32x2_t s2 = vpadd_f32(vget_low_f32(a), vget_high_f32(a));
            row[t] = std::fma(vget_lane_f32(s2, 0) + vget_lane_f32(s2, 1), sc, row[t]);
        }
    }
#else
    for (int gi = 0; gi < ng; ++gi) {
        const float sc = sct[scales[mx ? gi >> 1 : gi]];
        float c[16];
        for (int i = 0; i < 8; ++i) {
            const uint8_t b = codes[8 * gi + i];
            c[2 * i] = kE2M1[b & 15];
            c[2 * i + 1] = kE2M1[b >> 4];
        }
        for (int t = 0; t < NT; ++t) {
            const float* xv = v[t] + 16 * gi;
            float a[4] = {0.f, 0.f, 0.f, 0.f};
            for (int q = 0; q < 4; ++q)
                for (int j = 0; j < 4; ++j) a[j] = std::fma(c[4 * q + j], xv[4 * q + j], a[j]);
            row[t] = std::fma(group_sum(a), sc, row[t]);
        }
    }
#endif
    for (int t = 0; t < NT; ++t) out[t] = row[t];
}

#if defined(FT_HOST_FMLAL)
// The same sums for NT vectors of f16 values (the gate/up rows): FMLAL multiplies f16
// pairs exactly and adds them into fp32 lanes with one rounding, in the lane order
// above.
template <int NT>
void row_dot_h(const uint8_t* codes, const uint8_t* scales, int K, bool mx, const uint16_t* const* v, float* out) {
    const float* sct = mx ? tables().e8m0 : tables().e4m3;
    float row[NT];
    for (int t = 0; t < NT; ++t) row[t] = 0.f;
    const int ng = K / 16;
    const uint8x16_t tab = vld1q_u8(kE2M1f16hi);
    const uint8x8_t m15 = vdup_n_u8(15);
    const uint8x16_t zero = vdupq_n_u8(0);
    for (int gi = 0; gi < ng; ++gi) {
        const float sc = sct[scales[mx ? gi >> 1 : gi]];
        const uint8x8_t b = vld1_u8(codes + 8 * gi);
        const uint8x8x2_t z = vzip_u8(vand_u8(b, m15), vshr_n_u8(b, 4));
        const uint8x16_t hi = vqtbl1q_u8(tab, vcombine_u8(z.val[0], z.val[1]));
        const float16x8_t h0 = vreinterpretq_f16_u8(vzip1q_u8(zero, hi));
        const float16x8_t h1 = vreinterpretq_f16_u8(vzip2q_u8(zero, hi));
        for (int t = 0; t < NT; ++t) {
            const float16x8_t x0 = vreinterpretq_f16_u16(vld1q_u16(v[t] + 16 * gi));
            const float16x8_t x1 = vreinterpretq_f16_u16(vld1q_u16(v[t] + 16 * gi + 8));
            float32x4_t a = vfmlalq_low_f16(vdupq_n_f32(0.f), h0, x0);
            a = vfmlalq_high_f16(a, h0, x0);
            a = vfmlalq_low_f16(a, h1, x1);
            a = vfmlalq_high_f16(a, h1, x1);
            const float32x2_t s2 = vpadd_f32(vget_low_f32(a), vget_high_f32(a));
            row[t] = std::fma(vget_lane_f32(s2, 0) + vget_lane_f32(s2, 1), sc, row[t]);
        }
    }
    for (int t = 0; t < NT; ++t) out[t] = row[t];
}
#endif

// Any number of vectors, in groups of up to four.
void row_dot_n(const uint8_t* codes, const uint8_t* scales, int K, bool mx, const float* const* v, int n,
               float* out) {
    for (int t0 = 0; t0 < n; t0 += 4) {
        switch (std::min(4, n - t0)) {
            case 1: row_dot<1>(codes, scales, K, mx, v + t0, out + t0); break;
            case 2: row_dot<2>(codes, scales, K, mx, v + t0, out + t0); break;
            case 3: row_dot<3>(codes, scales, K, mx, v + t0, out + t0); break;
            default: row_dot<4>(codes, scales, K, mx, v + t0, out + t0); break;
        }
    }
}

// The gate/up rows: x as f16 (vh) or as the fp32 values of the same f16 numbers (vf).
void row_dot_x(const uint8_t* codes, const uint8_t* scales, int K, bool mx, const uint16_t* const* vh,
               const float* const* vf, int n, float* out) {
#if defined(FT_HOST_FMLAL)
    (void)vf;
    for (int t0 = 0; t0 < n; t0 += 4) {
        switch (std::min(4, n - t0)) {
            case 1: row_dot_h<1>(codes, scales, K, mx, vh + t0, out + t0); break;
            case 2: row_dot_h<2>(codes, scales, K, mx, vh + t0, out + t0); break;
            case 3: row_dot_h<3>(codes, scales, K, mx, vh + t0, out + t0); break;
            default: row_dot_h<4>(codes, scales, K, mx, vh + t0, out + t0); break;
        }
    }
#else
    (void)vh;
    row_dot_n(codes, scales, K, mx, vf, n, out);
#endif
}

inline float bf16_to_float(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

constexpr int kChunk = 32;   // rows of one work item

// One expert of the host share: its flat id and its tokens with their summed gates.
struct Unit {
    int flat;
    int ntok;
    int pair0;                 // first h row of the unit
    int tok[32];
    float w[32];
};

}  // namespace
}  // namespace ft

struct ft_host_branch {
    // configuration
    int L, E, H, I, k_max, B_max, format;
    ft::RecordLayout rl;
    const uint8_t* pool;
    uint8_t* mailbox;
    ft::MailboxLayout ml;
    int nthreads;
    std::vector<int> cpus;
    // workers
    std::vector<std::thread> th;
    std::atomic<uint32_t> gen{0};
    std::atomic<bool> stop{false};
    std::mutex job_mu;
    // the current job
    std::vector<ft::Unit> units;
    int n_pairs = 0;
    int B = 0;
    std::vector<float> xf;     // [B_max, H] x / xmul rounded to f16, as fp32
    std::vector<uint16_t> xh;  // the same numbers as f16
    float xmul[32];            // per-token power-of-two prescale
    std::vector<float> h;      // [pairs, I]
    float* y = nullptr;        // [B, H]
    int n1 = 0, n2 = 0;
    std::atomic<int> next1{0}, done1{0}, next2{0}, done2{0}, finished{0};
    std::atomic<uint64_t> jobs{0}, mailbox_jobs{0};

    // --------------------------------------------------------------- work items
    // Phase 1 item: kChunk gate/up row pairs of one unit -> h rows of its tokens.
    void gate_up_item(int i) {
        const int per = I / ft::kChunk;
        const ft::Unit& u = units[i / per];
        const int p0 = (i % per) * ft::kChunk;
        const uint8_t* rec = pool + (size_t)u.flat * rl.bytes;
        const int sb = ft::scale_block(format);
        const bool mx = format == FT_FORMAT_MXFP4;
        float s_gu;
        std::memcpy(&s_gu, rec + rl.s_gu, 4);
        const float* xv[32];
        const uint16_t* xhv[32];
        for (int t = 0; t < u.ntok; ++t) {
            xv[t] = xf.data() + (size_t)u.tok[t] * H;
            xhv[t] = xh.data() + (size_t)u.tok[t] * H;
        }
        float g[32], uu[32];
        for (int p = p0; p < p0 + ft::kChunk; ++p) {
            ft::row_dot_x(rec + rl.gu_codes + (size_t)p * (H / 2), rec + rl.gu_scales + (size_t)p * (H / sb), H,
                          mx, xhv, xv, u.ntok, g);
            ft::row_dot_x(rec + rl.gu_codes + (size_t)(I + p) * (H / 2),
                          rec + rl.gu_scales + (size_t)(I + p) * (H / sb), H, mx, xhv, xv, u.ntok, uu);
            for (int t = 0; t < u.ntok; ++t) {
                const float xm = xmul[u.tok[t]];
                const float gv = g[t] * s_gu * xm, uv = uu[t] * s_gu * xm;
                h[(size_t)(u.pair0 + t) * I + p] = gv / (1.f + std::exp(-gv)) * uv;
            }
        }
    }
    // Phase 2 item: kChunk output rows, every unit in ascending flat id.
    void down_item(int i) {
        const int r0 = i * ft::kChunk;
        const int sb = ft::scale_block(format);
        const bool mx = format == FT_FORMAT_MXFP4;
        for (const ft::Unit& u : units) {
            const uint8_t* rec = pool + (size_t)u.flat * rl.bytes;
            float s_d;
            std::memcpy(&s_d, rec + rl.s_d, 4);
            const float* hv[32];
            for (int t = 0; t < u.ntok; ++t) hv[t] = h.data() + (size_t)(u.pair0 + t) * I;
            float o[32];
            for (int r = r0; r < r0 + ft::kChunk; ++r) {
                ft::row_dot_n(rec + rl.d_codes + (size_t)r * (I / 2), rec + rl.d_scales + (size_t)r * (I / sb), I,
                              mx, hv, u.ntok, o);
                for (int t = 0; t < u.ntok; ++t) y[(size_t)u.tok[t] * H + r] += u.w[t] * (o[t] * s_d);
            }
        }
    }
    void work() {
        for (int i; (i = next1.fetch_add(1, std::memory_order_relaxed)) < n1;) {
            gate_up_item(i);
            done1.fetch_add(1, std::memory_order_release);
        }
        while (done1.load(std::memory_order_acquire) < n1) std::this_thread::yield();
        for (int i; (i = next2.fetch_add(1, std::memory_order_relaxed)) < n2;) {
            down_item(i);
            done2.fetch_add(1, std::memory_order_release);
        }
    }

    // --------------------------------------------------------------- jobs
    // The units of a host share: unique flat ids ascending; per unit its tokens
    // ascending with the sum of their gates to it.
    bool set_units(const int32_t* deferred, const float* w, int B_, int k) {
        units.clear();
        std::vector<std::pair<int, int>> fr;   // (flat, route)
        for (int r = 0; r < B_ * k; ++r)
            if (deferred[r] >= 0 && deferred[r] < L * E) fr.push_back({deferred[r], r});
        std::sort(fr.begin(), fr.end());
        n_pairs = 0;
        for (size_t i = 0; i < fr.size();) {
            ft::Unit u;
            u.flat = fr[i].first;
            u.ntok = 0;
            u.pair0 = n_pairs;
            for (; i < fr.size() && fr[i].first == u.flat; ++i) {
                const int b = fr[i].second / k;
                if (u.ntok > 0 && u.tok[u.ntok - 1] == b) {
                    u.w[u.ntok - 1] += w[fr[i].second];
                } else {
                    if (u.ntok == 32) return false;
                    u.tok[u.ntok] = b;
                    u.w[u.ntok] = w[fr[i].second];
                    ++u.ntok;
                }
            }
            n_pairs += u.ntok;
            units.push_back(u);
        }
        if ((size_t)n_pairs * I > h.size()) h.resize((size_t)n_pairs * I);
        return true;
    }
    // Runs the job set up in units / xf / y with every worker; `helpers` workers take
    // part besides the caller.  Returns when every item is done and every helper left.
    void run(int helpers) {
        n1 = (int)units.size() * (I / ft::kChunk);
        n2 = units.empty() ? 0 : H / ft::kChunk;
        next1.store(0, std::memory_order_relaxed);
        done1.store(0, std::memory_order_relaxed);
        next2.store(0, std::memory_order_relaxed);
        done2.store(0, std::memory_order_relaxed);
        finished.store(0, std::memory_order_relaxed);
        gen.fetch_add(1, std::memory_order_release);
        work();
        while (done2.load(std::memory_order_acquire) < n2 || finished.load(std::memory_order_acquire) < helpers)
            std::this_thread::yield();
        jobs.fetch_add(1, std::memory_order_relaxed);
    }
    // x of the job's tokens: per token a power of two 2^k (k = 0 unless |x| reaches 2^15)
    // and x / 2^k rounded to f16.
    void load_x(const uint16_t* x, int B_) {
        for (int b = 0; b < B_; ++b) {
            float amax = 0.f;
            for (int i = 0; i < H; ++i) amax = std::max(amax, std::fabs(ft::bf16_to_float(x[(size_t)b * H + i])));
            const int k = amax >= 32768.f ? std::ilogb(amax) - 14 : 0;
            xmul[b] = std::ldexp(1.f, k);
            for (int i = 0; i < H; ++i) {
                const size_t j = (size_t)b * H + i;
                xh[j] = ft::f16_bits(std::ldexp(ft::bf16_to_float(x[j]), -k));
                xf[j] = ft::f16_value(xh[j]);
            }
        }
    }
    ft::MailboxHeader* header() { return reinterpret_cast<ft::MailboxHeader*>(mailbox); }
    // A call published by the decode kernel: compute it into the mailbox's y, then
    // raise done.  Worker 0 runs this; the other workers help.
    void mailbox_job() {
        ft::MailboxHeader* hd = header();
        const int B_ = hd->B, k = hd->k;
        B = B_;
        y = reinterpret_cast<float*>(mailbox + ml.y);
        std::memset(y, 0, (size_t)B_ * H * 4);
        if (B_ >= 1 && B_ <= B_max && k >= 1 && k <= k_max &&
            set_units(reinterpret_cast<const int32_t*>(mailbox + ml.def),
                      reinterpret_cast<const float*>(mailbox + ml.w), B_, k)) {
            load_x(reinterpret_cast<const uint16_t*>(mailbox + ml.x), B_);
            run(nthreads - 1);
        }
        mailbox_jobs.fetch_add(1, std::memory_order_relaxed);
        __atomic_store_n(&hd->done, 1u, __ATOMIC_RELEASE);
    }

    // --------------------------------------------------------------- workers
    void worker(int w) {
        if (w < (int)cpus.size() && cpus[w] >= 0) {
            cpu_set_t set;
            CPU_ZERO(&set);
            CPU_SET(cpus[w], &set);
            pthread_setaffinity_np(pthread_self(), sizeof(set), &set);
        }
        uint32_t seen = 0;                       // gen starts at 0, before any worker runs
        unsigned spins = 0;
        auto idle_since = std::chrono::steady_clock::now();
        while (!stop.load(std::memory_order_relaxed)) {
            // (the mailbox lives in memory the GPU writes: read it every 8th round only)
            if (w == 0 && mailbox && (spins & 7u) == 0 && __atomic_load_n(&header()->task, __ATOMIC_ACQUIRE) == 1u) {
                std::unique_lock<std::mutex> lk(job_mu, std::try_to_lock);
                if (lk.owns_lock()) {
                    __atomic_store_n(&header()->task, 0u, __ATOMIC_RELAXED);
                    mailbox_job();
                    seen = gen.load(std::memory_order_acquire);
                    spins = 0;
                    idle_since = std::chrono::steady_clock::now();
                    continue;
                }
            }
            const uint32_t g = gen.load(std::memory_order_acquire);
            if (g != seen) {
                seen = g;
                work();
                finished.fetch_add(1, std::memory_order_release);
                spins = 0;
                idle_since = std::chrono::steady_clock::now();
                continue;
            }
            // hot spin first (decode calls come every few tens of microseconds), then
            // yield, then short sleeps once idle for a while
            if (++spins < 4096) continue;
            if ((spins & 1023u) == 0 &&
                std::chrono::steady_clock::now() - idle_since > std::chrono::milliseconds(20))
                std::this_thread::sleep_for(std::chrono::microseconds(20));
            else
                std::this_thread::yield();
        }
    }
};

namespace ft {

bool host_branch_info(const ft_host_branch* hb, HostBranchInfo* out) {
    if (!hb || !out) return false;
    out->L = hb->L;
    out->E = hb->E;
    out->H = hb->H;
    out->I = hb->I;
    out->k_max = hb->k_max;
    out->B_max = hb->B_max;
    out->format = hb->format;
    out->pool = hb->pool;
    out->mailbox = hb->mailbox;
    return true;
}

double host_branch_run_flats(ft_host_branch* hb, const int32_t* flats, int n) {
    std::lock_guard<std::mutex> lk(hb->job_mu);
    std::vector<int32_t> def(flats, flats + n);
    std::vector<float> w(n, 1.f);
    std::vector<float> y((size_t)hb->H);
    std::vector<uint16_t> x((size_t)hb->H, 0x3F80);   // bf16 1.0
    const auto t0 = std::chrono::steady_clock::now();
    hb->B = 1;
    hb->y = y.data();
    if (!hb->set_units(def.data(), w.data(), 1, n)) return -1.0;
    hb->load_x(x.data(), 1);
    hb->run(hb->nthreads);
    return std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
}

}  // namespace ft

extern "C" {

ft_status ft_host_mailbox_bytes(int32_t H, int32_t k_max, int32_t B_max, size_t* bytes) {
    if (!bytes || H < 64 || H % 64 || k_max < 1 || k_max > 32 || B_max < 1 || B_max > 32) return FT_ERR_ARG;
    *bytes = ft::mailbox_layout(H, k_max, B_max).bytes;
    return FT_OK;
}

ft_status ft_host_branch_create(const ft_host_desc* d, ft_host_branch** out) {
    if (!d || !out) return FT_ERR_ARG;
    *out = nullptr;
    if (d->L < 1 || d->E < 1 || d->E > 4096 || d->H < 64 || d->H % 64 || d->I < 32 || d->I % 32 ||
        d->k_max < 1 || d->k_max > 32 || d->B_max < 1 || d->B_max > 32 || !d->host_pool ||
        d->n_threads < 1 || d->n_threads > 1024 ||
        (d->format != FT_FORMAT_NVFP4 && d->format != FT_FORMAT_MXFP4))
        return FT_ERR_ARG;
    if (d->mailbox && (reinterpret_cast<uintptr_t>(d->mailbox) & 255)) return FT_ERR_ARG;
    std::vector<int> cpus;
    if (d->cpus) {
        cpus.assign(d->cpus, d->cpus + d->n_threads);
    } else {
        cpu_set_t set;
        CPU_ZERO(&set);
        if (sched_getaffinity(0, sizeof(set), &set) == 0)
            for (int c = 0; c < CPU_SETSIZE && (int)cpus.size() < d->n_threads; ++c)
                if (CPU_ISSET(c, &set)) cpus.push_back(c);
    }
    ft_host_branch* hb = new (std::nothrow) ft_host_branch();
    if (!hb) return FT_ERR_ARG;
    hb->L = d->L;
    hb->E = d->E;
    hb->H = d->H;
    hb->I = d->I;
    hb->k_max = d->k_max;
    hb->B_max = d->B_max;
    hb->format = d->format;
    hb->rl = ft::record_layout(d->H, d->I, d->format);
    hb->pool = static_cast<const uint8_t*>(d->host_pool);
    hb->mailbox = static_cast<uint8_t*>(d->mailbox);
    hb->ml = ft::mailbox_layout(d->H, d->k_max, d->B_max);
    hb->nthreads = d->n_threads;
    hb->cpus = cpus;
    hb->xf.resize((size_t)d->B_max * d->H);
    hb->xh.resize((size_t)d->B_max * d->H);
    hb->h.resize((size_t)(d->B_max * d->k_max) * d->I);
    if (hb->mailbox) {
        ft::MailboxHeader* hd = hb->header();
        __atomic_store_n(&hd->task, 0u, __ATOMIC_RELAXED);
        __atomic_store_n(&hd->done, 0u, __ATOMIC_RELAXED);
        hd->n_def = 0;
    }
    for (int w = 0; w < d->n_threads; ++w) hb->th.emplace_back(&ft_host_branch::worker, hb, w);
    *out = hb;
    return FT_OK;
}

void ft_host_branch_destroy(ft_host_branch* hb) {
    if (!hb) return;
    hb->stop.store(true);
    for (auto& t : hb->th) t.join();
    delete hb;
}

ft_status ft_host_moe(ft_host_branch* hb, const void* x, const int32_t* deferred, const float* w, int32_t B,
                      int32_t k, float* y) {
    if (!hb || !x || !deferred || !w || !y || B < 1 || B > hb->B_max || k < 1 || k > hb->k_max) return FT_ERR_ARG;
    std::lock_guard<std::mutex> lk(hb->job_mu);
    hb->B = B;
    hb->y = y;
    std::memset(y, 0, (size_t)B * hb->H * 4);
    if (!hb->set_units(deferred, w, B, k)) return FT_ERR_ARG;
    hb->load_x(static_cast<const uint16_t*>(x), B);
    hb->run(hb->nthreads);
    return FT_OK;
}

ft_status ft_host_branch_stats(const ft_host_branch* hb, int64_t* jobs, int64_t* mailbox_jobs) {
    if (!hb) return FT_ERR_ARG;
    if (jobs) *jobs = (int64_t)hb->jobs.load();
    if (mailbox_jobs) *mailbox_jobs = (int64_t)hb->mailbox_jobs.load();
    return FT_OK;
}

}  // extern "C"
