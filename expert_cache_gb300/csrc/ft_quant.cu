// NVFP4 encoders and the expert-record quantiser (pool builder).
//
// Record layout: [EXPLAINER §8.4] (one flat id names a whole expert across banks);
// here the banks of one flat id are contiguous so a fill is one copy.
// Quantiser (fp32 IEEE steps, explicit _rn intrinsics so no FMA contraction):
//   s_t = amax(W) / 2688;  scale = E4M3_RNE((amax16 / 6) / s_t);
//   code = E2M1_RNE_sat(w / (scale * s_t));  a zero scale gives a zero block.
#include "ft_quant.cuh"

namespace ft {

// One CTA per matrix: amax over the matrix, s_t written into the record tail.
__global__ void __launch_bounds__(1024) tensor_scale_kernel(const float* w_gu, const float* w_d,
                                                            int H, int I, uint8_t* records,
                                                            size_t rec_bytes, size_t off_s_gu,
                                                            size_t off_s_d) {
    const int n = blockIdx.x >> 1, which = blockIdx.x & 1;
    const size_t count = (size_t)2 * I * H / (which ? 2 : 1);   // W_gu: 2IH, W_d: HI
    const float* src = which ? w_d + (size_t)n * H * I : w_gu + (size_t)n * 2 * I * H;
    float m = 0.f;
    const float4* s4 = reinterpret_cast<const float4*>(src);
    for (size_t i = threadIdx.x; i < count / 4; i += blockDim.x) {
        const float4 v = s4[i];
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    __shared__ float red[32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (threadIdx.x == 0) {
            const float st = __fdiv_rn(m, 2688.0f);
            *reinterpret_cast<float*>(records + (size_t)n * rec_bytes +
                                      (which ? off_s_d : off_s_gu)) = st;
        }
    }
}

// One thread per 16-element block of every matrix.
__global__ void block_quant_kernel(const float* w_gu, const float* w_d, int n_exp, int H, int I,
                                   uint8_t* records, size_t rec_bytes, RecordOffsets off) {
    const size_t blocks_gu = (size_t)2 * I * H / 16, blocks_d = (size_t)H * I / 16;
    const size_t per = blocks_gu + blocks_d;
    const size_t total = per * n_exp;
    for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
         g += (size_t)gridDim.x * blockDim.x) {
        const size_t n = g / per, bi = g % per;
        uint8_t* rec = records + n * rec_bytes;
        const float* src;
        uint8_t* codes;
        uint8_t* scale;
        float st;
        if (bi < blocks_gu) {
            src = w_gu + (size_t)n * 2 * I * H + bi * 16;
            codes = rec + off.gu_codes + bi * 8;
            scale = rec + off.gu_scales + bi;
            st = *reinterpret_cast<const float*>(rec + off.s_gu);
        } else {
            const size_t b = bi - blocks_gu;
            src = w_d + (size_t)n * H * I + b * 16;
            codes = rec + off.d_codes + b * 8;
            scale = rec + off.d_scales + b;
            st = *reinterpret_cast<const float*>(rec + off.s_d);
        }
        float v[16];
        const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 t = s4[j];
            v[4 * j] = t.x; v[4 * j + 1] = t.y; v[4 * j + 2] = t.z; v[4 * j + 3] = t.w;
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
        uint8_t sc = 0;
        float denom = 0.f;
        if (st != 0.f) {
            sc = e4m3_encode_rne(__fdiv_rn(__fdiv_rn(amax, 6.0f), st));
            denom = __fmul_rn(e4m3_value(sc), st);
        }
        uint32_t lo = 0, hi = 0;
        if (denom != 0.f) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                lo |= (uint32_t)e2m1_encode_rne(__fdiv_rn(v[j], denom)) << (4 * j);
                hi |= (uint32_t)e2m1_encode_rne(__fdiv_rn(v[8 + j], denom)) << (4 * j);
            }
        }
        *reinterpret_cast<uint2*>(codes) = make_uint2(lo, hi);
        *scale = sc;
    }
}

// MXFP4: one thread per 32-element block of every matrix (the microscaling
// conversion rule; fp32 IEEE steps): shared = floor(log2(amax)) - 2 clamped to
// [-127, 127] (amax 0: -127); code = E2M1_RNE_sat(v * 2^-shared).
__global__ void block_quant_mx_kernel(const float* w_gu, const float* w_d, int n_exp, int H, int I,
                                      uint8_t* records, size_t rec_bytes, RecordOffsets off) {
    const size_t blocks_gu = (size_t)2 * I * H / 32, blocks_d = (size_t)H * I / 32;
    const size_t per = blocks_gu + blocks_d;
    const size_t total = per * n_exp;
    for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
         g += (size_t)gridDim.x * blockDim.x) {
        const size_t n = g / per, bi = g % per;
        uint8_t* rec = records + n * rec_bytes;
        const float* src;
        uint8_t* codes;
        uint8_t* scale;
        if (bi < blocks_gu) {
            src = w_gu + (size_t)n * 2 * I * H + bi * 32;
            codes = rec + off.gu_codes + bi * 16;
            scale = rec + off.gu_scales + bi;
        } else {
            const size_t b = bi - blocks_gu;
            src = w_d + (size_t)n * H * I + b * 32;
            codes = rec + off.d_codes + b * 16;
            scale = rec + off.d_scales + b;
        }
        float v[32];
        const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 t = s4[j];
            v[4 * j] = t.x; v[4 * j + 1] = t.y; v[4 * j + 2] = t.z; v[4 * j + 3] = t.w;
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
        int shared = -127;
        if (amax > 0.f) {
            const uint32_t b = __float_as_uint(amax);
            const int ef = (int)(b >> 23);
            // floor(log2(amax)): the exponent of a normal number, or the position of the
            // leading mantissa bit of a subnormal one
            const int fl = ef ? ef - 127 : (31 - __clz((int)(b & 0x7FFFFFu))) - 149;
            shared = max(-127, min(127, fl - 2));
        }
        const int mexp = 127 - shared;                     // 2^-shared as fp32 bits
        const float mul = __uint_as_float(mexp ? (uint32_t)mexp << 23 : 0x00400000u);
        uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 32; ++j)
            w[j >> 3] |= (uint32_t)e2m1_encode_rne(__fmul_rn(v[j], mul)) << (4 * (j & 7));
        *reinterpret_cast<uint4*>(codes) = make_uint4(w[0], w[1], w[2], w[3]);
        *scale = (uint8_t)(shared + 127);
    }
}

__global__ void unit_tensor_scales_kernel(uint8_t* records, size_t rec_bytes, size_t off_s_gu, size_t off_s_d,
                                          int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        *reinterpret_cast<float*>(records + (size_t)i * rec_bytes + off_s_gu) = 1.0f;
        *reinterpret_cast<float*>(records + (size_t)i * rec_bytes + off_s_d) = 1.0f;
    }
}

cudaError_t launch_quantize_mx(const float* w_gu, const float* w_d, int n, int H, int I,
                               uint8_t* records, size_t rec_bytes, cudaStream_t s) {
    const RecordLayout r = record_layout(H, I, FT_FORMAT_MXFP4);
    RecordOffsets off{r.gu_codes, r.gu_scales, r.d_codes, r.d_scales, r.s_gu, r.s_d};
    cudaMemsetAsync(records, 0, (size_t)n * rec_bytes, s);
    unit_tensor_scales_kernel<<<(n + 255) / 256, 256, 0, s>>>(records, rec_bytes, r.s_gu, r.s_d, n);
    const size_t total = ((size_t)2 * I * H / 32 + (size_t)H * I / 32) * n;
    size_t grid = (total + 255) / 256;
    if (grid > (size_t)sm_count() * 16) grid = (size_t)sm_count() * 16;
    block_quant_mx_kernel<<<(unsigned)grid, 256, 0, s>>>(w_gu, w_d, n, H, I, records, rec_bytes, off);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const float* w_gu, const float* w_d, int n, int H, int I,
                            uint8_t* records, size_t rec_bytes, cudaStream_t s) {
    const RecordLayout r = record_layout(H, I);
    RecordOffsets off{r.gu_codes, r.gu_scales, r.d_codes, r.d_scales, r.s_gu, r.s_d};
    cudaMemsetAsync(records, 0, (size_t)n * rec_bytes, s);
    tensor_scale_kernel<<<2 * n, 1024, 0, s>>>(w_gu, w_d, H, I, records, rec_bytes, r.s_gu, r.s_d);
    const size_t total = ((size_t)2 * I * H / 16 + (size_t)H * I / 16) * n;
    size_t grid = (total + 255) / 256;
    if (grid > (size_t)sm_count() * 16) grid = (size_t)sm_count() * 16;
    block_quant_kernel<<<(unsigned)grid, 256, 0, s>>>(w_gu, w_d, n, H, I, records, rec_bytes, off);
    return cudaGetLastError();
}

}  // namespace ft
