// quantize.cuh -- quantisation of one 16-value BF16 block into the paged pool.
//
// Shared by the quantise-append kernel and the decode kernel's fused append.
// Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV
// Cache", section A3 and Fig. 1 (E2M1 values, one E4M3 scale per 16 values,
// FP32 tensor scale); the rounding argument is in quantize_append.cu.
#pragma once

#include "common.cuh"

namespace nvfp4kv {

// Round a float to 13 significant bits (half-way cases away from zero); exact
// values with <= 13 bits are unchanged.
__device__ __forceinline__ float snap13(float y) {
    uint32_t b = __float_as_uint(y);
    b = (b + 0x400u) & ~0x7ffu;
    return __uint_as_float(b);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// (a.x * b, a.y * b), each rounded to nearest, in one instruction
__device__ __forceinline__ float2 mul2(float2 a, float b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"((uint64_t)__float_as_uint(a.x) | ((uint64_t)__float_as_uint(a.y) << 32)),
          "l"((uint64_t)__float_as_uint(b) | ((uint64_t)__float_as_uint(b) << 32)));
    return make_float2(__uint_as_float((uint32_t)d), __uint_as_float((uint32_t)(d >> 32)));
}

// Approximate reciprocal (the hardware's, at most one unit in the last place off).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// fl32(1/6).  For every non-negative BF16 amax, E4M3(fl32(amax * kOneSixth))
// equals E4M3(fl32(amax / 6)) (checked over all of them on the host), so the
// unit-scale path multiplies where the scale decision is defined by a division.
constexpr float kOneSixth = 0.16666667163372039794921875f;

template <bool kUnitScale>
__device__ __forceinline__ void quantize_block16(const uint4 &a, const uint4 &b, float g, uint2 &codes,
                                                 uint32_t &scale_byte) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    // amax over BF16 magnitudes: unsigned order of |bf16| bit patterns is numeric order
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) m = max_u16x2(m, w[i] & 0x7fff7fffu);
    const uint32_t amax_bits = (m >> 16) > (m & 0xffffu) ? (m >> 16) : (m & 0xffffu);
    const float amax = __uint_as_float(amax_bits << 16);
    const float q = kUnitScale ? __fmul_rn(amax, kOneSixth) : __fdiv_rn(amax, __fmul_rn(6.0f, g));
    const uint32_t s = f32x2_to_e4m3x2(0.0f, q) & 0xffu;
    scale_byte = s;
    const float sd = __half2float(__ushort_as_half((uint16_t)(e4m3x2_to_f16x2(s) & 0xffffu)));
    uint32_t packed[2] = {0u, 0u};
    if (sd == 0.0f) {
        // signed zeros: code 8 where the input is negative
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t lo_neg = (w[i] >> 15) & 1u, hi_neg = w[i] >> 31;
            const uint32_t byte = (lo_neg << 3) | (hi_neg << 7);
            packed[i / 4] |= byte << (8 * (i % 4));
        }
    } else if (kUnitScale) {
        const float r = rcp_approx(sd);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float2 y = mul2(make_float2(bf16_lo(w[i]), bf16_hi(w[i])), r);
            packed[i / 4] |= f32x2_to_e2m1x2(snap13(y.y), snap13(y.x)) << (8 * (i % 4));
        }
    } else {
        const float d = __fmul_rn(sd, g);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float lo = __fdiv_rn(bf16_lo(w[i]), d);
            const float hi = __fdiv_rn(bf16_hi(w[i]), d);
            packed[i / 4] |= f32x2_to_e2m1x2(hi, lo) << (8 * (i % 4));
        }
    }
    codes = make_uint2(packed[0], packed[1]);
}

__device__ __forceinline__ float f16_lo(uint32_t x) { return __half2float(__ushort_as_half((uint16_t)(x & 0xffffu))); }
__device__ __forceinline__ float f16_hi(uint32_t x) { return __half2float(__ushort_as_half((uint16_t)(x >> 16))); }

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float hi, float lo) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// f16x2 holding exact values -> bf16x2 of (value * g), one rounding to BF16
// after the FP32 product (exact when g = 1).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_scaled(uint32_t x, float g) {
    return f32x2_to_bf16x2(__fmul_rn(f16_hi(x), g), __fmul_rn(f16_lo(x), g));
}

// One NVFP4 16-value block (8 code bytes, one E4M3 scale byte) -> 8 BF16 pairs
// of e2m1 * e4m3 * g, rounded to BF16 once (exact for g = 1): the prefix
// dequant kernel and the paged extend kernel both expand blocks this way.
__device__ __forceinline__ void nvfp4_block_to_bf16(uint2 codes, uint32_t sbyte, float g, uint32_t (&o)[8]) {
    const uint32_t s2 = e4m3x2_to_f16x2(sbyte | (sbyte << 8));  // {s, s}
    uint32_t f[8];
    e2m1x8_to_f16x2x4(codes.x, f[0], f[1], f[2], f[3]);
    e2m1x8_to_f16x2x4(codes.y, f[4], f[5], f[6], f[7]);
#pragma unroll
    for (int i = 0; i < 8; i++) o[i] = f16x2_to_bf16x2_scaled(hmul2(f[i], s2), g);
}

// Quantise block `blk` (0..7) of K (which = 0) or V (which = 1) of one
// head_dim row -- the 16 BF16 values at src[0..1] -- and store it at row `r`
// of the (page, h) slab.  NVFP4 slabs are 16-token groups of 2304 bytes
// (K codes | K scales | V codes | V scales [8][16]); FP8 slabs are groups of
// 4096 bytes (K codes [16][128] | V codes [16][128]).
template <bool kUnitScale>
__device__ __forceinline__ void store_block_values(uint8_t *slab_base, int dtype, int r, int which, int blk,
                                                   const uint4 &x0, const uint4 &x1, float g) {
    if (dtype == NVFP4KV_DTYPE_NVFP4) {
        uint2 codes;
        uint32_t sbyte;
        quantize_block16<kUnitScale>(x0, x1, g, codes, sbyte);
        uint8_t *grp = slab_base + (r >> 4) * 2304;
        const int rr = r & 15;
        *reinterpret_cast<uint2 *>(grp + (which ? 1152 : 0) + rr * 64 + blk * 8) = codes;
        grp[which ? 2176 + blk * 16 + rr : 1024 + rr * 8 + blk] = (uint8_t)sbyte;
    } else {
        const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float e0 = bf16_lo(w[2 * i]), e1 = bf16_hi(w[2 * i]), e2 = bf16_lo(w[2 * i + 1]), e3 = bf16_hi(w[2 * i + 1]);
            if (!kUnitScale) {
                e0 = __fdiv_rn(e0, g);
                e1 = __fdiv_rn(e1, g);
                e2 = __fdiv_rn(e2, g);
                e3 = __fdiv_rn(e3, g);
            }
            out[i] = f32x2_to_e4m3x2(e1, e0) | (f32x2_to_e4m3x2(e3, e2) << 16);
        }
        uint8_t *dst = slab_base + (r >> 4) * 4096 + (which ? 2048 : 0) + (r & 15) * 128 + blk * 16;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

// The same, loading the 16 values from src[0..1] first.
template <bool kUnitScale>
__device__ __forceinline__ void store_block(uint8_t *slab_base, int dtype, int r, int which, int blk,
                                            const uint4 *src, float g) {
    const uint4 x0 = __ldg(src), x1 = __ldg(src + 1);
    store_block_values<kUnitScale>(slab_base, dtype, r, which, blk, x0, x1, g);
}

}  // namespace nvfp4kv
