// quantize.cuh -- quantisation of one 16-value BF16 block into the paged pool.
//
// Shared by the quantise-append kernel and the decode kernel's fused append.
// Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV
// Cache", section A3 and Fig. 1 (E2M1 values, one E4M3 scale per 16 values,
// FP32 tensor scale); the rounding argument for g = 1 is in quantize_append.cu,
// the one for other tensor scales beside e4m3_code_exact below.
#pragma once

#include "common.cuh"

namespace nvfp4kv {

// (hi, lo) floats -> f16x2, each rounded to nearest-even (11 significant
// bits; beyond the FP16 range: infinity).
__device__ __forceinline__ uint32_t f32x2_to_f16x2_rn(float hi, float lo) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four f16x2 -> one word of eight E2M1 codes (element 2i in the low nibble of
// byte i), each rounded to nearest-even and saturated (infinity -> 6).
__device__ __forceinline__ uint32_t f16x2x4_to_e2m1x8(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    uint32_t r;
    asm("{ .reg .b8 p, q, s, t;\n"
        "  cvt.rn.satfinite.e2m1x2.f16x2 p, %1; cvt.rn.satfinite.e2m1x2.f16x2 q, %2;\n"
        "  cvt.rn.satfinite.e2m1x2.f16x2 s, %3; cvt.rn.satfinite.e2m1x2.f16x2 t, %4;\n"
        "  mov.b32 %0, {p, q, s, t}; }"
        : "=r"(r)
        : "r"(a), "r"(b), "r"(c), "r"(d));
    return r;
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

// ---------------------------------------------------------------------------
// Tensor scale g != 1: every scale and code is the rounding of the EXACT
// quotient (amax / (6 g), x / (s g), x / g), nearest-even, saturating.  An FP32
// estimate (a / g) / den lands within two units in its last place of the exact
// quotient, so its rounding is right or one code off; each neighbouring midpoint mu is then
// checked exactly: quotient >= mu  <=>  a <= mu' g, where mu' (= mu, 6 mu or
// mu s, at most 7 significant bits) is exact in FP32 and fma(mu', g, -a) is the
// exact difference rounded once, so its sign (and zero) is exact.  That holds
// while mu' g >= 2^-117 (the difference is then a multiple of 2^-148, never
// lost to underflow); below g = 2^-100 both sides are scaled by 2^64 first.
// ---------------------------------------------------------------------------

constexpr float kTinyTensorScale = 0x1p-100f;
constexpr float kTinyRescale = 0x1p64f;

// Magnitude of E2M1 code c (0..7): 0, 0.5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ float e2m1_magnitude(uint32_t c) {
    const uint32_t e = c >> 1, m = c & 1u;
    return e == 0 ? 0.5f * (float)m : __uint_as_float(((e + 126u) << 23) | (m << 22));
}

// Magnitude of E4M3 code c (0..126), exact.
__device__ __forceinline__ float e4m3_magnitude(uint32_t c) {
    return __half2float(__ushort_as_half((uint16_t)(e4m3x2_to_f16x2(c) & 0xffffu)));
}

// Move magnitude code c (0..cmax) to the exact rounding of a / (den g), where
// the caller's estimate c is at most one code off.  mag(k) = value of code k;
// the midpoint between k and k+1, times den, is exact in FP32.
template <typename Mag>
__device__ __forceinline__ uint32_t fix_code(uint32_t c, uint32_t cmax, float a, float den, float g, Mag mag) {
    if (c < cmax) {
        const float mu = 0.5f * (mag(c) + mag(c + 1)) * den;
        const float d = __fmaf_rn(mu, g, -a);            // sign of mu g - a, exact
        if (d < 0.0f || (d == 0.0f && ((c + 1) & 1u) == 0)) return c + 1;
    }
    if (c > 0) {
        const float mu = 0.5f * (mag(c - 1) + mag(c)) * den;
        const float d = __fmaf_rn(mu, g, -a);
        if (d > 0.0f || (d == 0.0f && ((c - 1) & 1u) == 0)) return c - 1;
    }
    return c;
}

// The estimate divides by g first: den g may overflow FP32 (g near its
// largest value), a / g cannot go wrong by more than a code (it overflows only
// where every code saturates and underflows only where every code is 0).
__device__ __forceinline__ uint32_t e4m3_code_exact(float a, float den, float g) {
    const uint32_t c = f32x2_to_e4m3x2(0.0f, __fdiv_rn(__fdiv_rn(a, g), den)) & 0x7fu;
    return fix_code(c, 126u, a, den, g, [](uint32_t k) { return e4m3_magnitude(k); });
}

__device__ __forceinline__ uint32_t e2m1_code_exact(float a, float den, float g) {
    const uint32_t c = f32x2_to_e2m1x2(0.0f, __fdiv_rn(__fdiv_rn(a, g), den)) & 7u;
    return fix_code(c, 7u, a, den, g, [](uint32_t k) { return e2m1_magnitude(k); });
}

// The e2m1 * e4m3 (or e4m3) value p, exact in FP32, times g, rounded once to
// BF16 (nearest-even; subnormal steps of 2^-133; infinity on overflow).
// hi = fl(p g) and lo = p g - hi exactly (an FMA, exact while p g >= 2^-118);
// hi decides the rounding unless it sits exactly on a BF16 midpoint, where the
// sign of lo does.  Below g = 2^-100 the product is formed at g 2^64.
__device__ __forceinline__ uint32_t bf16_of_product(float p, float g) {
    const uint32_t sign = (__float_as_uint(p) >> 16) & 0x8000u;
    const float a = fabsf(p);
    if (a == 0.0f) return sign;
    const bool tiny = g < kTinyTensorScale;
    const float gs = tiny ? g * kTinyRescale : g;
    const float hi = a * gs;
    const float lo = __fmaf_rn(a, gs, -hi);
    if (!tiny || hi >= 0x1p-62f) {      // a BF16 normal (or infinity) after unscaling
        uint32_t b = __float_as_uint(hi);
        if ((b & 0xffffu) == 0x8000u && lo != 0.0f) b += (lo > 0.0f) ? 1u : 0xffffffffu;  // off the tie, toward p g
        uint32_t r = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(b)));
        if (tiny) r = __float_as_uint(__uint_as_float(r << 16) * (1.0f / kTinyRescale)) >> 16;  // exact: >= 2^-126
        return r | sign;
    }
    // below 2^-126 after unscaling: BF16 steps of 2^-133, i.e. units of hi 2^69
    const float t = hi * 0x1p69f;
    float f = floorf(t);
    const float r = t - f;
    if (r > 0.5f || (r == 0.5f && (lo > 0.0f || (lo == 0.0f && fmodf(f, 2.0f) != 0.0f)))) f += 1.0f;
    return (uint32_t)f | sign;
}

template <bool kUnitScale>
__device__ __forceinline__ void quantize_block16(const uint4 &a, const uint4 &b, float g, uint2 &codes,
                                                 uint32_t &scale_byte) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    // amax over BF16 magnitudes: unsigned order of |bf16| bit patterns is numeric order
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) m = max_u16x2(m, w[i] & 0x7fff7fffu);
    const uint32_t amax_bits = (m >> 16) > (m & 0xffffu) ? (m >> 16) : (m & 0xffffu);
    float amax = __uint_as_float(amax_bits << 16);
    const bool tiny = !kUnitScale && g < kTinyTensorScale;   // decide at (x, g) 2^64: same quotients
    const float gs = tiny ? g * kTinyRescale : g;
    if (tiny) amax *= kTinyRescale;
    const uint32_t s = kUnitScale ? f32x2_to_e4m3x2(0.0f, __fmul_rn(amax, kOneSixth)) & 0xffu
                                  : e4m3_code_exact(amax, 6.0f, gs);
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
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float2 y = mul2(make_float2(bf16_lo(w[i]), bf16_hi(w[i])), r);
            h[i] = f32x2_to_f16x2_rn(y.y, y.x);
        }
        packed[0] = f16x2x4_to_e2m1x8(h[0], h[1], h[2], h[3]);
        packed[1] = f16x2x4_to_e2m1x8(h[4], h[5], h[6], h[7]);
    } else {
        const float xs = tiny ? kTinyRescale : 1.0f;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t clo = e2m1_code_exact(fabsf(bf16_lo(w[i])) * xs, sd, gs) | ((w[i] >> 12) & 8u);
            const uint32_t chi = e2m1_code_exact(fabsf(bf16_hi(w[i])) * xs, sd, gs) | ((w[i] >> 28) & 8u);
            packed[i / 4] |= (clo | (chi << 4)) << (8 * (i % 4));
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

// f16x2 holding exact values -> bf16x2 of (value * g), each the exact product
// rounded to BF16 once; kUnit (g = 1): a plain, exact conversion.  Callers pick
// kUnit outside their loops (the general form is long).
template <bool kUnit>
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_scaled(uint32_t x, float g) {
    if (kUnit) return f32x2_to_bf16x2(f16_hi(x), f16_lo(x));
    return bf16_of_product(f16_lo(x), g) | (bf16_of_product(f16_hi(x), g) << 16);
}

// One NVFP4 16-value block (8 code bytes, one E4M3 scale byte) -> 8 BF16 pairs
// of e2m1 * e4m3 * g, the exact product rounded to BF16 once (exact for g = 1:
// at most 6 significant bits): the prefix dequant kernel and the paged extend
// kernel both expand blocks this way.  kUnit: g = 1.
template <bool kUnit>
__device__ __forceinline__ void nvfp4_block_to_bf16(uint2 codes, uint32_t sbyte, float g, uint32_t (&o)[8]) {
    const uint32_t s2 = e4m3x2_to_f16x2(sbyte | (sbyte << 8));  // {s, s}
    uint32_t f[8];
    e2m1x8_to_f16x2x4(codes.x, f[0], f[1], f[2], f[3]);
    e2m1x8_to_f16x2x4(codes.y, f[4], f[5], f[6], f[7]);
#pragma unroll
    for (int i = 0; i < 8; i++) o[i] = f16x2_to_bf16x2_scaled<kUnit>(hmul2(f[i], s2), g);
}

// L2 policy "evict last" (all of a request's lines), for st_u8_policy.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void st_u8_policy(uint8_t *p, uint32_t v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.u8 [%0], %1, %2;" ::"l"(p), "h"((unsigned short)v), "l"(policy) : "memory");
}

// Quantise block `blk` (0..7) of K (which = 0) or V (which = 1) of one
// head_dim row -- the 16 BF16 values at src[0..1] -- and store it at row `r`
// of the (page, h) slab.  NVFP4 slabs are 16-token groups of 2304 bytes
// (K codes | K scales | V codes | V scales [8][16]); FP8 slabs are groups of
// 4096 bytes (K codes [16][128] | V codes [16][128]).  kScalePolicy: the scale
// byte is stored with the L2 policy `policy` (a 32-byte sector of scales holds
// bytes of four (K) or sixteen (V) tokens, so a token alone writes it partly).
template <bool kUnitScale, bool kScalePolicy = false>
__device__ __forceinline__ void store_block_values(uint8_t *slab_base, int dtype, int r, int which, int blk,
                                                   const uint4 &x0, const uint4 &x1, float g,
                                                   uint64_t policy = 0) {
    if (dtype == NVFP4KV_DTYPE_NVFP4) {
        uint2 codes;
        uint32_t sbyte;
        quantize_block16<kUnitScale>(x0, x1, g, codes, sbyte);
        uint8_t *grp = slab_base + (r >> 4) * 2304;
        const int rr = r & 15;
        *reinterpret_cast<uint2 *>(grp + (which ? 1152 : 0) + rr * 64 + blk * 8) = codes;
        uint8_t *sdst = grp + (which ? 2176 + blk * 16 + rr : 1024 + rr * 8 + blk);
        if (kScalePolicy)
            st_u8_policy(sdst, sbyte, policy);
        else
            *sdst = (uint8_t)sbyte;
    } else {
        const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float e0 = bf16_lo(w[2 * i]), e1 = bf16_hi(w[2 * i]), e2 = bf16_lo(w[2 * i + 1]),
                        e3 = bf16_hi(w[2 * i + 1]);
            if (kUnitScale) {
                out[i] = f32x2_to_e4m3x2(e1, e0) | (f32x2_to_e4m3x2(e3, e2) << 16);
            } else {
                const bool tiny = g < kTinyTensorScale;
                const float gs = tiny ? g * kTinyRescale : g, xs = tiny ? kTinyRescale : 1.0f;
                const float e[4] = {e0, e1, e2, e3};
                uint32_t o = 0;
#pragma unroll
                for (int j = 0; j < 4; j++)
                    o |= (e4m3_code_exact(fabsf(e[j]) * xs, 1.0f, gs) | ((__float_as_uint(e[j]) >> 24) & 0x80u))
                         << (8 * j);
                out[i] = o;
            }
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
