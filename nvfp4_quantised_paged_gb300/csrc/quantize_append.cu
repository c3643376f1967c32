// quantize_append.cu -- BF16 K/V rows -> NVFP4 (or FP8) rows in the paged pool.
//
// Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV
// Cache", section A2, paths 1 and 2 (the KV of a prefill or of a new chunk is
// quantised and written into the persistent paged cache), format of section A3
// and Fig. 1 (E2M1 values, one E4M3 scale per 16 values, FP32 tensor scale).
//
// One thread quantises one 16-value block: 32 bytes of BF16 in (two 16-byte
// loads), 8 bytes of packed codes + 1 scale byte out.  Eight consecutive
// threads cover one head_dim row, so reads are fully coalesced and the 64-byte
// code row is written by one 8-thread group.  The kernel is HBM-bound: per
// token and KV head it reads 512 B of BF16 and writes 144 B.
//
// Rounding (must match the CPU oracle bit for bit):
//   q     = amax / (6 g)                         FP32, correctly rounded
//   scale = cvt.rn.satfinite.e4m3 (q)            nearest-even, saturating
//   y_i   = x_i / (scale g)                      see below
//   code  = cvt.rn.satfinite.e2m1 (y_i)          nearest-even, saturating
// For g = 1 the kernel forms y_i as x_i * rcp(scale) and then rounds y_i to 13
// significant bits.  x_i has at most 8 significant bits and the scale at most
// 4, so every exact quotient that is not exactly an E2M1 rounding midpoint lies
// more than 2^-8 (relative) away from every midpoint, far outside the 2^-23
// error of the reciprocal product; an exact midpoint has at most 3 significant
// bits and the 13-bit rounding lands on it exactly.  Hence the codes equal
// those of the exactly rounded quotient (the GPU tests check every BF16 value
// against every scale).  For g != 1 the kernel divides with IEEE division.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4kv {

namespace {

struct AppendArgs {
    uint8_t *pool;
    int64_t num_slots;  // num_pages * P
    int P;
    int log2P;
    int Hkv;
    int64_t slab;       // bytes per (page, kv_head)
    const uint4 *k;     // BF16 rows viewed as 16-byte vectors
    const uint4 *v;
    int64_t num_tokens;
    int64_t stride16;   // token stride in 16-byte units
    const int64_t *slots;
    float gk, gv;
    unsigned *err;
};

// Round a float to 13 significant bits (half-way cases away from zero); exact
// values with <= 13 bits are unchanged.
__device__ __forceinline__ float snap13(float y) {
    uint32_t b = __float_as_uint(y);
    b = (b + 0x400u) & ~0x7ffu;
    return __uint_as_float(b);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <bool kUnitScale>
__device__ __forceinline__ void quantize_block16(const uint4 &a, const uint4 &b, float g, uint2 &codes,
                                                 uint32_t &scale_byte) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    // amax over BF16 magnitudes: unsigned order of |bf16| bit patterns is numeric order
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) m = __vmaxu2(m, w[i] & 0x7fff7fffu);
    const uint32_t amax_bits = (m >> 16) > (m & 0xffffu) ? (m >> 16) : (m & 0xffffu);
    const float amax = __uint_as_float(amax_bits << 16);
    const float q = kUnitScale ? __fdiv_rn(amax, 6.0f) : __fdiv_rn(amax, __fmul_rn(6.0f, g));
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
        const float r = __frcp_rn(sd);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float lo = snap13(bf16_lo(w[i]) * r);
            const float hi = snap13(bf16_hi(w[i]) * r);
            packed[i / 4] |= f32x2_to_e2m1x2(hi, lo) << (8 * (i % 4));
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

// Thread id -> (token, kv_head, which, block), block fastest.
template <bool kUnitScale>
__global__ void __launch_bounds__(256) append_nvfp4_kernel(AppendArgs a) {
    pdl_launch_dependents();  // a dependent decode plan may launch early; it waits for this kernel
    // the host guarantees num_tokens * Hkv * 16 < 2^31
    const uint32_t id = blockIdx.x * blockDim.x + threadIdx.x;
    if (id >= (uint32_t)(a.num_tokens * a.Hkv * 16)) return;
    const int blk = (int)(id & 7);
    const int which = (int)((id >> 3) & 1);
    const uint32_t th = id >> 4;
    const uint32_t t32 = th / (uint32_t)a.Hkv;
    const int h = (int)(th - t32 * (uint32_t)a.Hkv);
    const int64_t t = t32;
    const int64_t slot = __ldg(a.slots + t);
    if (slot < 0) return;
    if (slot >= a.num_slots) {
        if (blk == 0 && which == 0 && h == 0) flag_error(a.err, kErrSlot);
        return;
    }
    const uint4 *src = (which ? a.v : a.k) + t * a.stride16 + h * (kHeadDim / 8) + blk * 2;
    const uint4 x0 = __ldg(src), x1 = __ldg(src + 1);
    uint2 codes;
    uint32_t sbyte;
    quantize_block16<kUnitScale>(x0, x1, which ? a.gv : a.gk, codes, sbyte);
    const int64_t page = slot >> a.log2P;
    const int r = (int)(slot & (a.P - 1));
    // 16-token groups of 2304 bytes: K codes | K scales | V codes | V scales [8][16]
    uint8_t *grp = a.pool + (page * a.Hkv + h) * a.slab + (r >> 4) * 2304;
    const int rr = r & 15;
    *reinterpret_cast<uint2 *>(grp + (which ? 1152 : 0) + rr * 64 + blk * 8) = codes;
    grp[which ? 2176 + blk * 16 + rr : 1024 + rr * 8 + blk] = (uint8_t)sbyte;
}

// FP8 pool: one thread converts one 16-value block to 16 E4M3 bytes.
template <bool kUnitScale>
__global__ void __launch_bounds__(256) append_fp8_kernel(AppendArgs a) {
    pdl_launch_dependents();  // a dependent decode plan may launch early; it waits for this kernel
    // the host guarantees num_tokens * Hkv * 16 < 2^31
    const uint32_t id = blockIdx.x * blockDim.x + threadIdx.x;
    if (id >= (uint32_t)(a.num_tokens * a.Hkv * 16)) return;
    const int blk = (int)(id & 7);
    const int which = (int)((id >> 3) & 1);
    const uint32_t th = id >> 4;
    const uint32_t t32 = th / (uint32_t)a.Hkv;
    const int h = (int)(th - t32 * (uint32_t)a.Hkv);
    const int64_t t = t32;
    const int64_t slot = __ldg(a.slots + t);
    if (slot < 0) return;
    if (slot >= a.num_slots) {
        if (blk == 0 && which == 0 && h == 0) flag_error(a.err, kErrSlot);
        return;
    }
    const uint4 *src = (which ? a.v : a.k) + t * a.stride16 + h * (kHeadDim / 8) + blk * 2;
    const uint4 x0 = __ldg(src), x1 = __ldg(src + 1);
    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const float g = which ? a.gv : a.gk;
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
    const int64_t page = slot >> a.log2P;
    const int r = (int)(slot & (a.P - 1));
    // 16-token groups of 4096 bytes: K codes [16][128] | V codes [16][128]
    uint8_t *dst = a.pool + (page * a.Hkv + h) * a.slab + (r >> 4) * 4096 + (which ? 2048 : 0) + (r & 15) * 128 +
                   blk * 16;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
}

}  // namespace

cudaError_t launch_quantize_append(const nvfp4kv_cache &c, const void *k, const void *v, int64_t num_tokens,
                                   int64_t token_stride, const int64_t *slot_mapping, unsigned *err,
                                   cudaStream_t stream) {
    AppendArgs a;
    a.pool = static_cast<uint8_t *>(c.pool);
    a.num_slots = c.num_pages * (int64_t)c.page_size;
    a.P = c.page_size;
    a.log2P = __builtin_ctz((unsigned)c.page_size);
    a.Hkv = c.num_kv_heads;
    a.slab = (int64_t)(c.dtype == NVFP4KV_DTYPE_NVFP4 ? 144 : 256) * c.page_size;
    a.k = static_cast<const uint4 *>(k);
    a.v = static_cast<const uint4 *>(v);
    a.num_tokens = num_tokens;
    a.stride16 = token_stride / 8;
    a.slots = slot_mapping;
    a.gk = c.k_global_scale;
    a.gv = c.v_global_scale;
    a.err = err;
    const int64_t threads = num_tokens * c.num_kv_heads * 2 * 8;
    const int block = 256;
    const int64_t grid = ceil_div64(threads, block);
    const bool unit = c.k_global_scale == 1.0f && c.v_global_scale == 1.0f;
    if (c.dtype == NVFP4KV_DTYPE_NVFP4) {
        if (unit)
            append_nvfp4_kernel<true><<<(unsigned)grid, block, 0, stream>>>(a);
        else
            append_nvfp4_kernel<false><<<(unsigned)grid, block, 0, stream>>>(a);
    } else {
        if (unit)
            append_fp8_kernel<true><<<(unsigned)grid, block, 0, stream>>>(a);
        else
            append_fp8_kernel<false><<<(unsigned)grid, block, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace nvfp4kv
