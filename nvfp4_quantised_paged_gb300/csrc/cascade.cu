// cascade.cu -- attention of every sequence's decode queries over a prefix they all share.
//
// Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV
// Cache", section A4 (the agentic workload: many sequences carry the same
// system prompt and tool definitions; SGLang's radix cache keeps one copy of
// those pages) and section A2, path 3 (decode reads the NVFP4 cache and
// dequantises it in the kernel).  A plain decode reads the shared pages once
// per sequence; this kernel reads and dequantises them once per kv head and
// multiplies them with the queries of all sequences together, which makes the
// shared part a dense contraction (rows = sequence x query head).  Its
// (max, sum, acc) partials are merged with the per-sequence suffix partials by
// the decode reduction (log-sum-exp), so the result is the decode attention
// of each whole sequence.
//
// One CTA = 4 warps = 64 query rows (row = sequence * G + head) of one kv head
// and one contiguous slice of the shared prefix.  Each 64-token stage is
// fetched raw (4 NVFP4 groups, cp.async) into a double buffer, dequantised by
// all threads into FP16 K and V tiles (e2m1 x e4m3 products are exact FP16
// values) in a 16-byte-chunk XOR swizzle, and consumed by FP16 mma.sync
// (S = Q K^T through ldmatrix, O += P V through ldmatrix.trans), with the same
// per-head power-of-two pre-scale of Q and base-2 lazy-rescale softmax as the
// decode kernel.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4kv {

namespace {

constexpr int kCThreads = 128;
constexpr int kCRows = 64;                  // query rows per CTA
constexpr int kCKeys = 64;                  // tokens per stage
constexpr int kCGroupBytes = 2304;          // one 16-token NVFP4 group
constexpr int kCRaw = 4 * kCGroupBytes;     // one raw stage
constexpr int kCRowBytes = 256;             // one FP16 row of 128 dims
constexpr int kCTile = kCKeys * kCRowBytes;
constexpr int kCKOff = 2 * kCRaw, kCVOff = kCKOff + kCTile, kCSmem = kCVOff + kCTile;
constexpr float kCNegInf = -__builtin_huge_valf();
constexpr uint32_t kCOnesF16x2 = 0x3c003c00u;
constexpr int kCMaxSplits = 16;
constexpr int kCTargetCtas = 608;           // about 4 CTAs per SM of a 152-SM GPU

struct SharedArgs {
    const uint8_t *pool;
    int64_t num_pages;
    int P, log2P, Hkv, G, Hq, B;
    int64_t slab;
    const int32_t *shared_pages;
    int tiles_per_split, ntiles;
    const uint32_t *q;   // BF16 pairs
    float score_log2;    // sm_scale * g_K * log2(e)
    float2 *ml;          // [split][B * Hkv][G]
    float *acc;
    unsigned *err;
};

__device__ __forceinline__ uint32_t cswz(int row, int chunk) {
    return (uint32_t)(row * kCRowBytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void c_cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void c_ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                          bool trans) {
    if (trans)
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                     : "r"(addr));
    else
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                     : "r"(addr));
}

__device__ __forceinline__ float c_bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float c_bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Q of one row as FP16 A-operand words (dims 16ks + 2c, +1 and 16ks + 2c + 8, +9)
// after a power-of-two pre-scale that puts the head's largest |q| in
// [2^14, 2^15); returns the score factor that undoes it.
__device__ __forceinline__ float load_q_row(const uint32_t *qrow, bool valid, int c, float score_log2,
                                            uint32_t (&w)[8][2]) {
    uint32_t raw[8][2];
    uint32_t m = 0;
#pragma unroll
    for (int ks = 0; ks < 8; ks++) {
        raw[ks][0] = valid ? __ldg(qrow + 8 * ks + c) : 0u;
        raw[ks][1] = valid ? __ldg(qrow + 8 * ks + 4 + c) : 0u;
        m = __vmaxu2(m, raw[ks][0] & 0x7fff7fffu);
        m = __vmaxu2(m, raw[ks][1] & 0x7fff7fffu);
    }
    m = max(m >> 16, m & 0xffffu);
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
    int kq = 0;
    if (m != 0) {
        const int e = (int)((m >> 7) & 0xff) - 127;
        kq = min(126, max(-126, 14 - e));
    }
    const float s = __uint_as_float((uint32_t)(kq + 127) << 23);
#pragma unroll
    for (int ks = 0; ks < 8; ks++)
#pragma unroll
        for (int h = 0; h < 2; h++) w[ks][h] = f32x2_to_f16x2(c_bf16_hi(raw[ks][h]) * s, c_bf16_lo(raw[ks][h]) * s);
    return score_log2 * __uint_as_float((uint32_t)(127 - kq) << 23);
}

__global__ void __launch_bounds__(kCThreads, 3) shared_prefix_kernel(SharedArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();
    pdl_wait();  // q and the cache may come from earlier work on the stream
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int kv = blockIdx.y, split = blockIdx.z;
    const int rows = a.B * a.G;
    const int row0 = blockIdx.x * kCRows;
    const int t_begin = split * a.tiles_per_split;
    const int t_end = min(a.ntiles, t_begin + a.tiles_per_split);
    if (row0 >= rows || t_begin >= t_end) return;

    const int ra = row0 + 16 * warp + g, rb = ra + 8;
    const bool va = ra < rows, vb = rb < rows;
    const int ba = va ? ra / a.G : 0, ha = va ? ra % a.G : 0;
    const int bb = vb ? rb / a.G : 0, hb = vb ? rb % a.G : 0;
    uint32_t qa[8][2], qb[8][2];
    const float fa = load_q_row(a.q + ((int64_t)ba * a.Hq + kv * a.G + ha) * (kHeadDim / 2), va, c, a.score_log2, qa);
    const float fb = load_q_row(a.q + ((int64_t)bb * a.Hq + kv * a.G + hb) * (kHeadDim / 2), vb, c, a.score_log2, qb);

    const uint32_t sbase = smem_u32(smem);
    // raw stage of tile i into slot s: 4 groups x 144 chunks of 16 bytes
    auto issue = [&](int i, int s) {
        for (int idx = tid; idx < 4 * 144; idx += kCThreads) {
            const int gi = idx / 144, ci = idx - gi * 144;
            const int t = i * kCKeys + 16 * gi;
            const int32_t pg = __ldg(a.shared_pages + (t >> a.log2P));
            const bool ok = pg >= 0 && (int64_t)pg < a.num_pages;
            if (!ok && ci == 0) flag_error(a.err, kErrPage);
            const uint8_t *src = ok ? a.pool + ((int64_t)pg * a.Hkv + kv) * a.slab +
                                          ((t & (a.P - 1)) >> 4) * kCGroupBytes + ci * 16
                                    : a.pool;
            c_cp_async16(sbase + s * kCRaw + gi * kCGroupBytes + ci * 16, src, ok);
        }
    };

    float o[16][4], ol[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 16; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_a = kCNegInf, m_b = kCNegInf;

    issue(t_begin, 0);
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (t_begin + 1 < t_end) issue(t_begin + 1, 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int i = t_begin; i < t_end; i++) {
        const int slot = (i - t_begin) & 1;
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncthreads();
        // ---- dequantise the raw stage into FP16 K and V tiles
        const uint8_t *raw = smem + slot * kCRaw;
#pragma unroll
        for (int it = 0; it < 8; it++) {
            const int u = tid + it * kCThreads;  // 0..1023: K units then V units
            const int which = u >> 9, key = (u >> 3) & 63, blk = u & 7;
            const uint8_t *grp = raw + (key >> 4) * kCGroupBytes;
            const int rr = key & 15;
            const uint2 codes = *reinterpret_cast<const uint2 *>(grp + (which ? 1152 : 0) + rr * 64 + blk * 8);
            const uint32_t sb = grp[which ? 2176 + blk * 16 + rr : 1024 + rr * 8 + blk];
            const uint32_t s2 = e4m3x2_to_f16x2(sb | (sb << 8));
            uint32_t f[8];
            e2m1x8_to_f16x2x4(codes.x, f[0], f[1], f[2], f[3]);
            e2m1x8_to_f16x2x4(codes.y, f[4], f[5], f[6], f[7]);
#pragma unroll
            for (int j = 0; j < 8; j++) f[j] = hmul2(f[j], s2);
            uint8_t *tile = smem + (which ? kCVOff : kCKOff);
            *reinterpret_cast<uint4 *>(tile + cswz(key, 2 * blk)) = make_uint4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<uint4 *>(tile + cswz(key, 2 * blk + 1)) = make_uint4(f[4], f[5], f[6], f[7]);
        }
        __syncthreads();
        if (i + 2 < t_end) issue(i + 2, slot);  // the raw slot has been consumed
        asm volatile("cp.async.commit_group;" ::: "memory");

        // ---- S = Q K^T (16 rows x 64 keys per warp)
        const uint32_t kt = sbase + kCKOff, vt = sbase + kCVOff;
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; n++) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ks++) {
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int m = lane >> 3;
                const int key = 16 * j + (m >> 1) * 8 + (lane & 7);
                uint32_t b0, b1, b2, b3;
                c_ldsm_x4(kt + cswz(key, 2 * ks + (m & 1)), b0, b1, b2, b3, false);
                mma_f16_16816(s[2 * j], qa[ks][0], qb[ks][0], qa[ks][1], qb[ks][1], b0, b1);
                mma_f16_16816(s[2 * j + 1], qa[ks][0], qb[ks][0], qa[ks][1], qb[ks][1], b2, b3);
            }
        }
        // ---- online softmax, base 2 (every key of the shared prefix is valid)
        float mx_a = kCNegInf, mx_b = kCNegInf;
#pragma unroll
        for (int n = 0; n < 8; n++) {
            s[n][0] *= fa;
            s[n][1] *= fa;
            s[n][2] *= fb;
            s[n][3] *= fb;
            mx_a = fmaxf(mx_a, fmaxf(s[n][0], s[n][1]));
            mx_b = fmaxf(mx_b, fmaxf(s[n][2], s[n][3]));
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        if (__any_sync(0xffffffffu, mx_a > m_a + 8.0f || mx_b > m_b + 8.0f)) {
            const float na = fmaxf(m_a, mx_a), nb = fmaxf(m_b, mx_b);
            const float ca = m_a == kCNegInf ? 0.f : ex2(m_a - na), cb = m_b == kCNegInf ? 0.f : ex2(m_b - nb);
            m_a = na;
            m_b = nb;
            ol[0] *= ca;
            ol[1] *= ca;
            ol[2] *= cb;
            ol[3] *= cb;
#pragma unroll
            for (int d = 0; d < 16; d++) {
                o[d][0] *= ca;
                o[d][1] *= ca;
                o[d][2] *= cb;
                o[d][3] *= cb;
            }
        }
        uint32_t pa[4][4];
#pragma unroll
        for (int n = 0; n < 8; n++) {
            pa[n >> 1][(n & 1) * 2 + 0] = f32x2_to_f16x2(ex2(s[n][1] - m_a), ex2(s[n][0] - m_a));
            pa[n >> 1][(n & 1) * 2 + 1] = f32x2_to_f16x2(ex2(s[n][3] - m_b), ex2(s[n][2] - m_b));
        }
        // ---- O += P V, and the row sums of the same FP16 P
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {
#pragma unroll
            for (int nd = 0; nd < 16; nd += 2) {
                const int m = lane >> 3;
                const int key = 16 * kk + (m & 1) * 8 + (lane & 7);
                uint32_t b0, b1, b2, b3;
                c_ldsm_x4(vt + cswz(key, nd + (m >> 1)), b0, b1, b2, b3, true);
                mma_f16_16816(o[nd], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
                mma_f16_16816(o[nd + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
            }
            mma_f16_16816(ol, pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], kCOnesF16x2, kCOnesF16x2);
        }
        __syncthreads();  // the tiles are rewritten by the next stage
    }

    // ---- partials of this slice: (m, l) and unnormalised acc per row
    const int64_t pairs = (int64_t)a.B * a.Hkv;
    if (va) {
        const int64_t idx = ((int64_t)split * pairs + (int64_t)ba * a.Hkv + kv) * a.G + ha;
        if (c == 0) a.ml[idx] = make_float2(m_a, ol[0]);
        float *dst = a.acc + idx * kHeadDim;
#pragma unroll
        for (int d = 0; d < 16; d++) *reinterpret_cast<float2 *>(dst + 8 * d + 2 * c) = make_float2(o[d][0], o[d][1]);
    }
    if (vb) {
        const int64_t idx = ((int64_t)split * pairs + (int64_t)bb * a.Hkv + kv) * a.G + hb;
        if (c == 0) a.ml[idx] = make_float2(m_b, ol[2]);
        float *dst = a.acc + idx * kHeadDim;
#pragma unroll
        for (int d = 0; d < 16; d++) *reinterpret_cast<float2 *>(dst + 8 * d + 2 * c) = make_float2(o[d][2], o[d][3]);
    }
}

}  // namespace

int cascade_splits(const nvfp4kv_cache &c, int batch, int num_q_heads, int shared_len) {
    const int ntiles = shared_len / kCKeys;
    if (ntiles <= 0 || batch <= 0) return 1;
    const int64_t G = num_q_heads / c.num_kv_heads;
    const int64_t ctas = ceil_div64((int64_t)batch * G, kCRows) * c.num_kv_heads;
    int64_t s = ceil_div64(kCTargetCtas, ctas);
    if (s > kCMaxSplits) s = kCMaxSplits;
    if (s > ntiles) s = ntiles;
    if (s < 1) s = 1;
    const int64_t per = ceil_div64(ntiles, s);  // tiles per slice; no slice is left empty
    return (int)ceil_div64(ntiles, per);
}

cudaError_t launch_shared_prefix(const nvfp4kv_cache &c, const void *q, int batch, int num_q_heads,
                                 const int32_t *shared_pages, int shared_len, int splits, float sm_scale,
                                 float2 *casc_ml, float *casc_acc, unsigned *err, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(reinterpret_cast<const void *>(&shared_prefix_kernel),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kCSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    SharedArgs a;
    a.pool = static_cast<const uint8_t *>(c.pool);
    a.num_pages = c.num_pages;
    a.P = c.page_size;
    a.log2P = __builtin_ctz((unsigned)c.page_size);
    a.Hkv = c.num_kv_heads;
    a.G = num_q_heads / c.num_kv_heads;
    a.Hq = num_q_heads;
    a.B = batch;
    a.slab = (int64_t)144 * c.page_size;
    a.shared_pages = shared_pages;
    a.ntiles = shared_len / kCKeys;
    a.tiles_per_split = (a.ntiles + splits - 1) / splits;
    a.q = static_cast<const uint32_t *>(q);
    a.score_log2 = (float)((double)sm_scale * (double)c.k_global_scale * 1.4426950408889634);
    a.ml = casc_ml;
    a.acc = casc_acc;
    a.err = err;
    // every slice must leave a partial for every row: the reduce reads all `splits`
    const int eff = (a.ntiles + a.tiles_per_split - 1) / a.tiles_per_split;
    if (eff != splits) return cudaErrorInvalidValue;
    dim3 grid((unsigned)ceil_div64((int64_t)batch * a.G, kCRows), (unsigned)c.num_kv_heads, (unsigned)splits);
    void *args[] = {&a};
    return launch_pdl(reinterpret_cast<const void *>(&shared_prefix_kernel), grid, kCThreads, kCSmem, stream, args);
}

}  // namespace nvfp4kv
