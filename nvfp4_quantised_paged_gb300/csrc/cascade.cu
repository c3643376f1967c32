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
// One CTA = 4 warps = 128 query rows (row = sequence * G + head, one TMEM lane
// each) of one kv head and one contiguous slice of the shared prefix.  Per
// 64-token stage: thread 0 fetches the four raw NVFP4 groups with 1-D bulk
// copies into a double buffer; all threads dequantise them (e2m1 x e4m3 is an
// exact FP16 value) into FP16 K and V tiles in the tensor core's 128-byte
// swizzle layout; thread 0 issues S = Q K^T as tcgen05.mma (FP16 inputs, FP32
// accumulator in TMEM; Q pre-scaled per row by a power of two, exact, undone
// in the score factor); each thread runs the base-2 lazy-rescale softmax of
// its row from tcgen05.ld and stores P (FP16) into TMEM; thread 0 runs
// O += P V and the row sums (all-ones operand) with P read from TMEM.
// Two CTAs share an SM.  Every wait is bounded.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace nvfp4kv {

namespace {

constexpr int kCThreads = 128;              // one thread per query row
constexpr int kCRows = 128;                 // query rows per CTA
constexpr int kCKeys = 64;                  // tokens per stage
constexpr int kCGroupBytes = 2304;          // one 16-token NVFP4 group
constexpr int kCRaw = 4 * kCGroupBytes;     // one raw stage
constexpr int kCKVBlock = kCKeys * 128;     // one column block of a K or V tile
constexpr int kCKVTile = 2 * kCKVBlock;
constexpr int kCOffQ = 0;                                   // FP16 Q: 2 blocks of [128][64]
constexpr int kCOffRaw = kCOffQ + kCRows * 256;             // raw stages [2]
constexpr int kCOffKV = 53248;                              // K | V FP16 tiles (1024-aligned)
constexpr int kCOffOnes = kCOffKV + 2 * kCKVTile;           // FP16 1.0 [16][64]
constexpr int kCOffBar = kCOffOnes + 16 * 128;              // bar_s, bar_pv, raw_full[2]
constexpr int kCOffTmem = kCOffBar + 32;
constexpr int kCSmem = kCOffTmem + 16;
static_assert(kCOffRaw + 2 * kCRaw <= kCOffKV, "raw stages overlap the tiles");
constexpr uint32_t kCTmemCols = 256;        // S 0..63, P 64..95, O 96..223, row sums 224..239
constexpr uint32_t kCColP = 64, kCColO = 96, kCColL = 224;
constexpr float kCNegInf = -__builtin_huge_valf();
constexpr uint32_t kCWaitLimit = 1u << 24;
constexpr int kCMaxSplits = 16;
constexpr int kCTargetCtas = 152;           // about one CTA per SM of a 152-SM GPU: fewer slices, fewer partials to merge

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

__device__ __forceinline__ float c_bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float c_bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kCThreads, 2) shared_prefix_kernel(SharedArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t &bar_s = *reinterpret_cast<uint64_t *>(smem + kCOffBar);
    uint64_t &bar_pv = *reinterpret_cast<uint64_t *>(smem + kCOffBar + 8);
    uint64_t *raw_full = reinterpret_cast<uint64_t *>(smem + kCOffBar + 16);
    uint32_t &tmem_base = *reinterpret_cast<uint32_t *>(smem + kCOffTmem);
    // q and the cache may come from earlier work on the stream.  The decode
    // kernel launched behind this one reads the plan's results without a wait
    // of its own: every CTA here first waits for the plan to complete, then
    // lets the decode grid launch.
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5;
    const int kv = blockIdx.y, split = blockIdx.z;
    const int rows = a.B * a.G;
    const int row0 = blockIdx.x * kCRows;
    const int t_begin = split * a.tiles_per_split;
    const int t_end = min(a.ntiles, t_begin + a.tiles_per_split);
    if (row0 >= rows || t_begin >= t_end) return;
    const int nt = t_end - t_begin;
    const uint32_t sbase = smem_u32(smem);

    // raw stage of tile i (0-based in this slice) into slot s: four groups, thread 0
    auto issue_raw = [&](int i, int s) {
        mbar_arrive_expect_tx(&raw_full[s], kCRaw);
        for (int gi = 0; gi < 4; gi++) {
            const int t = (t_begin + i) * kCKeys + 16 * gi;
            const int32_t pg = __ldg(a.shared_pages + (t >> a.log2P));
            const uint8_t *src = a.pool;
            if (pg >= 0 && (int64_t)pg < a.num_pages)
                src = a.pool + ((int64_t)pg * a.Hkv + kv) * a.slab + ((t & (a.P - 1)) >> 4) * kCGroupBytes;
            else
                flag_error(a.err, kErrPage);  // the group is fetched from the pool start, i.e. garbage
            bulk_g2s(smem + kCOffRaw + s * kCRaw + gi * kCGroupBytes, src, kCGroupBytes, &raw_full[s]);
        }
    };
    if (tid == 0) {
        mbar_init(&bar_s, 1);
        mbar_init(&bar_pv, 1);
        mbar_init(&raw_full[0], 1);
        mbar_init(&raw_full[1], 1);
        fence_mbar_init();
        issue_raw(0, 0);
        if (nt > 1) issue_raw(1, 1);
    }
    if (warp == 0) tc_alloc(&tmem_base, kCTmemCols);

    // ---- this thread's query row, FP16 after a power-of-two pre-scale that puts
    // its largest |q| in [2^14, 2^15); the score factor undoes it
    const int R = row0 + tid;
    const bool row_ok = R < rows;
    const int b = row_ok ? R / a.G : 0, h = row_ok ? R % a.G : 0;
    float fac;
    {
        const uint4 *qrow = reinterpret_cast<const uint4 *>(a.q + ((int64_t)b * a.Hq + kv * a.G + h) * (kHeadDim / 2));
        uint4 w[16];
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            w[i] = row_ok ? __ldg(qrow + i) : make_uint4(0, 0, 0, 0);
            m = __vmaxu2(m, w[i].x & 0x7fff7fffu);
            m = __vmaxu2(m, w[i].y & 0x7fff7fffu);
            m = __vmaxu2(m, w[i].z & 0x7fff7fffu);
            m = __vmaxu2(m, w[i].w & 0x7fff7fffu);
        }
        m = max(m >> 16, m & 0xffffu);
        int kq = 0;
        if (m != 0) kq = min(126, max(-126, 14 - ((int)((m >> 7) & 0xff) - 127)));
        const float sc = __uint_as_float((uint32_t)(kq + 127) << 23);
        fac = a.score_log2 * __uint_as_float((uint32_t)(127 - kq) << 23);
#pragma unroll
        for (int i = 0; i < 16; i++) {  // chunk i = dims 8i .. 8i+7
            const uint32_t x[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
            uint32_t f[4];
#pragma unroll
            for (int e = 0; e < 4; e++) f[e] = f32x2_to_f16x2(c_bf16_hi(x[e]) * sc, c_bf16_lo(x[e]) * sc);
            *reinterpret_cast<uint4 *>(smem + kCOffQ + (i >> 3) * (kCRows * 128) + sw128_off(tid, i & 7)) =
                make_uint4(f[0], f[1], f[2], f[3]);
        }
    }
    for (int idx = tid; idx < 16 * 128 / 16; idx += kCThreads) {  // FP16 1.0 everywhere
        const uint32_t one2 = 0x3c003c00u;
        *reinterpret_cast<uint4 *>(smem + kCOffOnes + idx * 16) = make_uint4(one2, one2, one2, one2);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t sQ = sbase + kCOffQ, sK = sbase + kCOffKV, sV = sK + kCKVTile, sOnes = sbase + kCOffOnes;
    constexpr uint32_t idesc_s = idesc_f16_f32(128, kCKeys, false);
    constexpr uint32_t idesc_o = idesc_f16_f32(128, kHeadDim, true);
    constexpr uint32_t idesc_l = idesc_f16_f32(128, 16, false);
    float m_run = kCNegInf;
    bool aborted = false;

    for (int i = 0; i < nt; i++) {
        const int slot = i & 1;
        bool ok = mbar_wait_bounded(&raw_full[slot], (uint32_t)((i >> 1) & 1), kCWaitLimit, nullptr);
        if (i > 0) ok = ok && mbar_wait_bounded(&bar_pv, (uint32_t)((i - 1) & 1), kCWaitLimit, nullptr);
        if (__syncthreads_or(!ok)) {  // the raw stage landed and P V of the previous tile is done
            if (tid == 0) flag_error(a.err, kErrTimeout);
            aborted = true;
            break;
        }
        tc_fence_after();
        // ---- dequantise the raw stage into the FP16 K and V tiles
        const uint8_t *raw = smem + kCOffRaw + slot * kCRaw;
#pragma unroll
        for (int it = 0; it < 8; it++) {
            const int u = tid + it * kCThreads;  // K units then V units
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
            uint8_t *tile = smem + kCOffKV + which * kCKVTile + (blk >> 2) * kCKVBlock;
            *reinterpret_cast<uint4 *>(tile + sw128_off(key, (blk & 3) * 2)) = make_uint4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<uint4 *>(tile + sw128_off(key, (blk & 3) * 2 + 1)) = make_uint4(f[4], f[5], f[6], f[7]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the tiles for the tensor core
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            if (i + 2 < nt) issue_raw(i + 2, slot);  // this raw slot has been dequantised
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {  // S = Q K^T over head_dim, 16 at a time
                const uint32_t blk = (uint32_t)(kk >> 2), sub = (uint32_t)(kk & 3) * 32;
                tc_mma_bf16(tmem, smem_desc_sw128(sQ + blk * (kCRows * 128) + sub, 16, 1024),
                            smem_desc_sw128(sK + blk * kCKVBlock + sub, 16, 1024), idesc_s, kk > 0);
            }
            tc_commit(&bar_s);
        }
        ok = mbar_wait_bounded(&bar_s, (uint32_t)(i & 1), kCWaitLimit, nullptr);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) flag_error(a.err, kErrTimeout);
            aborted = true;
            break;
        }
        tc_fence_after();

        // ---- softmax of this thread's row (every shared token is visible)
        uint32_t sr[2][32];
        tc_ld32(tmem + lane_base + 0, sr[0]);
        tc_ld32(tmem + lane_base + 32, sr[1]);
        tc_wait_ld();
        float smax = __uint_as_float(sr[0][0]);
#pragma unroll
        for (int j = 1; j < 64; j++) smax = fmaxf(smax, __uint_as_float(sr[j >> 5][j & 31]));
        const float mx = smax * fac;
        const bool need = mx > m_run + 8.0f;
        if (__any_sync(0xffffffffu, need)) {
            const float m_new = need ? fmaxf(m_run, mx) : m_run;
            const float alpha = need ? (m_run == kCNegInf ? 0.f : ex2(m_run - m_new)) : 1.f;
            if (i > 0) {  // O and the row sums hold earlier tiles
#pragma unroll
                for (int cblk = 0; cblk < 5; cblk++) {
                    uint32_t ov[32];
                    const uint32_t col = cblk < 4 ? kCColO + 32 * cblk : kCColL;
                    tc_ld32(tmem + lane_base + col, ov);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j++) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
                    tc_st32(tmem + lane_base + col, ov);
                }
                tc_wait_st();
            }
            m_run = m_new;
        }
        const float neg_m = -m_run;
        uint32_t pw[32];
#pragma unroll
        for (int c = 0; c < 32; c++)
            pw[c] = f32x2_to_f16x2(ex2(fmaf(__uint_as_float(sr[(2 * c + 1) >> 5][(2 * c + 1) & 31]), fac, neg_m)),
                                   ex2(fmaf(__uint_as_float(sr[(2 * c) >> 5][(2 * c) & 31]), fac, neg_m)));
        tc_st32(tmem + lane_base + kCColP, pw);
        tc_wait_st();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {  // O += P V; row sums += P 1
                const uint32_t pa = tmem + kCColP + kk * 8;
                const uint32_t accf = (i > 0 || kk > 0) ? 1u : 0u;
                tc_mma_bf16_tmem_a(tmem + kCColO, pa, smem_desc_sw128(sV + kk * 16 * 128, kCKVBlock, 1024), idesc_o,
                                   accf);
                tc_mma_bf16_tmem_a(tmem + kCColL, pa, smem_desc_sw128(sOnes + kk * 32, 16, 1024), idesc_l, accf);
            }
            tc_commit(&bar_pv);
        }
    }
    if (!aborted) {
        const bool ok = mbar_wait_bounded(&bar_pv, (uint32_t)((nt - 1) & 1), kCWaitLimit, nullptr);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) flag_error(a.err, kErrTimeout);
            aborted = true;
        }
        tc_fence_after();
    }
    if (!aborted) {
        // ---- this slice's partial of the row: (m, l) and the unnormalised acc
        uint32_t lv[32];
        tc_ld32(tmem + lane_base + kCColL, lv);
        tc_wait_ld();
        const int64_t idx = ((int64_t)split * a.B * a.Hkv + (int64_t)b * a.Hkv + kv) * a.G + h;
        if (row_ok) a.ml[idx] = make_float2(m_run, __uint_as_float(lv[0]));
        float4 *dst = reinterpret_cast<float4 *>(a.acc + idx * kHeadDim);
#pragma unroll
        for (int cblk = 0; cblk < 4; cblk++) {
            uint32_t ov[32];
            tc_ld32(tmem + lane_base + kCColO + 32 * cblk, ov);
            tc_wait_ld();
            if (row_ok) {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    dst[8 * cblk + j] = make_float4(__uint_as_float(ov[4 * j]), __uint_as_float(ov[4 * j + 1]),
                                                    __uint_as_float(ov[4 * j + 2]), __uint_as_float(ov[4 * j + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, kCTmemCols);
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
