// extend_attention.cu -- attention of a new chunk over [cached prefix || chunk], causal in the chunk.
//
// Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV
// Cache", section A2, path 2 (chunked prefill / extend): the attention takes
// two KV sources, the cached prefix -- gathered from the NVFP4 pages and
// dequantised into a workspace shared across layers (prefix_dequant.cu
// writes it, in BF16) -- and the current chunk's own K/V.  Chunk token i
// attends to the whole prefix and to chunk tokens 0..i.
//
// GB300 design: a flash-attention forward on the 5th-generation tensor cores.
// One CTA = 4 warps = 128 query rows of one (request, kv head), row = chunk
// token * G + query head of the group, so the G heads that share a KV head
// share every K/V tile.  Per 64-key tile:
//   * thread 0 loads K and V with four TMA boxes (3-D tensor maps, 128-byte
//     swizzle = the tensor core's canonical operand layout) into one of two
//     stages, completing on that stage's mbarrier;
//   * thread 0 issues S = Q K^T as eight tcgen05.mma (M 128, N 64, K 16) with
//     Q and K read from shared memory by descriptor, accumulating in TMEM
//     columns 0..63, and commits to an mbarrier;
//   * each thread owns one query row = one TMEM lane: it loads its 64 scores
//     (tcgen05.ld), masks them on edge tiles only, runs the base-2 online
//     softmax with a lazily updated running max (O and the row sums in TMEM
//     are rescaled only when a score exceeds the max by 2^8), forms
//     P = 2^(s * scale - m) with one FFMA per score, rounds it to BF16 and
//     stores its row of P into TMEM (tcgen05.st);
//   * thread 0 then runs O += P V as four tcgen05.mma with P read from TMEM
//     (M 128, N 128, K 16, V as an MN-major operand) into TMEM columns
//     96..223, and the row sums as four more with an all-ones B operand, so
//     numerator and denominator see the same rounded P.
// The commit after the next S means S and every earlier MMA are done, which
// also frees P and the previous K/V stage (refilled right then).  Two CTAs
// share an SM (99 KB of shared memory and 256 TMEM columns each), so one
// CTA's softmax overlaps the other's MMAs.  Every wait is bounded; a timeout
// is reported in the device error word and taken by all threads together.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace nvfp4kv {

namespace {

constexpr int kEThreads = 128;            // one thread per query row
constexpr int kQRows = 128;               // query rows per CTA
constexpr int kKeys = 64;                 // keys per K/V tile
constexpr int kQBytes = kQRows * 256;     // Q: 2 column blocks of [128][64] BF16
constexpr int kKVBlock = kKeys * 128;     // one column block of a K or V tile (one TMA box)
constexpr int kKVTile = 2 * kKVBlock;     // a whole K (or V) tile
constexpr int kStageBytes = 2 * kKVTile;  // K | V
constexpr int kOnesBytes = 16 * 128;      // all-ones B operand [16][64] for the row sums
constexpr int kOffQ = 0, kOffStage = kQBytes, kOffOnes = kOffStage + 2 * kStageBytes;
constexpr int kOffBar = kOffOnes + kOnesBytes;  // bar_mma, full[2]
constexpr int kOffTmem = kOffBar + 24;
constexpr int kOffOrder = kOffTmem + 8;   // int[128]: requests by decreasing prefix length
constexpr int kESmem = kOffOrder + 4 * 128;
// TMEM columns: S 0..63 (FP32), P 64..95 (BF16 pairs), O 96..223, row sums 224..239
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColP = 64, kColO = 96, kColL = 224;
constexpr float kRescale = 8.0f;
constexpr float kNegInfE = -__builtin_huge_valf();
constexpr uint32_t kWaitLimitE = 1u << 24;
constexpr int kOrderMax = kEThreads;      // requests ordered by prefix length up to this many

struct ExtendArgs {
    const uint16_t *q;                 // BF16 [total_q][Hq][128]
    const int32_t *cu_prefix, *cu_q;   // [num_reqs + 1]
    int Hq, Hkv, G, max_q_len;
    float score_log2;                  // sm_scale * log2(e)
    uint16_t *out;                     // BF16 [total_q][Hq][128]
    unsigned *err;
};

// K/V tensors [rows][Hkv][128] BF16 as 3-D TMA maps with 64 x 1 x 64 boxes, 128-byte swizzle.
struct ExtendMaps {
    CUtensorMap k_pre, v_pre, k_new, v_new;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__global__ void __launch_bounds__(kEThreads, 2) extend_kernel(const __grid_constant__ ExtendMaps maps, ExtendArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t &bar_mma = *reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar + 8);  // [2]: stage landed
    uint32_t &tmem_base = *reinterpret_cast<uint32_t *>(smem + kOffTmem);
    const int tid = threadIdx.x, warp = tid >> 5;
    // Requests in order of decreasing prefix length (the longest CTAs start
    // first, so the tail of the grid holds short ones): blockIdx.z is the
    // rank; thread j ranks request j.
    int r = blockIdx.z;
    if (gridDim.z <= kOrderMax) {
        int *order = reinterpret_cast<int *>(smem + kOffOrder);
        const int nr = (int)gridDim.z;
        if (tid < nr) {
            const int nj = a.cu_prefix[tid + 1] - a.cu_prefix[tid];
            int rank = 0;
            for (int c = 0; c < nr; c++) {
                const int nc = a.cu_prefix[c + 1] - a.cu_prefix[c];
                rank += nc > nj || (nc == nj && c < tid);
            }
            order[rank] = tid;
        }
        __syncthreads();
        r = order[blockIdx.z];
    }
    const int kv = blockIdx.y;
    const int q0 = a.cu_q[r], p0 = a.cu_prefix[r];
    int L = a.cu_q[r + 1] - q0;
    const int np = a.cu_prefix[r + 1] - p0;
    if (L < 0 || np < 0) {
        if (tid == 0 && blockIdx.x == 0 && kv == 0) flag_error(a.err, kErrCuPrefix);
        return;
    }
    if (L > a.max_q_len) {
        if (tid == 0 && blockIdx.x == 0 && kv == 0) flag_error(a.err, kErrSeqLen);
        L = a.max_q_len;
    }
    const int rows = L * a.G;
    const int row0 = blockIdx.x * kQRows;
    if (row0 >= rows) return;
    const int t_last = (min(row0 + kQRows, rows) - 1) / a.G;  // last chunk token of this CTA
    const int nt_pre = (np + kKeys - 1) / kKeys;
    const int nt = nt_pre + t_last / kKeys + 1;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + kOffQ;

    // ---- Q tile: 128 rows x 16 chunks of 16 bytes
#pragma unroll 4
    for (int it = 0; it < 16; it++) {
        const int idx = tid + it * kEThreads;
        const int row = idx >> 4, c16 = idx & 15;
        const int R = row0 + row;
        const bool ok = R < rows;
        const int64_t src = ok ? (((int64_t)q0 + R / a.G) * a.Hq + kv * a.G + R % a.G) * kHeadDim + c16 * 8 : 0;
        cp_async16(sQ + (c16 >> 3) * (kQRows * 128) + sw128_off(row, c16 & 7), a.q + src, ok);
    }
    // K/V tile i into stage s: four TMA boxes (K and V, head_dim 0..63 and
    // 64..127) completing on full[s]; rows past the tensor are zero-filled,
    // rows of a neighbouring request are masked by the softmax
    auto issue = [&](int i, int s) {  // thread 0
        const bool pre = i < nt_pre;
        const int row = pre ? p0 + i * kKeys : q0 + (i - nt_pre) * kKeys;
        const CUtensorMap *mk = pre ? &maps.k_pre : &maps.k_new;
        const CUtensorMap *mv = pre ? &maps.v_pre : &maps.v_new;
        const uint32_t st = sbase + kOffStage + s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        tma_load_3d(st, mk, 0, kv, row, &full[s]);
        tma_load_3d(st + kKVBlock, mk, 64, kv, row, &full[s]);
        tma_load_3d(st + kKVTile, mv, 0, kv, row, &full[s]);
        tma_load_3d(st + kKVTile + kKVBlock, mv, 64, kv, row, &full[s]);
    };
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int idx = tid; idx < kOnesBytes / 16; idx += kEThreads) {  // BF16 1.0 everywhere
        const uint32_t one2 = 0x3f803f80u;
        *reinterpret_cast<uint4 *>(smem + kOffOnes + idx * 16) = make_uint4(one2, one2, one2, one2);
    }

    if (warp == 0) tc_alloc(&tmem_base, kTmemCols);
    if (tid == 0) {
        mbar_init(&bar_mma, 1);
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_mbar_init();
        issue(0, 0);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q and the ones tile for the tensor core
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lanes

    // this thread's query row
    const int R = row0 + tid;
    const bool row_ok = R < rows;
    const int token = row_ok ? R / a.G : 0;

    constexpr uint32_t idesc_s = idesc_bf16_f32(128, kKeys, false);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, kHeadDim, true);
    constexpr uint32_t idesc_l = idesc_bf16_f32(128, 16, false);
    const uint32_t sOnes = sbase + kOffOnes;
    float m_run = kNegInfE;
    uint32_t phase = 0;
    bool aborted = false;

    for (int i = 0; i < nt && !aborted; i++) {
        const int s_cur = i & 1;
        const uint32_t sK = sbase + kOffStage + s_cur * kStageBytes, sV = sK + kKVTile;
        if (tid == 0 && mbar_wait_bounded(&full[s_cur], (uint32_t)((i >> 1) & 1), kWaitLimitE, nullptr)) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {  // S = Q K^T over head_dim, 16 at a time
                const uint32_t blk = (uint32_t)(kk >> 2), sub = (uint32_t)(kk & 3) * 32;
                tc_mma_bf16(tmem, smem_desc_sw128(sQ + blk * (kQRows * 128) + sub, 16, 1024),
                            smem_desc_sw128(sK + blk * kKVBlock + sub, 16, 1024), idesc_s, kk > 0);
            }
            tc_commit(&bar_mma);
        }
        // S of this tile (and every earlier MMA) done: the other stage and P are free
        const bool ok = mbar_wait_bounded(&bar_mma, phase, kWaitLimitE, nullptr);
        if (__syncthreads_or(!ok)) {  // all threads take the same decision
            if (tid == 0) flag_error(a.err, kErrTimeout);
            aborted = true;
            break;
        }
        phase ^= 1u;
        tc_fence_after();
        if (tid == 0 && i + 1 < nt) issue(i + 1, s_cur ^ 1);  // its stage held tile i - 1, now done

        // ---- softmax of this thread's row (base 2; masked scores are -inf)
        uint32_t sr[2][32];
        tc_ld32(tmem + lane_base + 0, sr[0]);
        tc_ld32(tmem + lane_base + 32, sr[1]);
        tc_wait_ld();
        float sc[64];
#pragma unroll
        for (int j = 0; j < 64; j++) sc[j] = __uint_as_float(sr[j >> 5][j & 31]);
        {
            const bool pre = i < nt_pre;
            const int base = pre ? i * kKeys : (i - nt_pre) * kKeys;
            const int visible = (pre ? np : token + 1) - base;  // keys [0, visible) of the tile are seen
            if (__any_sync(0xffffffffu, visible < kKeys)) {     // an edge tile: mask
#pragma unroll
                for (int j = 0; j < 64; j++)
                    if (j >= visible) sc[j] = kNegInfE;
            }
        }
        float smax = sc[0];
#pragma unroll
        for (int j = 1; j < 64; j++) smax = fmaxf(smax, sc[j]);
        const float mx = smax * a.score_log2;  // the scale is positive
        const bool need = mx > m_run + kRescale;
        if (__any_sync(0xffffffffu, need)) {
            const float m_new = need ? fmaxf(m_run, mx) : m_run;
            const float alpha = need ? (m_run == kNegInfE ? 0.f : ex2(m_run - m_new)) : 1.f;
            if (i > 0) {  // O and the row sums hold earlier tiles: rescale this warp's rows in TMEM
#pragma unroll
                for (int cblk = 0; cblk < 5; cblk++) {  // O (4 x 32 columns), then the sums
                    uint32_t ov[32];
                    const uint32_t col = cblk < 4 ? kColO + 32 * cblk : kColL;
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
        // P row = 2^(s * scale - m), rounded to BF16, into this lane's P columns of TMEM
        const float neg_m = -m_run;
        uint32_t pw[32];
#pragma unroll
        for (int c = 0; c < 32; c++) {
            const __nv_bfloat162 pr =
                __floats2bfloat162_rn(ex2(fmaf(sc[2 * c], a.score_log2, neg_m)), ex2(fmaf(sc[2 * c + 1], a.score_log2, neg_m)));
            pw[c] = *reinterpret_cast<const uint32_t *>(&pr);
        }
        tc_st32(tmem + lane_base + kColP, pw);
        tc_wait_st();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {  // O += P V over this tile's 64 keys; sums += P 1
                const uint32_t pa = tmem + kColP + kk * 8;  // P from TMEM: 8 columns = 16 keys
                const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                tc_mma_bf16_tmem_a(tmem + kColO, pa, smem_desc_sw128(sV + kk * 16 * 128, kKVBlock, 1024), idesc_o,
                                   acc);
                tc_mma_bf16_tmem_a(tmem + kColL, pa, smem_desc_sw128(sOnes + kk * 32, 16, 1024), idesc_l, acc);
            }
        }
    }
    if (!aborted) {
        if (tid == 0) tc_commit(&bar_mma);
        const bool ok = mbar_wait_bounded(&bar_mma, phase, kWaitLimitE, nullptr);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) flag_error(a.err, kErrTimeout);
            aborted = true;
        }
        tc_fence_after();
    }
    if (!aborted) {
        // ---- O / l -> BF16 row of the output
        uint32_t lv[32];
        tc_ld32(tmem + lane_base + kColL, lv);
        tc_wait_ld();
        const float l_run = __uint_as_float(lv[0]);
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        uint4 *dst = reinterpret_cast<uint4 *>(a.out + (((int64_t)q0 + token) * a.Hq + kv * a.G + R % a.G) * kHeadDim);
#pragma unroll
        for (int cblk = 0; cblk < 4; cblk++) {
            uint32_t ov[32];
            tc_ld32(tmem + lane_base + kColO + 32 * cblk, ov);
            tc_wait_ld();
            if (row_ok) {
#pragma unroll
                for (int q4 = 0; q4 < 4; q4++) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(ov[8 * q4 + 2 * e]) * inv,
                                                                        __uint_as_float(ov[8 * q4 + 2 * e + 1]) * inv);
                        w[e] = *reinterpret_cast<const uint32_t *>(&h);
                    }
                    dst[4 * cblk + q4] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, kTmemCols);
}

// cuTensorMapEncodeTiled, resolved from the driver once.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// [rows][Hkv][128] BF16 at `base` as a 3-D map with 64 x 1 x 64 boxes.
bool make_kv_map(CUtensorMap *map, const void *base, int64_t rows, int Hkv) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)Hkv, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)Hkv * kHeadDim * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kKeys};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_extend(const void *q, const void *k_prefix, const void *v_prefix, const int32_t *cu_prefix,
                          int64_t total_prefix, const void *k_chunk, const void *v_chunk, const int32_t *cu_q,
                          int64_t total_q, int num_reqs, int max_q_len, int num_q_heads, int num_kv_heads,
                          float sm_scale, void *out, unsigned *err, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(reinterpret_cast<const void *>(&extend_kernel),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kESmem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    ExtendMaps maps;
    if (!make_kv_map(&maps.k_pre, k_prefix, total_prefix, num_kv_heads) ||
        !make_kv_map(&maps.v_pre, v_prefix, total_prefix, num_kv_heads) ||
        !make_kv_map(&maps.k_new, k_chunk, total_q, num_kv_heads) ||
        !make_kv_map(&maps.v_new, v_chunk, total_q, num_kv_heads))
        return cudaErrorInvalidValue;
    ExtendArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.cu_prefix = cu_prefix;
    a.cu_q = cu_q;
    a.Hq = num_q_heads;
    a.Hkv = num_kv_heads;
    a.G = num_q_heads / num_kv_heads;
    a.max_q_len = max_q_len;
    a.score_log2 = (float)((double)sm_scale * 1.4426950408889634);
    a.out = static_cast<uint16_t *>(out);
    a.err = err;
    const int64_t qtiles = ceil_div64((int64_t)max_q_len * a.G, kQRows);
    dim3 grid((unsigned)qtiles, (unsigned)num_kv_heads, (unsigned)num_reqs);
    extend_kernel<<<grid, kEThreads, kESmem, stream>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace nvfp4kv
