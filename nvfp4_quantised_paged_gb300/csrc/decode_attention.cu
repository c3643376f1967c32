// decode_attention.cu -- paged GQA decode attention that dequantises the cache on chip.
//
// Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV
// Cache", section A2, path 3 and Fig. 3: packed K/V tiles and their E4M3 block
// scales are staged in shared memory, unpacked to 16-bit floats in registers,
// multiplied by the scales with packed multiplies, and fed to the matrix
// products; the FP32 tensor scales are applied as scaling of those products.
// Dequantised KV never goes back to HBM.
//
// GB300 design (not the page's SM120 kernel):
//   * Work split.  The KV of every (sequence, kv_head) pair is cut into
//     64-token chunks; all chunks of all pairs form one flat range that is cut
//     into `grid` equal contiguous pieces, one per warp pair (grid = SM count x
//     resident warp pairs for an auto split), so every warp pair streams the
//     same number of bytes whatever the mix of sequence lengths.  The two
//     warps of a pair take alternate chunks of its range and each leaves one
//     (max, sum, acc) partial per sequence-head pair it touched; a separate
//     log-sum-exp reduction kernel merges the partials of a pair and
//     normalises.
//   * One CTA per SM holds all its warp pairs (eight for NVFP4 with up to 8
//     heads per group, four otherwise; 16 warps of 128 registers).  Eight
//     CTAs of one warp pair each did the same work with the same code 2%
//     slower: the SM's warp schedulers favour the warps of the CTAs placed on
//     it first, so those ranges finished first (in four tiers, ~80 us apart
//     on the 32K workload) and the SM ran its last stretch with few warps.
//   * Staging.  The warps of a pair share a ring of three chunk stages: the
//     warp that used a stage refills it (lane 0, one 1-D bulk (TMA) copy of
//     9,216 contiguous bytes for NVFP4 when pages hold >= 64 tokens, else one
//     copy per page, completed on the stage's mbarrier) with the chunk three
//     places ahead, which belongs to the other warp, and publishes the chunk
//     index so that a warp never waits on a barrier phase that belongs to an
//     earlier use of the stage.  The lanes resolve the sources of the next
//     8-32 refills (one page each) well ahead of their copies.  The eight
//     rings of an SM hold ~220 KB; the data of a chunk has always landed when
//     its warp gets to it.  Every wait is bounded and reports a timeout in the
//     device error word instead of spinning forever.
//   * The four 16-token groups of a chunk are processed together, step by
//     step, so their conversions and products interleave and the per-stage
//     bookkeeping is paid once per 64 tokens.
//   * Tensor cores on the real contraction only: per warp and 16 tokens,
//     S^T (16 tokens x 8 query heads of the group) = K Q^T and
//     O^T (128 dims x 8 heads) += V^T P^T with mma.sync m16n8k16, FP16 inputs
//     and FP32 accumulation.  Tokens sit on the M dimension, so a GQA group of
//     up to 8 heads fills N = 8 with no padding; groups of 9-16 use two N tiles.
//     The softmax denominators come from the same unit: an all-ones A operand
//     times P^T.
//   * Unpack.  ptxas for sm_103a accepts cvt.rn.f16x2.e2m1x2 (not the BF16
//     form), so values are unpacked to FP16.  Every e2m1 x e4m3 product is an
//     FP16 normal with <= 6 significant bits, so the scaled values are exact.
//     Q is converted to FP16 after a per-head power-of-two pre-scale (exact for
//     every element above 2^-29 of the head's largest), undone in the score scale.
//   * V operand order.  The P.V product needs, per register, two consecutive
//     tokens of one channel; the cache stores two consecutive channels of one
//     token per byte.  Two lop3/shift pairs per 8 bytes swap nibbles between
//     the two tokens before the conversion, and the V scales (stored
//     block-major) arrive as the matching token pair.
//   * Softmax in base 2 with a lazily updated running max: the accumulators are
//     rescaled only when some score exceeds the running max by more than 2^8,
//     so most tiles skip the cross-lane max and the rescale.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "quantize.cuh"

namespace nvfp4kv {

namespace {

constexpr int kWarps = 2;                  // warps per CTA, sharing one ring
constexpr int kThreads = 32 * kWarps;
constexpr int kChunk = 64;                 // tokens per unit of the work split (one ring stage)
constexpr int kGroups = kChunk / 16;       // 16-token groups per stage
constexpr int kSlots = 3;                  // ring stages per CTA: two computed, one landing
constexpr uint32_t kWaitLimit = 1u << 24;  // polls before a wait gives up (>= ~1 s)
constexpr float kRescaleLog2 = 8.0f;
constexpr float kNegInf = -__builtin_huge_valf();

// One 16-token group of a page, as stored (see include/nvfp4kv.h).
template <int DTYPE>
struct Group;
template <>
struct Group<NVFP4KV_DTYPE_NVFP4> {
    static constexpr int kBytes = 2304;
    static constexpr int kKq = 0, kKs = 1024, kVq = 1152, kVs = 2176;
};
template <>
struct Group<NVFP4KV_DTYPE_FP8_E4M3> {
    static constexpr int kBytes = 4096;
    static constexpr int kKq = 0, kVq = 2048;
};

// Batches of up to kPlanInCta sequences are planned inside every decode CTA
// (the chunk prefix in shared memory, unsigned 32-bit: a sequence has at most
// 2^25 chunks, as seq_lens are int32) instead of by a separate plan kernel,
// whose launch and completion would sit between the previous work on the
// stream and the first bulk copy.
constexpr int kPlanInCta = 96;

// Shared memory of one CTA: a ring of kSlots 64-token stages, their
// mbarriers, the mask of groups each stage holds, the index of the chunk last
// issued into each stage, an abort flag and, for a batch planned in the CTA,
// the chunk prefix (B + 1 entries).
template <int DTYPE, int NT>
struct Smem {
    static constexpr int kSubs = DTYPE == NVFP4KV_DTYPE_NVFP4 && NT == 1 ? 8 : 4;  // warp pairs per CTA
    static constexpr int kStage = kGroups * Group<DTYPE>::kBytes;
    static constexpr int kBars = kSlots * kStage;           // u64 full[kSlots]
    static constexpr int kFlags = kBars + kSlots * 8;       // int valid[kSlots]
    static constexpr int kSeq = kFlags + kSlots * 4;        // int seq[kSlots]
    static constexpr int kAbort = kSeq + kSlots * 4;        // int abort
    static constexpr int kSub = (kAbort + 4 + 127) & ~127;  // one warp pair's region (offsets above within it)
    static constexpr int kPrefixBytes = (4 * (kPlanInCta + 1) + 127) & ~127;  // u32 prefix[B + 1] at offset 0
    static constexpr int kMax = kPrefixBytes + kSubs * kSub;
};

struct DecodeArgs {
    const uint8_t *pool;
    int64_t num_pages;
    int P, log2P;
    int Hkv, G, Hq, B, max_pages;
    int64_t slab;
    const uint4 *q;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int64_t *chunk_prefix;  // [B + 1], chunks of 64 tokens per sequence (exclusive scan)
    int plan_in_cta;              // 1: every CTA computes the prefix into shared memory (chunk_prefix unused)
    float score_log2;             // sm_scale * g_K * log2(e)
    float gv;
    __nv_bfloat16 *out;
    float *part_acc;  // [slots][kWarps][G][128]
    float2 *part_ml;  // [slots][kWarps][G]
    int grid;
    unsigned *err;
    // fused append (nullptr k_new: none): sequence b's new token, row b of
    // k_new / v_new, is quantised into position seq_lens[b] - 1 first
    const uint4 *k_new, *v_new;
    int64_t new_stride16;  // row stride in 16-byte units
    float gk_q, gv_q;      // tensor scales for the quantisation
    int dtype, unit_scale;
    uint8_t *pool_w;       // the pool, writable
    int skip;              // tokens at the start of every sequence left to the shared-prefix kernel
    int after_shared;      // launched behind the shared-prefix kernel (see decode_kernel)
};

__device__ __forceinline__ int clamp_len(int32_t n, int64_t cap) {
    if (n < 0) return 0;
    return (int64_t)n > cap ? (int)cap : n;
}

// 64-token chunks of a sequence of n tokens whose first `skip` are left to the
// shared-prefix kernel, n clamped to the block table's capacity: the plan
// kernel, the in-CTA plan and the reduction's own plan all count this way.
__device__ __forceinline__ int64_t seq_chunks(int32_t n, int64_t max_tokens, int skip) {
    const int64_t m = n < skip ? 0 : ((int64_t)n > max_tokens ? max_tokens : n) - skip;
    return (m + kChunk - 1) / kChunk;
}

// Entry i of the chunk prefix: from this CTA's shared memory when the batch
// is planned in the CTA, else from the plan kernel's array.
template <int DTYPE>
__device__ __forceinline__ int64_t chunk_prefix_at(const DecodeArgs &a, int i) {
    if (a.plan_in_cta) {
        extern __shared__ __align__(128) uint8_t smem[];
        return reinterpret_cast<const uint32_t *>(smem)[i];
    }
    return a.chunk_prefix[i];
}

// A unit of the CTA's range: chunk ch (of nch) of KV head kv of sequence b,
// whose clamped length is n.
struct Cursor {
    int b, kv, ch, nch, n;
};

template <int DTYPE>
__device__ __forceinline__ void cursor_seq(Cursor &cu, const DecodeArgs &a) {
    cu.nch = (int)(chunk_prefix_at<DTYPE>(a, cu.b + 1) - chunk_prefix_at<DTYPE>(a, cu.b));
    cu.n = clamp_len(a.seq_lens[cu.b], (int64_t)a.max_pages * a.P);
}

// Move the cursor `steps` units forward (the caller keeps it inside the range).
template <int DTYPE>
__device__ __forceinline__ void cursor_advance(Cursor &cu, const DecodeArgs &a, int steps) {
    cu.ch += steps;
    while (cu.ch >= cu.nch) {
        cu.ch -= cu.nch;
        if (++cu.kv < a.Hkv) continue;
        cu.kv = 0;
        do {
            ++cu.b;
        } while (cu.b < a.B && chunk_prefix_at<DTYPE>(a, cu.b + 1) == chunk_prefix_at<DTYPE>(a, cu.b));
        if (cu.b >= a.B) return;
        cursor_seq<DTYPE>(cu, a);
    }
}

// A 64-token chunk spans npp = max(1, 64 / P) pages, so it is fetched as npp
// parts of min(P, 64) tokens, each contiguous in its page's slab.  A part's
// source is one 64-bit code: 0 when the part starts past the sequence end,
// kBadPage when its block-table entry is out of range, else the global address
// of its first group (256-byte aligned: groups are 2,304 or 4,096 bytes and the
// pool is 256-byte aligned) plus the number of its groups holding tokens in the
// low bits.  The 32 lanes of the warp resolve the parts of 32 / npp upcoming
// units (binary search over the chunk prefix, block-table read) long before
// their copies are issued.
constexpr uint64_t kBadPage = 0xff;

template <int DTYPE>
__device__ __forceinline__ uint64_t part_src(const DecodeArgs &a, int64_t u0, int nstages, int j, int part) {
    if (j >= nstages) return 0;
    const int64_t u = u0 + j;
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)a.Hkv * chunk_prefix_at<DTYPE>(a, mid) <= u) lo = mid;
        else hi = mid - 1;
    }
    const int64_t p_lo = chunk_prefix_at<DTYPE>(a, lo);
    const int nch = (int)(chunk_prefix_at<DTYPE>(a, lo + 1) - p_lo);
    const int rem = (int)(u - (int64_t)a.Hkv * p_lo);
    const int kv = rem / nch, ch = rem - kv * nch;
    const int n = clamp_len(a.seq_lens[lo], (int64_t)a.max_pages * a.P);
    const int span = a.P < kChunk ? a.P : kChunk;
    const int t = a.skip + ch * kChunk + part * span;
    if (t >= n) return 0;
    const int32_t pg = __ldg(a.block_table + (int64_t)lo * a.max_pages + (t >> a.log2P));
    if (pg < 0 || (int64_t)pg >= a.num_pages) return kBadPage;
    const int ng = (min(span, n - t) + 15) >> 4;
    return reinterpret_cast<uint64_t>(a.pool + ((int64_t)pg * a.Hkv + kv) * a.slab +
                                      ((t & (a.P - 1)) >> 4) * Group<DTYPE>::kBytes) |
           (uint64_t)ng;
}

// Fetch one 64-token stage.  Every lane passes the codes of the stage's parts
// (lanes first .. first + npp - 1 of `codes`); lane 0 issues one bulk copy per
// part into `dst` and records which groups arrive in *valid (bit i = group i).
// Groups that are not fetched (past the end, or a bad page, which is flagged)
// are masked out of the tile arithmetic.
template <int DTYPE>
__device__ __forceinline__ void issue_stage(const DecodeArgs &a, uint64_t codes, int first, int npp, int lane,
                                            uint8_t *dst, uint64_t *full, int *valid) {
    constexpr int kGB = Group<DTYPE>::kBytes;
    if (npp == 1) {  // pages of >= 64 tokens: one copy (the common case, kept short)
        uint64_t s0 = __shfl_sync(0xffffffffu, codes, first);
        if (lane != 0) return;
        if (s0 == kBadPage) {
            flag_error(a.err, kErrPage);
            s0 = 0;
        }
        const int ng = (int)(s0 & 0xff);
        *valid = (1 << ng) - 1;
        if (ng == 0) {
            mbar_arrive(full);
            return;
        }
        mbar_arrive_expect_tx(full, (uint32_t)ng * kGB);
        bulk_g2s(dst, reinterpret_cast<const void *>(s0 & ~(uint64_t)0xff), (uint32_t)ng * kGB, full);
        return;
    }
    const int gpp = kGroups / npp;  // groups per part
    uint64_t src[kGroups];
#pragma unroll
    for (int p = 0; p < kGroups; p++) {
        src[p] = 0;
        if (p < npp) src[p] = __shfl_sync(0xffffffffu, codes, first + p);
    }
    if (lane != 0) return;
    uint32_t tx = 0;
    int mask = 0;
#pragma unroll
    for (int p = 0; p < kGroups; p++) {
        if (src[p] == kBadPage) {
            flag_error(a.err, kErrPage);
            src[p] = 0;
        }
        const int ng = (int)(src[p] & 0xff);
        tx += (uint32_t)ng * kGB;
        mask |= ((1 << ng) - 1) << (p * gpp);
    }
    *valid = mask;
    if (tx == 0) {
        mbar_arrive(full);
        return;
    }
    mbar_arrive_expect_tx(full, tx);
#pragma unroll
    for (int p = 0; p < kGroups; p++) {
        const int ng = (int)(src[p] & 0xff);
        if (ng)
            bulk_g2s(dst + p * gpp * kGB, reinterpret_cast<const void *>(src[p] & ~(uint64_t)0xff), (uint32_t)ng * kGB,
                     full);
    }
}


// (a & m) | (b & ~m)
__device__ __forceinline__ uint32_t bitsel(uint32_t m, uint32_t a, uint32_t b) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(r) : "r"(a), "r"(b), "r"(m));
    return r;
}

// Orders this thread's generic-proxy shared-memory accesses before its
// following bulk (async-proxy) copies into the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Q fragments of one (sequence, kv_head): lane (g, c) holds head nt*8+g,
// channels 32c .. 32c+31 as the B operand of the 8 k-steps (k-step j covers
// channels 32c+4j .. 32c+4j+3 of every lane c); fac = score scale per head of
// the lane's S columns (heads nt*8 + 2c, +1), including the undo of the
// power-of-two pre-scale.
template <int NT>
__device__ __forceinline__ void load_q(const DecodeArgs &a, int b, int kv, int lane, uint32_t (&qf)[NT][8][2],
                                       float (&fac)[NT][2]) {
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
        const int head = nt * 8 + g;
        uint32_t w[16];
        if (head < a.G) {
            const uint4 *src = a.q + ((int64_t)b * a.Hq + (int64_t)kv * a.G + head) * (kHeadDim / 8) + c * 4;
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const uint4 v = __ldg(src + k);
                w[4 * k] = v.x;
                w[4 * k + 1] = v.y;
                w[4 * k + 2] = v.z;
                w[4 * k + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 16; k++) w[k] = 0u;
        }
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 16; k++) m = __vmaxu2(m, w[k] & 0x7fff7fffu);
        m = max(m >> 16, m & 0xffffu);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        // pre-scale 2^kq puts the head's largest |q| in [2^14, 2^15)
        int kq = 0;
        if (m != 0) {
            const int e = (int)((m >> 7) & 0xff) - 127;  // exponent of the BF16 amax (subnormal -> -127)
            kq = min(126, max(-126, 14 - e));
        }
        const float s = __uint_as_float((uint32_t)(kq + 127) << 23);
#pragma unroll
        for (int j = 0; j < 8; j++) {
            qf[nt][j][0] = f32x2_to_f16x2(bf16_hi(w[2 * j]) * s, bf16_lo(w[2 * j]) * s);
            qf[nt][j][1] = f32x2_to_f16x2(bf16_hi(w[2 * j + 1]) * s, bf16_lo(w[2 * j + 1]) * s);
        }
        const int kq0 = __shfl_sync(0xffffffffu, kq, 8 * c);
        const int kq1 = __shfl_sync(0xffffffffu, kq, 8 * c + 4);
        fac[nt][0] = a.score_log2 * __uint_as_float((uint32_t)(127 - kq0) << 23);
        fac[nt][1] = a.score_log2 * __uint_as_float((uint32_t)(127 - kq1) << 23);
    }
}

// Accumulator tile kLTile of o[nt] holds the softmax denominators: it is the
// product of an all-ones A operand with P^T, so its c0 / c1 are the sums of
// the tile's probabilities for heads nt*8+2c, +1.
constexpr int kLTile = 8;
constexpr uint32_t kOnesF16x2 = 0x3c003c00u;

// Online softmax over T 16-token S^T tiles at once (rows g, g+8 of each tile;
// columns = heads nt*8+2c, +1), producing the P^T operands of the P.V
// products.  Scores are in base 2; the running max moves only when a score
// exceeds it by more than 2^kRescaleLog2, so probabilities stay <= 2^8 (exact
// enough in FP16) and most calls skip the cross-lane max and the rescale.
// vt[t] = valid rows of tile t (0..16); tile 0 holds at least one.  FULL:
// every row of every tile is valid (vt is not read).
template <int NT, int T, bool FULL = false>
__device__ __forceinline__ void softmax_tiles(const float (&s)[T][NT][4], int g, const int (&vt)[T],
                                              const float (&fac)[NT][2], float (&m_run)[NT][2], float (&o)[NT][9][4],
                                              uint32_t (&pb)[T][NT][2]) {
    float x[T][NT][4];
    bool need = false;
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) x[t][nt][e] = fmaf(s[t][nt][e], fac[nt][e & 1], -m_run[nt][e & 1]);
            if (!FULL && vt[t] < 16) {
                if (g >= vt[t]) x[t][nt][0] = x[t][nt][1] = kNegInf;
                if (g + 8 >= vt[t]) x[t][nt][2] = x[t][nt][3] = kNegInf;
            }
#pragma unroll
            for (int e = 0; e < 4; e++) need |= x[t][nt][e] > kRescaleLog2;  // +inf on a segment's first stage
        }
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            float y[T][4];
            float t0 = kNegInf, t1 = kNegInf;
#pragma unroll
            for (int t = 0; t < T; t++) {
#pragma unroll
                for (int e = 0; e < 4; e++) y[t][e] = x[t][nt][e] == kNegInf ? kNegInf : s[t][nt][e] * fac[nt][e & 1];
                t0 = fmaxf(t0, fmaxf(y[t][0], y[t][2]));
                t1 = fmaxf(t1, fmaxf(y[t][1], y[t][3]));
            }
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) {
                t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, sh));
                t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, sh));
            }
            const float n0 = fmaxf(m_run[nt][0], t0), n1 = fmaxf(m_run[nt][1], t1);
            const float a0 = ex2(m_run[nt][0] - n0), a1 = ex2(m_run[nt][1] - n1);
            m_run[nt][0] = n0;
            m_run[nt][1] = n1;
#pragma unroll
            for (int i = 0; i < 9; i++) {
                o[nt][i][0] *= a0;
                o[nt][i][1] *= a1;
                o[nt][i][2] *= a0;
                o[nt][i][3] *= a1;
            }
#pragma unroll
            for (int t = 0; t < T; t++) {
                x[t][nt][0] = y[t][0] - n0;
                x[t][nt][1] = y[t][1] - n1;
                x[t][nt][2] = y[t][2] - n0;
                x[t][nt][3] = y[t][3] - n1;
            }
        }
    }
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            const float p0 = ex2(x[t][nt][0]), p1 = ex2(x[t][nt][1]), p2 = ex2(x[t][nt][2]), p3 = ex2(x[t][nt][3]);
            pb[t][nt][0] = movmatrix_trans(f32x2_to_f16x2(p1, p0));
            pb[t][nt][1] = movmatrix_trans(f32x2_to_f16x2(p3, p2));
        }
}

// One warp, T consecutive 16-token NVFP4 groups (st = the first), written
// step by step for all T tiles together so that their conversions and
// products interleave.  vt[t] = valid rows of group t (0..16); FULL: all 16
// rows of every group are valid (the masking code is left out).
template <int NT, int T, bool FULL = false>
__device__ __forceinline__ void tiles_nvfp4(const uint8_t *st, const int (&vt)[T], int lane,
                                            const uint32_t (&qf)[NT][8][2], const float (&fac)[NT][2],
                                            float (&m_run)[NT][2], float (&o)[NT][9][4]) {
    using L = Group<NVFP4KV_DTYPE_NVFP4>;
    const int g = lane >> 2, c = lane & 3;
    // ---- S^T = K Q^T.  Lane loads channels 32c..32c+31 (16 bytes) of rows g, g+8.
    float s[T][NT][4];
#pragma unroll
    for (int t = 0; t < T; t++) {
        const uint8_t *gt = st + t * L::kBytes;
        const uint8_t *krow = gt + L::kKq + g * 64 + 16 * c;
        const uint4 kA = *reinterpret_cast<const uint4 *>(krow);
        const uint4 kB = *reinterpret_cast<const uint4 *>(krow + 8 * 64);
        const uint8_t *ks = gt + L::kKs + g * 8 + 2 * c;
        const uint32_t sA = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t *>(ks));
        const uint32_t sB = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t *>(ks + 8 * 8));
        const uint32_t sA_lo = __byte_perm(sA, 0, 0x1010), sA_hi = __byte_perm(sA, 0, 0x3232);
        const uint32_t sB_lo = __byte_perm(sB, 0, 0x1010), sB_hi = __byte_perm(sB, 0, 0x3232);
        const uint32_t kAw[4] = {kA.x, kA.y, kA.z, kA.w}, kBw[4] = {kB.x, kB.y, kB.z, kB.w};
        float sacc[2][NT][4];
#pragma unroll
        for (int x = 0; x < 2; x++)
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
#pragma unroll
                for (int e = 0; e < 4; e++) sacc[x][nt][e] = 0.f;
#pragma unroll
        for (int m = 0; m < 4; m++) {  // word m = bytes 4m..4m+3 = k-steps 2m, 2m+1; block 2c + (m >= 2)
            uint32_t fa[4], fb[4];
            e2m1x8_to_f16x2x4(kAw[m], fa[0], fa[1], fa[2], fa[3]);
            e2m1x8_to_f16x2x4(kBw[m], fb[0], fb[1], fb[2], fb[3]);
            const uint32_t sa = m < 2 ? sA_lo : sA_hi, sb = m < 2 ? sB_lo : sB_hi;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                fa[e] = hmul2(fa[e], sa);
                fb[e] = hmul2(fb[e], sb);
            }
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                mma_f16_16816(sacc[0][nt], fa[0], fb[0], fa[1], fb[1], qf[nt][2 * m][0], qf[nt][2 * m][1]);
                mma_f16_16816(sacc[1][nt], fa[2], fb[2], fa[3], fb[3], qf[nt][2 * m + 1][0], qf[nt][2 * m + 1][1]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int e = 0; e < 4; e++) s[t][nt][e] = sacc[0][nt][e] + sacc[1][nt][e];
    }
    uint32_t pb[T][NT][2];
    softmax_tiles<NT, T, FULL>(s, g, vt, fac, m_run, o, pb);

    // ---- O^T += V^T P^T.  Lane owns channels 16g..16g+15 (block g) of tokens 2c, 2c+1, 2c+8, 2c+9.
#pragma unroll
    for (int t = 0; t < T; t++) {
        const uint8_t *gt = st + t * L::kBytes;
        const uint8_t *vrow = gt + L::kVq + (2 * c) * 64 + 8 * g;
        uint2 v0 = *reinterpret_cast<const uint2 *>(vrow);
        uint2 v1 = *reinterpret_cast<const uint2 *>(vrow + 64);
        uint2 v2 = *reinterpret_cast<const uint2 *>(vrow + 8 * 64);
        uint2 v3 = *reinterpret_cast<const uint2 *>(vrow + 9 * 64);
        const uint8_t *vs = gt + L::kVs + g * 16 + 2 * c;  // V scales [8][16]: rows 2c, 2c+1 and 2c+8, 2c+9
        uint32_t vs01 = *reinterpret_cast<const uint16_t *>(vs);
        uint32_t vs23 = *reinterpret_cast<const uint16_t *>(vs + 8);
        if (!FULL && vt[t] < 16) {  // rows past the end or not fetched may hold stale bytes: zero codes and scales
            const int j = 2 * c;
            if (j >= vt[t]) { v0 = make_uint2(0, 0); vs01 &= 0xff00u; }
            if (j + 1 >= vt[t]) { v1 = make_uint2(0, 0); vs01 &= 0x00ffu; }
            if (j + 8 >= vt[t]) { v2 = make_uint2(0, 0); vs23 &= 0xff00u; }
            if (j + 9 >= vt[t]) { v3 = make_uint2(0, 0); vs23 &= 0x00ffu; }
        }
        const uint32_t sv01 = e4m3x2_to_f16x2(vs01), sv23 = e4m3x2_to_f16x2(vs23);
        // swap nibbles so each byte holds (token a, token b) of one channel
        const uint32_t M = 0x0f0f0f0fu;
        const uint32_t E[4] = {bitsel(M, v0.x, v1.x << 4), bitsel(M, v0.y, v1.y << 4), bitsel(M, v2.x, v3.x << 4),
                               bitsel(M, v2.y, v3.y << 4)};
        const uint32_t O[4] = {bitsel(M, v0.x >> 4, v1.x), bitsel(M, v0.y >> 4, v1.y), bitsel(M, v2.x >> 4, v3.x),
                               bitsel(M, v2.y >> 4, v3.y)};
#pragma unroll
        for (int half = 0; half < 2; half++) {  // m-tiles 4*half .. 4*half+3
            uint32_t e01[4], o01[4], e23[4], o23[4];
            e2m1x8_to_f16x2x4(E[half], e01[0], e01[1], e01[2], e01[3]);
            e2m1x8_to_f16x2x4(O[half], o01[0], o01[1], o01[2], o01[3]);
            e2m1x8_to_f16x2x4(E[2 + half], e23[0], e23[1], e23[2], e23[3]);
            e2m1x8_to_f16x2x4(O[2 + half], o23[0], o23[1], o23[2], o23[3]);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int i = 4 * half + q;  // m-tile i: rows g -> channel 16g+2i, g+8 -> 16g+2i+1
                const uint32_t A0 = hmul2(e01[q], sv01), A1 = hmul2(o01[q], sv01);
                const uint32_t A2 = hmul2(e23[q], sv23), A3 = hmul2(o23[q], sv23);
#pragma unroll
                for (int nt = 0; nt < NT; nt++) mma_f16_16816(o[nt][i], A0, A1, A2, A3, pb[t][nt][0], pb[t][nt][1]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
            mma_f16_16816(o[nt][kLTile], kOnesF16x2, kOnesF16x2, kOnesF16x2, kOnesF16x2, pb[t][nt][0], pb[t][nt][1]);
    }
}

// One warp, one 16-token FP8 group.
template <int NT>
__device__ __forceinline__ void tile_fp8(const uint8_t *st, int vt, int lane, const uint32_t (&qf)[NT][8][2],
                                         const float (&fac)[NT][2], float (&m_run)[NT][2], float (&o)[NT][9][4]) {
    using L = Group<NVFP4KV_DTYPE_FP8_E4M3>;
    const int g = lane >> 2, c = lane & 3;
    uint32_t kA[8], kB[8];
    {
        const uint4 *pa = reinterpret_cast<const uint4 *>(st + L::kKq + g * 128 + 32 * c);
        const uint4 *pbk = reinterpret_cast<const uint4 *>(st + L::kKq + (g + 8) * 128 + 32 * c);
        const uint4 a0 = pa[0], a1 = pa[1], b0 = pbk[0], b1 = pbk[1];
        kA[0] = a0.x; kA[1] = a0.y; kA[2] = a0.z; kA[3] = a0.w; kA[4] = a1.x; kA[5] = a1.y; kA[6] = a1.z; kA[7] = a1.w;
        kB[0] = b0.x; kB[1] = b0.y; kB[2] = b0.z; kB[3] = b0.w; kB[4] = b1.x; kB[5] = b1.y; kB[6] = b1.z; kB[7] = b1.w;
    }
    float sacc[2][NT][4];
#pragma unroll
    for (int x = 0; x < 2; x++)
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int e = 0; e < 4; e++) sacc[x][nt][e] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) {  // word j = channels 32c+4j .. +3
        const uint32_t A0 = e4m3x2_to_f16x2(kA[j] & 0xffffu), A2 = e4m3x2_to_f16x2(kA[j] >> 16);
        const uint32_t A1 = e4m3x2_to_f16x2(kB[j] & 0xffffu), A3 = e4m3x2_to_f16x2(kB[j] >> 16);
#pragma unroll
        for (int nt = 0; nt < NT; nt++) mma_f16_16816(sacc[j & 1][nt], A0, A1, A2, A3, qf[nt][j][0], qf[nt][j][1]);
    }
    float s[1][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int e = 0; e < 4; e++) s[0][nt][e] = sacc[0][nt][e] + sacc[1][nt][e];
    uint32_t pb1[1][NT][2];
    const int vt1[1] = {vt};
    softmax_tiles<NT, 1>(s, g, vt1, fac, m_run, o, pb1);
    const uint32_t(&pb)[NT][2] = pb1[0];

    // V: lane owns channels 16g..16g+15 (16 bytes) of tokens 2c, 2c+1, 2c+8, 2c+9.
    const uint8_t *vrow = st + L::kVq + (2 * c) * 128 + 16 * g;
    uint4 v[4];
    v[0] = *reinterpret_cast<const uint4 *>(vrow);
    v[1] = *reinterpret_cast<const uint4 *>(vrow + 128);
    v[2] = *reinterpret_cast<const uint4 *>(vrow + 8 * 128);
    v[3] = *reinterpret_cast<const uint4 *>(vrow + 9 * 128);
    if (vt < 16) {
        const int rel[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
#pragma unroll
        for (int k = 0; k < 4; k++)
            if (rel[k] >= vt) v[k] = make_uint4(0, 0, 0, 0);
    }
    const uint32_t w0[4] = {v[0].x, v[0].y, v[0].z, v[0].w}, w1[4] = {v[1].x, v[1].y, v[1].z, v[1].w};
    const uint32_t w2[4] = {v[2].x, v[2].y, v[2].z, v[2].w}, w3[4] = {v[3].x, v[3].y, v[3].z, v[3].w};
#pragma unroll
    for (int i = 0; i < 8; i++) {  // m-tile i: channels 16g+2i (row g), 16g+2i+1 (row g+8)
        const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
        const uint32_t x01 = __byte_perm(w0[i >> 1], w1[i >> 1], sel);  // [t0 ch_e, t1 ch_e, t0 ch_o, t1 ch_o]
        const uint32_t x23 = __byte_perm(w2[i >> 1], w3[i >> 1], sel);
        const uint32_t A0 = e4m3x2_to_f16x2(x01 & 0xffffu), A1 = e4m3x2_to_f16x2(x01 >> 16);
        const uint32_t A2 = e4m3x2_to_f16x2(x23 & 0xffffu), A3 = e4m3x2_to_f16x2(x23 >> 16);
#pragma unroll
        for (int nt = 0; nt < NT; nt++) mma_f16_16816(o[nt][i], A0, A1, A2, A3, pb[nt][0], pb[nt][1]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
        mma_f16_16816(o[nt][kLTile], kOnesF16x2, kOnesF16x2, kOnesF16x2, kOnesF16x2, pb[nt][0], pb[nt][1]);
}

__device__ __forceinline__ void st_release_shared(int *p, int v) {
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_shared(const int *p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

// Bounded wait until chunk `want` has been issued into its stage (seq == want).
__device__ __forceinline__ bool wait_issued(const int *seq, int want, const volatile int *abort) {
    for (uint32_t it = 0; it < kWaitLimit; it++) {
        if (ld_acquire_shared(seq) == want) return true;
        if (*abort) return false;
        if (it > 64) __nanosleep(64);
    }
    return false;
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Fused append: the CTA that owns the last unit of a (sequence, kv_head) pair
// is the only one that reads the sequence's last token, so it quantises that
// token (16 threads per pair: K and V x 8 blocks) before any of its copies
// are issued.  Pairs are visited from the one holding unit u0 on.  Kept out
// of line: run once per warp pair, its quantiser code inlined into the kernel
// cost the main loop instruction-cache hits (the 32K decode kernel took 372
// instead of 365 us).
template <int DTYPE>
__device__ __noinline__ void fused_append(const DecodeArgs &a, int64_t u0, int64_t u1, int tid) {
    int lo = 0, hi = a.B - 1;  // the sequence holding unit u0
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)a.Hkv * chunk_prefix_at<DTYPE>(a, mid) <= u0) lo = mid;
        else hi = mid - 1;
    }
    const int64_t p_lo = chunk_prefix_at<DTYPE>(a, lo);
    const int nch0 = (int)(chunk_prefix_at<DTYPE>(a, lo + 1) - p_lo);
    const int64_t first_pair = (int64_t)lo * a.Hkv + (u0 - (int64_t)a.Hkv * p_lo) / nch0;
    const int part = tid & 15, which = part >> 3, blk = part & 7;
    for (int64_t p = first_pair + (tid >> 4);; p += kThreads / 16) {
        const int b = (int)(p / a.Hkv), kv = (int)(p - (int64_t)b * a.Hkv);
        if (b >= a.B) break;
        const int64_t pb = chunk_prefix_at<DTYPE>(a, b);
        const int64_t nch = chunk_prefix_at<DTYPE>(a, b + 1) - pb;
        const int64_t start = (int64_t)a.Hkv * pb + kv * nch;
        if (start >= u1) break;
        if (nch == 0 || start + nch - 1 >= u1) continue;  // its last unit belongs to a later CTA
        const int t = clamp_len(a.seq_lens[b], (int64_t)a.max_pages * a.P) - 1;
        const int32_t pg = __ldg(a.block_table + (int64_t)b * a.max_pages + (t >> a.log2P));
        if (pg < 0 || (int64_t)pg >= a.num_pages) {
            if (part == 0) flag_error(a.err, kErrPage);
            continue;
        }
        const uint4 *src = (which ? a.v_new : a.k_new) + (int64_t)b * a.new_stride16 + kv * (kHeadDim / 8) + blk * 2;
        uint8_t *slab = a.pool_w + ((int64_t)pg * a.Hkv + kv) * a.slab;
        if (a.unit_scale)
            store_block<true>(slab, a.dtype, t & (a.P - 1), which, blk, src, 1.0f);
        else
            store_block<false>(slab, a.dtype, t & (a.P - 1), which, blk, src, which ? a.gv_q : a.gk_q);
    }
}

// A CTA streams its contiguous range of 64-token units through a ring of
// kSlots stages shared by its kWarps warps: unit i of the range is computed
// by warp i % kWarps from stage i % kSlots, and the warp that used a stage
// refills it with unit i + kSlots.  Each warp keeps its own (max, sum, acc)
// per pair and leaves its own partial.
template <int DTYPE, int NT>
__global__ void __launch_bounds__(kThreads * Smem<DTYPE, NT>::kSubs, 1) decode_kernel(DecodeArgs a) {
    using S = Smem<DTYPE, NT>;
    extern __shared__ __align__(128) uint8_t smem_all[];
    // kSubs warp pairs per CTA, each with its own ring and its own range of
    // units (as a CTA of two warps would have): sub-CTA sub of CTA blockIdx.x
    // is unit range c = blockIdx.x * kSubs + sub of the split.
    const int sub = threadIdx.x / kThreads;
    const int tid = threadIdx.x % kThreads, lane = tid & 31, warp = tid >> 5;
    uint8_t *smem = smem_all + S::kPrefixBytes + sub * S::kSub;
    // chunk_prefix comes from the plan kernel, or, for a batch planned in the
    // CTA, from this CTA's own scan of seq_lens below.  Behind the
    // shared-prefix kernel, this grid starts only once every CTA of that
    // kernel has waited for the plan to complete (and flush) and then
    // triggered, so the plan's results are in global memory already and the
    // wait moves to the exit: the decode then runs beside the shared-prefix
    // kernel, and its own completion, which the reduction waits for, implies
    // that kernel's.
    if (!a.after_shared) pdl_wait();
    // The reduction may be scheduled once every CTA is past this point, so
    // with the plan (or, planned in the CTA, the work that wrote seq_lens)
    // complete: it reads chunk_prefix (or seq_lens) before its own wait.
    pdl_launch_dependents();

    if (a.plan_in_cta) {  // exclusive scan of the chunk counts, B <= 2 * kThreads (the first warp pair's threads)
        uint32_t *sp = reinterpret_cast<uint32_t *>(smem_all);
        uint32_t *wsum = reinterpret_cast<uint32_t *>(smem_all + S::kPrefixBytes);  // scratch: no copy issued yet
        const int64_t max_tokens = (int64_t)a.max_pages * a.P;
        const int b0 = 2 * tid, b1 = b0 + 1;
        uint32_t c0 = 0, c1 = 0;
        if (b0 < a.B) c0 = (uint32_t)seq_chunks(a.seq_lens[b0], max_tokens, 0);
        if (b1 < a.B) c1 = (uint32_t)seq_chunks(a.seq_lens[b1], max_tokens, 0);
        if (sub == 0 && blockIdx.x == 0 &&
            ((b0 < a.B && (a.seq_lens[b0] < 0 || (int64_t)a.seq_lens[b0] > max_tokens)) ||
             (b1 < a.B && (a.seq_lens[b1] < 0 || (int64_t)a.seq_lens[b1] > max_tokens))))
            flag_error(a.err, kErrSeqLen);
        uint32_t incl = c0 + c1;
#pragma unroll
        for (int x = 1; x < 32; x <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, x);
            if (lane >= x) incl += y;
        }
        if (sub == 0 && lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp > 0) incl += wsum[0];
        const uint32_t excl = incl - c0 - c1;
        if (sub == 0) {
            if (b0 < a.B) sp[b0] = excl;
            if (b1 < a.B) sp[b1] = excl + c0;
            if (tid == kThreads - 1) sp[a.B] = incl;
        }
        __syncthreads();
    }

    const int64_t U = (int64_t)a.Hkv * chunk_prefix_at<DTYPE>(a, a.B);
    const int64_t c = (int64_t)blockIdx.x * S::kSubs + sub;
    const int64_t u0 = c < a.grid ? c * U / a.grid : U, u1 = c < a.grid ? (c + 1) * U / a.grid : U;
    // a warp pair with no units (possible when grid > U, or past the grid in
    // the last CTA) skips to the end, where the CTA meets again
    const int nstages = (int)(u1 - u0);

    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kBars);
    int *valid = reinterpret_cast<int *>(smem + S::kFlags);
    int *seq = reinterpret_cast<int *>(smem + S::kSeq);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kAbort);

    if (tid == 0) {
        for (int s = 0; s < kSlots; s++) {
            mbar_init(&full[s], 1);
            valid[s] = 0;
            seq[s] = -1;
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (a.k_new && nstages > 0) {
        fused_append<DTYPE>(a, u0, u1, tid);
        fence_proxy_async_global();  // the stores above before this CTA's bulk reads of the same rows
    }
    __syncthreads();

    const int lnpp = a.P >= kChunk ? 0 : (a.P == 32 ? 1 : 2);
    const int npp = 1 << lnpp, upb = 32 >> lnpp;
    const int my_unit = lane >> lnpp, my_part = lane & (npp - 1);
    if (warp == 0) {  // the first kSlots units
        const uint64_t pro = my_unit < kSlots ? part_src<DTYPE>(a, u0, nstages, my_unit, my_part) : 0;
        const int first = nstages < kSlots ? nstages : kSlots;
        for (int s = 0; s < first; s++) {
            issue_stage<DTYPE>(a, pro, s << lnpp, npp, lane, ring + s * S::kStage, &full[s], &valid[s]);
            if (lane == 0) st_release_shared(&seq[s], s);
        }
    }

    // This warp computes units warp + k * kWarps (k = 0, 1, ...) and after
    // each refills its stage with unit warp + kSlots + k * kWarps.  Sources
    // of the refills: lane l resolves part l % npp of refill k0 + l / npp;
    // `cur` holds the batch of upb refills being issued, `nxt` the next one.
    auto refill_unit = [&](int k) { return warp + kSlots + k * kWarps; };
    uint64_t cur = part_src<DTYPE>(a, u0, nstages, refill_unit(my_unit), my_part);
    uint64_t nxt = part_src<DTYPE>(a, u0, nstages, refill_unit(upb + my_unit), my_part);

    Cursor cc;
    if (warp < nstages) {  // locate unit u0 + warp
        const int64_t uw = u0 + warp;
        int lo = 0, hi = a.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)a.Hkv * chunk_prefix_at<DTYPE>(a, mid) <= uw) lo = mid;
            else hi = mid - 1;
        }
        cc.b = lo;
        cursor_seq<DTYPE>(cc, a);
        const int rem = (int)(uw - (int64_t)a.Hkv * chunk_prefix_at<DTYPE>(a, lo));
        cc.kv = rem / cc.nch;
        cc.ch = rem - cc.kv * cc.nch;
    }

    uint32_t qf[NT][8][2];
    float fac[NT][2], m_run[NT][2], o[NT][9][4];
    int acc_pair = -1;  // pair (b * Hkv + kv, below 2^31) whose partial this warp is accumulating
    bool aborted = false;

    // this warp's partial of pair `pair`: (max, sum, acc)
    auto write_partial = [&](int pair) {
        const int g = lane >> 2, cq = lane & 3;
        const int64_t pidx = (c + pair) * kWarps + warp;
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
#pragma unroll
            for (int k = 0; k < 2; k++) {
                const int h = nt * 8 + 2 * cq + k;
                if (h >= a.G) continue;
                if (g == 0) a.part_ml[pidx * a.G + h] = make_float2(m_run[nt][k], o[nt][kLTile][k]);
                float *dst = a.part_acc + (pidx * a.G + h) * kHeadDim + 16 * g;
#pragma unroll
                for (int i2 = 0; i2 < 8; i2++)
                    *reinterpret_cast<float2 *>(dst + 2 * i2) = make_float2(o[nt][i2][k], o[nt][i2][k + 2]);
            }
        }
    };

    int k = 0;
    int slot = warp % kSlots;                     // i % kSlots
    uint32_t phase = (uint32_t)(warp / kSlots) & 1u;  // (i / kSlots) & 1
    for (int i = warp; i < nstages; i += kWarps, k++) {
        const int j = i + kSlots;  // refilled into this stage after this unit
        const bool refill = j < nstages;
        const int in_batch = k & (upb - 1);
        if (in_batch == 0 && k > 0) {  // entering the next batch of refills
            cur = nxt;
            nxt = part_src<DTYPE>(a, u0, nstages, refill_unit(k + upb + my_unit), my_part);
        }
        const int pair = cc.b * a.Hkv + cc.kv;
        if (pair != acc_pair) {  // this warp starts on a new (sequence, kv_head)
            if (acc_pair >= 0) write_partial(acc_pair);
            acc_pair = pair;
            load_q<NT>(a, cc.b, cc.kv, lane, qf, fac);
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                m_run[nt][0] = m_run[nt][1] = kNegInf;
#pragma unroll
                for (int q = 0; q < 9; q++) o[nt][q][0] = o[nt][q][1] = o[nt][q][2] = o[nt][q][3] = 0.f;
            }
        }
        bool ok = false;
        if (!aborted) {
            ok = wait_issued(&seq[slot], i, abort_flag) &&
                 mbar_wait_bounded(&full[slot], phase, kWaitLimit, abort_flag);
            if (!ok) {
                aborted = true;
                if (lane == 0) {
                    *abort_flag = 1;
                    flag_error(a.err, kErrTimeout);
                }
            }
        }
        const int mask = ok ? valid[slot] : 0;
        if (mask) {
            const int left = cc.n - a.skip - cc.ch * kChunk;
            const uint8_t *st = ring + slot * S::kStage;
            if (DTYPE == NVFP4KV_DTYPE_NVFP4 && left >= kChunk && mask == (1 << kGroups) - 1) {
                const int vt[kGroups] = {16, 16, 16, 16};  // a whole chunk: no masking
                tiles_nvfp4<NT, kGroups, true>(st, vt, lane, qf, fac, m_run, o);
            } else {
                int vt[kGroups];
#pragma unroll
                for (int t = 0; t < kGroups; t++) vt[t] = max(0, min(16, left - 16 * t));
                if (mask != (1 << min(kGroups, (left + 15) >> 4)) - 1) {  // a part was not fetched (bad page)
#pragma unroll
                    for (int t = 0; t < kGroups; t++)
                        if (!((mask >> t) & 1)) vt[t] = 0;
                }
                if (DTYPE == NVFP4KV_DTYPE_NVFP4) {
                    tiles_nvfp4<NT, kGroups, false>(st, vt, lane, qf, fac, m_run, o);
                } else {
#pragma unroll
                    for (int t = 0; t < kGroups; t++)
                        if (vt[t] > 0) tile_fp8<NT>(st + t * Group<DTYPE>::kBytes, vt[t], lane, qf, fac, m_run, o);
                }
            }
        }
        __syncwarp();
        if (refill && !aborted) {
            if (lane == 0) fence_proxy_async_smem();
            issue_stage<DTYPE>(a, cur, in_batch << lnpp, npp, lane, ring + slot * S::kStage, &full[slot],
                               &valid[slot]);
            if (lane == 0) st_release_shared(&seq[slot], j);
        }
        if (i + kWarps < nstages) cursor_advance<DTYPE>(cc, a, kWarps);
        slot += kWarps;
        if (slot >= kSlots) {
            slot -= kSlots;
            phase ^= 1u;
        }
    }
    if (acc_pair >= 0) write_partial(acc_pair);

    // After a timeout, no copy may still be writing shared memory when the
    // CTA exits: wait (bounded) for the last chunk issued into each stage.
    __syncthreads();
    if (*abort_flag && tid == 0) {
        for (int s = 0; s < kSlots; s++) {
            const int last = seq[s];
            if (last >= 0) mbar_wait_bounded(&full[s], (uint32_t)((last / kSlots) & 1), kWaitLimit, nullptr);
        }
    }
    if (a.after_shared) pdl_wait();
}

// Plan: chunk_prefix[b] = sum over b' < b of ceil((len(b') - skip) / 64); one CTA.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t *seq_lens, int B, int64_t max_tokens,
                                                    int64_t *prefix, unsigned *err, int skip) {
    __shared__ int64_t warp_sums[32];
    pdl_launch_dependents();  // let the decode kernel launch; it waits for this one to finish
    pdl_wait();               // seq_lens may come from earlier work on the stream
    const int tid = threadIdx.x;
    const int per = (B + 1023) / 1024;
    const int lo = min(B, tid * per), hi = min(B, lo + per);
    int64_t local = 0;
    for (int b = lo; b < hi; b++) {
        const int32_t n = seq_lens[b];
        if (n < skip || (int64_t)n > max_tokens) flag_error(err, kErrSeqLen);
        local += seq_chunks(n, max_tokens, skip);
    }
    // block-wide exclusive scan of `local`
    const int lane = tid & 31, warp = tid >> 5;
    int64_t incl = local;
#pragma unroll
    for (int x = 1; x < 32; x <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, x);
        if (lane >= x) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int64_t v = warp_sums[lane];
#pragma unroll
        for (int x = 1; x < 32; x <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, v, x);
            if (lane >= x) v += y;
        }
        warp_sums[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    int64_t run = incl - local + (warp > 0 ? warp_sums[warp - 1] : 0);
    for (int b = lo; b < hi; b++) {
        prefix[b] = run;
        run += seq_chunks(seq_lens[b], max_tokens, skip);
    }
    if (tid == 1023) prefix[B] = warp_sums[31];
}

struct ReduceArgs {
    int B, Hq, Hkv, G, grid;
    const int64_t *chunk_prefix;  // nullptr: the batch was planned in the decode CTAs (plan from seq_lens here)
    const int32_t *seq_lens;
    int64_t max_tokens;
    const float *part_acc;
    const float2 *part_ml;
    const float *casc_acc;  // shared-prefix partials [casc_splits][B * Hkv][G] (nullptr: none)
    const float2 *casc_ml;
    int casc_splits;
    float gv;
    __nv_bfloat16 *out;
};

// Log-sum-exp merge of the partials of every CTA that covered a pair, then
// normalisation and the V tensor scale.  A CTA of kReduceWarps warps serves
// kReduceWarps / wpr output rows (sequence, query head) with wpr warps each:
// the warps of a row split its partials (every wpr-th one, four loads in
// flight), each keeping a running (max, sum, acc) with lane l owning dims
// 4l..4l+3, and merge through shared memory.  The host picks wpr from the
// average number of partials per pair: one warp per row when pairs are
// covered by a handful of CTAs, all eight when a few long sequences are
// spread over hundreds.
constexpr int kReduceWarps = 8;

__device__ __forceinline__ float lse_factor(float m, float mx) { return m == kNegInf ? 0.f : ex2(m - mx); }

// n / d for n >= 0, d > 0; in 32 bits when both fit, the usual case.
__device__ __forceinline__ int64_t udiv64(int64_t n, int64_t d) {
    if ((((uint64_t)n | (uint64_t)d) >> 32) == 0) return (int64_t)((uint32_t)n / (uint32_t)d);
    return n / d;
}

__global__ void __launch_bounds__(32 * kReduceWarps) reduce_kernel(ReduceArgs a, int wpr) {
    __shared__ float4 s_acc[kReduceWarps][32];
    __shared__ float s_m[kReduceWarps], s_l[kReduceWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = (int64_t)blockIdx.x * (kReduceWarps / wpr) + warp / wpr;
    const int sub = warp % wpr;  // this warp's share of the row's partials
    const bool live = row < (int64_t)a.B * a.Hq;
    // Where the row's pair p = b * Hkv + kv lies, found before the wait: the
    // decode kernel lets this grid launch only once the plan that wrote
    // chunk_prefix is complete, so the arithmetic overlaps the decode's last
    // CTAs (loads through L2: the values come from an earlier grid).  The
    // pair's units [off, off + nch) of the flat order are covered by CTAs
    // c0 .. c1, CTA c owning units [c U / grid, (c + 1) U / grid); lo0 .. hi0
    // are the pair's units within CTA c0's range, 0 .. hi1 within CTA c1's.
    int b = 0, kv = 0, hh = 0;
    int64_t p = 0, U = 0, nch = 0, off = 0, c0 = 0, c1 = -1, lo0 = 0, hi0 = 0, hi1 = 0;
    if (live) {
        b = (int)(row / a.Hq);
        const int h = (int)(row % a.Hq);
        kv = h / a.G;
        hh = h % a.G;
        p = (int64_t)b * a.Hkv + kv;
        int64_t pb = 0, total = 0;
        if (a.chunk_prefix) {
            const long long *cp = reinterpret_cast<const long long *>(a.chunk_prefix);
            pb = __ldcg(cp + b);
            nch = __ldcg(cp + b + 1) - pb;
            total = __ldcg(cp + a.B);
        } else {  // the warp scans the chunk counts itself, as each decode CTA did (row, so b, is warp-uniform)
            for (int base = 0; base < a.B; base += 32) {
                const int bb = base + lane;
                const uint32_t cnt = bb < a.B ? (uint32_t)seq_chunks(a.seq_lens[bb], a.max_tokens, 0) : 0u;
                uint32_t incl = cnt;
#pragma unroll
                for (int x = 1; x < 32; x <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, x);
                    if (lane >= x) incl += y;
                }
                const int in_seg = b - base;
                if (in_seg >= 0 && in_seg < 32) {
                    pb = total + (int64_t)__shfl_sync(0xffffffffu, incl - cnt, in_seg);
                    nch = (int64_t)__shfl_sync(0xffffffffu, cnt, in_seg);
                }
                total += (int64_t)__shfl_sync(0xffffffffu, incl, 31);
            }
        }
        U = (int64_t)a.Hkv * total;
        if (nch > 0) {
            off = (int64_t)a.Hkv * pb + (int64_t)kv * nch;
            c0 = udiv64((off + 1) * a.grid - 1, U);
            c1 = udiv64((off + nch) * a.grid - 1, U);
            const int64_t a0 = udiv64(c0 * U, a.grid), e0 = udiv64((c0 + 1) * U, a.grid);
            lo0 = off - a0;
            hi0 = (off + nch < e0 ? off + nch : e0) - a0;
            hi1 = off + nch - udiv64(c1 * U, a.grid);
        }
    }
    // With every CTA's range at least two units long, a CTA strictly between
    // c0 and c1 holds two or more of the pair's units, so both of its warps
    // left a partial; otherwise each candidate CTA's range is recomputed.
    const bool dense = U >= 2 * (int64_t)a.grid;
    pdl_wait();  // partials come from the decode kernel
    float m_w = kNegInf, l_w = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
        const int64_t ncasc = a.casc_ml ? a.casc_splits : 0;
        // Candidate partials: first the ncasc shared-prefix partials of the pair,
        // then (CTA cc, warp w) for cc in [c0, c1].  Warp w of CTA cc left one iff
        // the CTA's units of this pair include one with index (within the CTA's
        // range) = w mod kWarps; an empty CTA (possible when grid > U) left none.
        auto left_one = [](int64_t lo, int64_t hi, int w) {
            if (hi <= lo) return false;
            return hi - lo > (int64_t)((w - lo % kWarps + kWarps) % kWarps);
        };
        auto has_partial = [&](int64_t cc, int w) {
            if (dense) {
                if (cc == c0) return left_one(lo0, hi0, w);
                if (cc == c1) return left_one(0, hi1, w);
                return true;
            }
            const int64_t cu0 = udiv64(cc * U, a.grid), cu1 = udiv64((cc + 1) * U, a.grid);
            return left_one((off > cu0 ? off : cu0) - cu0, (off + nch < cu1 ? off + nch : cu1) - cu0, w);
        };
        const int64_t ncand = ncasc + (c1 - c0 + 1) * kWarps;
        for (int64_t base = sub; base < ncand; base += 4 * wpr) {
            float2 ml[4];
            float4 v[4];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int64_t q = base + (int64_t)k * wpr;
                ml[k] = make_float2(kNegInf, 0.f);
                v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (q < ncasc) {
                    const int64_t idx = (q * a.B * a.Hkv + p) * a.G + hh;
                    ml[k] = a.casc_ml[idx];
                    v[k] = reinterpret_cast<const float4 *>(a.casc_acc + idx * kHeadDim)[lane];
                } else if (q < ncand) {
                    const int64_t cc = c0 + (q - ncasc) / kWarps;
                    const int w = (int)((q - ncasc) % kWarps);
                    if (has_partial(cc, w)) {
                        const int64_t idx = ((cc + p) * kWarps + w) * a.G + hh;
                        ml[k] = a.part_ml[idx];
                        v[k] = reinterpret_cast<const float4 *>(a.part_acc + idx * kHeadDim)[lane];
                    }
                }
            }
            float mx = m_w;
#pragma unroll
            for (int k = 0; k < 4; k++) mx = fmaxf(mx, ml[k].x);
            const float f0 = lse_factor(m_w, mx);
            l_w *= f0;
            acc.x *= f0;
            acc.y *= f0;
            acc.z *= f0;
            acc.w *= f0;
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const float f = lse_factor(ml[k].x, mx);
                l_w += f * ml[k].y;
                acc.x += f * v[k].x;
                acc.y += f * v[k].y;
                acc.z += f * v[k].z;
                acc.w += f * v[k].w;
            }
            m_w = mx;
        }
    }
    if (wpr > 1) {
        s_acc[warp][lane] = acc;
        if (lane == 0) {
            s_m[warp] = m_w;
            s_l[warp] = l_w;
        }
        __syncthreads();
        if (sub != 0) return;
        float mx = kNegInf;
        for (int w = 0; w < wpr; w++) mx = fmaxf(mx, s_m[warp + w]);
        l_w = 0.f;
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < wpr; w++) {
            const float f = lse_factor(s_m[warp + w], mx);
            const float4 v = s_acc[warp + w][lane];
            l_w += f * s_l[warp + w];
            acc.x += f * v.x;
            acc.y += f * v.y;
            acc.z += f * v.z;
            acc.w += f * v.w;
        }
    }
    if (!live) return;
    const float inv = l_w > 0.f ? a.gv / l_w : 0.f;  // a sequence of length 0 gets zeros
    const __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2 *>(a.out + row * kHeadDim)[lane] =
        make_uint2(*reinterpret_cast<const uint32_t *>(&lo2), *reinterpret_cast<const uint32_t *>(&hi2));
}

template <int DTYPE, int NT>
const void *kernel_fn() {
    return reinterpret_cast<const void *>(&decode_kernel<DTYPE, NT>);
}

// smem_bytes: the dynamic shared memory of every launch; subs: warp pairs per CTA.
const void *select_kernel(int dtype, int nt, int *smem_bytes, int *subs = nullptr) {
    int dummy = 0;
    int &n = subs ? *subs : dummy;
    if (dtype == NVFP4KV_DTYPE_NVFP4) {
        if (nt == 1) {
            *smem_bytes = Smem<0, 1>::kMax;
            n = Smem<0, 1>::kSubs;
            return kernel_fn<0, 1>();
        }
        *smem_bytes = Smem<0, 2>::kMax;
        n = Smem<0, 2>::kSubs;
        return kernel_fn<0, 2>();
    }
    if (nt == 1) {
        *smem_bytes = Smem<1, 1>::kMax;
        n = Smem<1, 1>::kSubs;
        return kernel_fn<1, 1>();
    }
    *smem_bytes = Smem<1, 2>::kMax;
    n = Smem<1, 2>::kSubs;
    return kernel_fn<1, 2>();
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_auto_grid[kMaxDevices][2][2];   // [device][dtype][nt-1], 0 = unknown
bool g_attr_set[kMaxDevices][2][2];

cudaError_t prepare_kernel(int dtype, int nt, int *grid_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    int smem = 0, subs = 1;
    const void *fn = select_kernel(dtype, nt, &smem, &subs);
    if (!g_attr_set[dev][dtype][nt - 1]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        g_attr_set[dev][dtype][nt - 1] = true;
    }
    if (!g_auto_grid[dev][dtype][nt - 1]) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads * subs, smem);
        if (e != cudaSuccess) return e;
        g_auto_grid[dev][dtype][nt - 1] = sms * (per_sm > 0 ? per_sm : 1) * subs;
    }
    if (grid_out) *grid_out = g_auto_grid[dev][dtype][nt - 1];
    return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

bool decode_plans_in_cta(int batch, bool shared_prefix) { return !shared_prefix && batch <= kPlanInCta; }

int decode_auto_grid(const nvfp4kv_cache &c, int group, cudaError_t *status) {
    int grid = 0;
    cudaError_t e = prepare_kernel(c.dtype, group <= 8 ? 1 : 2, &grid);
    if (status) *status = e;
    return e == cudaSuccess ? grid : 0;
}

// Workspace: chunk prefix | per-warp partials (m, l) | their acc; a cascade
// call appends the shared-prefix partials (m, l) | their acc.
size_t decode_workspace_bytes(const nvfp4kv_cache &c, int batch, int num_q_heads, int grid) {
    const int G = num_q_heads / c.num_kv_heads;
    const size_t slots = ((size_t)grid + (size_t)batch * c.num_kv_heads) * kWarps;
    return align256(sizeof(int64_t) * ((size_t)batch + 1)) + align256(sizeof(float2) * slots * G) +
           sizeof(float) * slots * G * kHeadDim;
}

size_t cascade_extra_bytes(const nvfp4kv_cache &c, int batch, int num_q_heads, int shared_len) {
    const size_t n = (size_t)cascade_splits(c, batch, num_q_heads, shared_len) * batch * num_q_heads;
    return align256(sizeof(float2) * n) + sizeof(float) * n * kHeadDim;
}

cudaError_t launch_decode(const nvfp4kv_cache &c, const void *q, int batch, int num_q_heads,
                          const int32_t *block_table, int max_pages, const int32_t *seq_lens, float sm_scale,
                          void *out, void *workspace, int grid, unsigned *err, cudaStream_t stream,
                          cudaEvent_t before, cudaEvent_t after, const void *k_new, const void *v_new,
                          int64_t new_stride, const int32_t *shared_pages, int shared_len) {
    const int G = num_q_heads / c.num_kv_heads;
    const int nt = G <= 8 ? 1 : 2;
    cudaError_t e = prepare_kernel(c.dtype, nt, nullptr);
    if (e != cudaSuccess) return e;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t slots = ((size_t)grid + (size_t)batch * c.num_kv_heads) * kWarps;
    int64_t *prefix = reinterpret_cast<int64_t *>(ws);
    float2 *part_ml = reinterpret_cast<float2 *>(ws + align256(sizeof(int64_t) * ((size_t)batch + 1)));
    float *part_acc = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(part_ml) + align256(sizeof(float2) * slots * G));
    const int csplits = shared_pages ? cascade_splits(c, batch, num_q_heads, shared_len) : 0;
    float2 *casc_ml = reinterpret_cast<float2 *>(part_acc + slots * G * kHeadDim);
    float *casc_acc = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(casc_ml) +
                                                align256(sizeof(float2) * (size_t)csplits * batch * num_q_heads));
    const int skip = shared_pages ? shared_len : 0;
    int64_t max_tokens = (int64_t)max_pages * c.page_size;
    // A small batch is planned in every decode CTA; otherwise by the plan kernel.
    const bool plan_in_cta = decode_plans_in_cta(batch, shared_pages != nullptr);
    if (!plan_in_cta) {
        int skip_arg = skip;
        void *pargs[] = {&seq_lens, &batch, &max_tokens, &prefix, &err, &skip_arg};
        e = launch_pdl(reinterpret_cast<const void *>(&plan_kernel), 1, 1024, 0, stream, pargs);
        if (e != cudaSuccess) return e;
    }
    if (shared_pages) {  // attention of every sequence's queries over the shared prefix, once per kv head
        e = launch_shared_prefix(c, q, batch, num_q_heads, shared_pages, shared_len, csplits, sm_scale, casc_ml,
                                 casc_acc, err, stream);
        if (e != cudaSuccess) return e;
    }

    DecodeArgs a;
    a.pool = static_cast<const uint8_t *>(c.pool);
    a.num_pages = c.num_pages;
    a.P = c.page_size;
    a.log2P = __builtin_ctz((unsigned)c.page_size);
    a.Hkv = c.num_kv_heads;
    a.G = G;
    a.Hq = num_q_heads;
    a.B = batch;
    a.max_pages = max_pages;
    a.slab = (int64_t)(c.dtype == NVFP4KV_DTYPE_NVFP4 ? 144 : 256) * c.page_size;
    a.q = static_cast<const uint4 *>(q);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.chunk_prefix = prefix;
    a.plan_in_cta = plan_in_cta ? 1 : 0;
    a.score_log2 = (float)((double)sm_scale * (double)c.k_global_scale * 1.4426950408889634);
    a.gv = c.v_global_scale;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.part_acc = part_acc;
    a.part_ml = part_ml;
    a.grid = grid;
    a.err = err;
    a.k_new = static_cast<const uint4 *>(k_new);
    a.v_new = static_cast<const uint4 *>(v_new);
    a.new_stride16 = new_stride / 8;
    a.gk_q = c.k_global_scale;
    a.gv_q = c.v_global_scale;
    a.dtype = c.dtype;
    a.unit_scale = c.k_global_scale == 1.0f && c.v_global_scale == 1.0f;
    a.pool_w = static_cast<uint8_t *>(c.pool);
    a.skip = skip;
    a.after_shared = shared_pages ? 1 : 0;
    int smem = 0, subs = 1;
    const void *fn = select_kernel(c.dtype, nt, &smem, &subs);
    void *args[] = {&a};
    if (before && (e = cudaEventRecord(before, stream)) != cudaSuccess) return e;
    e = launch_pdl(fn, (unsigned)ceil_div64(grid, subs), kThreads * subs, (size_t)smem, stream, args);
    if (e != cudaSuccess) return e;
    if (after && (e = cudaEventRecord(after, stream)) != cudaSuccess) return e;

    ReduceArgs r;
    r.B = batch;
    r.Hq = num_q_heads;
    r.Hkv = c.num_kv_heads;
    r.G = G;
    r.grid = grid;
    r.chunk_prefix = plan_in_cta ? nullptr : prefix;
    r.seq_lens = seq_lens;
    r.max_tokens = max_tokens;
    r.part_acc = part_acc;
    r.part_ml = part_ml;
    r.casc_ml = shared_pages ? casc_ml : nullptr;
    r.casc_acc = shared_pages ? casc_acc : nullptr;
    r.casc_splits = csplits;
    r.gv = c.v_global_scale;
    r.out = static_cast<__nv_bfloat16 *>(out);
    const int64_t rows = (int64_t)batch * num_q_heads;
    // warps per output row from the average number of partials per pair
    const int64_t pairs = (int64_t)batch * c.num_kv_heads;
    const int64_t avg_parts = (grid + 2 * pairs - 1) / pairs * kWarps + csplits;
    int wpr = avg_parts <= 8 ? 1 : avg_parts <= 16 ? 2 : avg_parts <= 32 ? 4 : 8;
    const int64_t rows_per_cta = kReduceWarps / wpr;
    void *rargs[] = {&r, &wpr};
    return launch_pdl(reinterpret_cast<const void *>(&reduce_kernel), (unsigned)ceil_div64(rows, rows_per_cta),
                      32 * kReduceWarps, 0, stream, rargs);
}

}  // namespace nvfp4kv
