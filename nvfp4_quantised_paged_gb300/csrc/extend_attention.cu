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
// A dependent chain of tcgen05.mma (the K = 16 steps of one product into one
// accumulator) runs at the tensor core's rate only when each instruction is
// large: M 128 x N 64 steps are latency-bound at about a third of it, N 128
// close to it.  So K/V tiles are 128 keys, and each CTA holds two 128-row
// query tiles whose four products per K/V tile (S0, S1, O0 += P0 V, O1 +=
// P1 V) are independent chains that the tensor core overlaps.
//
// One CTA = 256 query rows of one (request, kv head), row = chunk token * G +
// query head of the group, so the G heads that share a KV head share every
// K/V tile; one CTA per SM (193 KB of shared memory, 211 KB with the paged
// prefix; all 512 TMEM columns).  Nine warps (twelve with the paged prefix):
//   * warpgroup w (warps 4w .. 4w + 3, w = 0, 1), one thread per row of query
//     tile w = one TMEM lane, runs the softmax of that tile: wait for S_w(j)
//     (128 scores per row, FP32 in TMEM columns 128w ..), load it, mask edge
//     tiles only, base-2 online softmax with a lazily updated running max
//     (O_w in TMEM is rescaled only when a score exceeds the max by 2^8),
//     P = 2^(s * scale - m) rounded to BF16 and stored over the first half of
//     S_w's columns, the row sum of the rounded P kept in a register (the
//     numerator and the denominator see the same P); then signal P_w(j);
//   * one thread of warp 8 drives the TMA loads (3-D tensor maps, 128-byte
//     swizzle = the tensor core's canonical operand layout) and the MMAs, per
//     K/V tile j: S0(j) = Q0 K(j)^T and S1(j) = Q1 K(j)^T (eight M 128 x N 128
//     x K 16 steps each), then O_w += P_w(j) V(j) as P_w(j) arrives (eight
//     steps over the 128 keys, P read from TMEM, V an MN-major operand).
//     S_w(j + 1) waits for O_w += P_w(j) V(j), whose P shares its columns, so
//     while warpgroup 0 works on tile j + 1 the tensor core runs the products
//     of query tile 1, and the other way round.
// K and V have two-slot rings each; K(j + 2) is requested once S1(j) is done,
// V(j + 1) once O1 += P1(j - 1) V(j - 1) is done.  The MMA thread issues
// whatever is ready for either query tile, polling the barriers.
//
// Two instantiations: the prefix as BF16 workspace rows loaded by TMA
// (extend_kernel<false>), or read from the NVFP4 pages of the cache
// (extend_kernel<true>): seven more warps then bulk-copy each prefix tile's
// NVFP4 groups into raw shared-memory stages and expand them into the K / V
// slots in BF16 (as the prefix dequant kernel would), so the result is the
// same bit for bit and no workspace is written.  Every wait is bounded; a
// timeout is recorded in the device error word and ends every warp's loop.
#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "quantize.cuh"
#include "tcgen05.cuh"

namespace nvfp4kv {

namespace {

constexpr int kWGs = 2;                        // softmax warpgroups = query tiles per CTA
constexpr int kQRows = 128;                    // rows per query tile (one TMEM lane each)
constexpr int kCtaRows = kWGs * kQRows;
constexpr int kSoftThreads = kWGs * kQRows;
constexpr int kEThreads = kSoftThreads + 32;   // + the load / MMA warp
constexpr int kDqThreads = 224;                // paged prefix: seven warps expanding NVFP4 tiles
constexpr int kEThreadsPaged = kEThreads + kDqThreads;
// The paged instantiation is launched with 512 threads at 128 registers each;
// the two softmax warpgroups then take 152 and the other two (the load / MMA
// warp and the seven expanding warps) give back down to 104: 8 warps x 32 x
// 152 + 8 warps x 32 x 104 = 65,536, exactly the registers the CTA holds.
constexpr int kSoftRegs = 152, kOtherRegs = 104;
static_assert(kEThreadsPaged == 512 && (kSoftThreads / 32) * kSoftRegs + (kEThreadsPaged - kSoftThreads) / 32 * kOtherRegs ==
                                           (kEThreadsPaged / 32) * 128,
              "register split of the paged instantiation must add up to its launch");
constexpr int kKeys = 128;                     // keys per K/V tile
constexpr int kQBytes = kQRows * 256;          // a query tile: 2 column blocks of [128][64] BF16
constexpr int kKVBlock = kKeys * 128;          // one column block of a K or V tile (one TMA box)
constexpr int kKVTile = 2 * kKVBlock;          // a whole K (or V) tile, 32 KB
constexpr int kOffQ = 0;                                   // Q0 | Q1
constexpr int kOffK = kWGs * kQBytes;                      // K slots [2]
constexpr int kOffV = kOffK + 2 * kKVTile;                 // V slots [2]
constexpr int kOffBar = kOffV + 2 * kKVTile;
// mbarriers: k_full[2] v_full[2] s_done[2] p_full[2] pv_done[2] drain, and for a
// paged prefix k_go[2] v_go[2] (tile may be expanded) k_dq[2] v_dq[2] (expanded)
// rawk_full rawv_full[2] (raw halves landed) rawk_free rawv_free[2] (read)
constexpr int kNumBars = 25;
constexpr int kOffTmem = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmem + 4;
constexpr int kOffOrder = kOffBar + 256;       // int[256]: requests by decreasing prefix length
constexpr int kOrderMax = 256;
constexpr int kESmem = kOffOrder + 4 * kOrderMax;
// paged prefix: raw stages of a tile's NVFP4 groups, the K halves (codes and
// scales, 1,152 B of each 2,304-B group) single, the V halves double-buffered
// (V is needed a softmax later than K, so its copies get the longer lead)
constexpr int kGroupBytes = 2304, kHalfGroup = 1152;
constexpr int kRawHalf = 8 * kHalfGroup;       // one tile's K (or V) halves
constexpr int kOffRawK = kESmem;
constexpr int kOffRawV = kOffRawK + kRawHalf;  // [2]
constexpr int kESmemPaged = kOffRawV + 2 * kRawHalf;
static_assert(kOffRawK % 16 == 0 && kRawHalf % 16 == 0, "bulk copies need 16-byte aligned destinations");
static_assert(kESmemPaged <= 227 * 1024, "paged extend exceeds the shared memory of a CTA");
// TMEM columns: S_w at 128w (FP32; P_w as BF16 pairs over its first 64 columns), O_w at 256 + 128w
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescale = 8.0f;
constexpr float kNegInfE = -__builtin_huge_valf();
constexpr uint32_t kWaitLimitE = 1u << 24;

struct ExtendArgs {
    const uint16_t *q;                 // BF16 [total_q][Hq][128]
    const int32_t *cu_prefix, *cu_q;   // [num_reqs + 1]
    int Hq, Hkv, G, max_q_len;
    float score_log2;                  // sm_scale * log2(e)
    uint16_t *out;                     // BF16 [total_q][Hq][128]
    unsigned *err;
    // paged prefix: request r's prefix is tokens 0 .. prefix_lens[r] - 1 of its
    // pages in the NVFP4 pool (block_table row r), not workspace rows
    const uint8_t *pool;
    int64_t num_pages, slab;
    int P, log2P, max_pages;
    const int32_t *block_table, *prefix_lens;
    float gk, gv;
};

// K/V tensors [rows][Hkv][128] BF16 as 3-D TMA maps with 64 x 1 x 128 boxes, 128-byte swizzle.
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


// Bounded wait on an mbarrier phase without sleeping between polls (these
// waits are on the critical path); gives up when another warp has aborted.
__device__ __forceinline__ bool spin_wait(uint64_t *bar, uint32_t parity, const volatile int *abort_flag) {
    for (uint32_t n = 0; n < kWaitLimitE; n++) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    return false;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (a.x * b + c, a.y * b + c) in one instruction
__device__ __forceinline__ float2 fma2(float2 a, float b, float c) {
    uint64_t d;
    const uint64_t bb = (uint64_t)__float_as_uint(b) | ((uint64_t)__float_as_uint(b) << 32);
    const uint64_t cc = (uint64_t)__float_as_uint(c) | ((uint64_t)__float_as_uint(c) << 32);
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"((uint64_t)__float_as_uint(a.x) | ((uint64_t)__float_as_uint(a.y) << 32)), "l"(bb), "l"(cc));
    return make_float2(__uint_as_float((uint32_t)d), __uint_as_float((uint32_t)(d >> 32)));
}

// s0 += low BF16 of w, s1 += high BF16 of w (exact products by 1.0, FP32 sums)
__device__ __forceinline__ void add_bf16x2(float &s0, float &s1, uint32_t w) {
    const unsigned short one = 0x3f80;
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2;\n"
        "fma.rn.f32.bf16 %0, lo, %3, %0; fma.rn.f32.bf16 %1, hi, %3, %1; }"
        : "+f"(s0), "+f"(s1)
        : "r"(w), "h"(one));
}

template <bool kPaged>
__global__ void __launch_bounds__(kPaged ? kEThreadsPaged : kEThreads, 1)
    extend_kernel(const __grid_constant__ ExtendMaps maps, ExtendArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *k_full = bars, *v_full = bars + 2, *s_done = bars + 4, *p_full = bars + 6, *pv_done = bars + 8;
    uint64_t *drain = bars + 10, *k_go = bars + 11, *v_go = bars + 13, *k_dq = bars + 15, *v_dq = bars + 17;
    uint64_t *rawk_full = bars + 19, *rawv_full = bars + 20, *rawk_free = bars + 22, *rawv_free = bars + 23;
    uint32_t &tmem_base = *reinterpret_cast<uint32_t *>(smem + kOffTmem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffAbort);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Requests in order of decreasing prefix length (the longest CTAs start
    // first, so the tail of the grid holds short ones): blockIdx.z is the
    // rank; thread j ranks request j.
    int r = blockIdx.z;
    if (gridDim.z <= kOrderMax) {
        int *order = reinterpret_cast<int *>(smem + kOffOrder);
        const int nr = (int)gridDim.z;
        auto prefix_len = [&](int c) { return kPaged ? a.prefix_lens[c] : a.cu_prefix[c + 1] - a.cu_prefix[c]; };
        if (tid < nr) {
            const int nj = prefix_len(tid);
            int rank = 0;
            for (int c = 0; c < nr; c++) {
                const int nc = prefix_len(c);
                rank += nc > nj || (nc == nj && c < tid);
            }
            order[rank] = tid;
        }
        __syncthreads();
        r = order[blockIdx.z];
    }
    const int kv = blockIdx.y;
    const int q0 = a.cu_q[r], p0 = kPaged ? 0 : a.cu_prefix[r];
    int L = a.cu_q[r + 1] - q0;
    int np = kPaged ? a.prefix_lens[r] : a.cu_prefix[r + 1] - p0;
    if (L < 0 || np < 0) {
        if (tid == 0 && blockIdx.x == 0 && kv == 0) flag_error(a.err, kErrCuPrefix);
        return;
    }
    if (kPaged && (int64_t)np > (int64_t)a.max_pages * a.P) {
        if (tid == 0 && blockIdx.x == 0 && kv == 0) flag_error(a.err, kErrSeqLen);
        np = a.max_pages * a.P;
    }
    if (L > a.max_q_len) {
        if (tid == 0 && blockIdx.x == 0 && kv == 0) flag_error(a.err, kErrSeqLen);
        L = a.max_q_len;
    }
    const int rows = L * a.G;
    const int row0 = blockIdx.x * kCtaRows;
    if (row0 >= rows) return;
    const int nwg = row0 + kQRows < rows ? 2 : 1;               // query tiles holding rows
    const int t_last = (min(row0 + kCtaRows, rows) - 1) / a.G;  // last chunk token of this CTA
    const int nt_pre = (np + kKeys - 1) / kKeys;
    const int nt = nt_pre + t_last / kKeys + 1;

    const uint32_t sbase = smem_u32(smem);

    // ---- query tiles: 128 rows x 16 chunks of 16 bytes each, by their warpgroups
    if (tid < kSoftThreads) {
        const int w = tid >> 7, t = tid & 127;
        const uint32_t sQ = sbase + kOffQ + w * kQBytes;
#pragma unroll 4
        for (int it = 0; it < 16; it++) {
            const int idx = t + it * kQRows;
            const int row = idx >> 4, c16 = idx & 15;
            const int R = row0 + w * kQRows + row;
            const bool ok = R < rows;
            const int64_t src = ok ? (((int64_t)q0 + R / a.G) * a.Hq + kv * a.G + R % a.G) * kHeadDim + c16 * 8 : 0;
            cp_async16(sQ + (c16 >> 3) * (kQRows * 128) + sw128_off(row, c16 & 7), a.q + src, ok);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    // K (or V) of tile j into slot s: two TMA boxes (head_dim 0..63 and
    // 64..127) of 128 rows; rows past the tensor are zero-filled, rows of a
    // neighbouring request are masked by the softmax
    auto tile_row = [&](int j) { return j < nt_pre ? p0 + j * kKeys : q0 + (j - nt_pre) * kKeys; };
    // (paged prefix: the tile is expanded by the dequantising warps instead,
    // told to start by its go barrier; they complete the same full barrier)
    auto load_k = [&](int j, int s) {
        if (kPaged && j < nt_pre) {
            mbar_arrive(&k_go[s]);
            return;
        }
        const CUtensorMap *m = j < nt_pre ? &maps.k_pre : &maps.k_new;
        const uint32_t dst = sbase + kOffK + s * kKVTile;
        mbar_arrive_expect_tx(&k_full[s], kKVTile);
        tma_load_3d(dst, m, 0, kv, tile_row(j), &k_full[s]);
        tma_load_3d(dst + kKVBlock, m, 64, kv, tile_row(j), &k_full[s]);
    };
    auto load_v = [&](int j, int s) {
        if (kPaged && j < nt_pre) {
            mbar_arrive(&v_go[s]);
            return;
        }
        const CUtensorMap *m = j < nt_pre ? &maps.v_pre : &maps.v_new;
        const uint32_t dst = sbase + kOffV + s * kKVTile;
        mbar_arrive_expect_tx(&v_full[s], kKVTile);
        tma_load_3d(dst, m, 0, kv, tile_row(j), &v_full[s]);
        tma_load_3d(dst + kKVBlock, m, 64, kv, tile_row(j), &v_full[s]);
    };

    if (warp == 0) tc_alloc(&tmem_base, kTmemCols);
    if (tid == kSoftThreads) {
        for (int j = 0; j < kNumBars; j++)
            mbar_init(&bars[j], (j == 6 || j == 7) ? kQRows : ((j >= 15 && j < 19) || j >= 22) ? kDqThreads : 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int j = 0; j < 2 && j < nt; j++) {
            load_k(j, j);
            load_v(j, j);
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q for the tensor core
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    // The register split of the paged instantiation is taken per warpgroup at
    // one instruction each (setmaxnreg is aligned over a warpgroup): the load /
    // MMA warp and the expanding warps give registers back, the softmax
    // warpgroups take them.
    if (warp >= kSoftThreads / 32) {
        if (kPaged) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
        if (warp == kSoftThreads / 32) {
            // ---------------- load / MMA thread
            if (lane == 0) {
                constexpr uint32_t idesc_s = idesc_bf16_f32(128, kKeys, false);
                constexpr uint32_t idesc_o = idesc_bf16_f32(128, kHeadDim, true);
                auto mma_s = [&](int w, int s) {  // S_w = Q_w K(slot s)^T over head_dim, 16 at a time
                    const uint32_t sQ = sbase + kOffQ + w * kQBytes, sK = sbase + kOffK + s * kKVTile;
#pragma unroll
                    for (int kk = 0; kk < 8; kk++) {
                        const uint32_t blk = (uint32_t)(kk >> 2), sub = (uint32_t)(kk & 3) * 32;
                        tc_mma_bf16(tmem + 128u * w, smem_desc_sw128(sQ + blk * (kQRows * 128) + sub, 16, 1024),
                                    smem_desc_sw128(sK + blk * kKVBlock + sub, 16, 1024), idesc_s, kk > 0);
                    }
                    tc_commit(&s_done[w]);
                };
                auto mma_pv = [&](int w, int j, int s) {  // O_w += P_w V(slot s) over the tile's 128 keys
                    const uint32_t sV = sbase + kOffV + s * kKVTile;
#pragma unroll
                    for (int kk = 0; kk < 8; kk++)  // P from TMEM: 8 columns = 16 keys
                        tc_mma_bf16_tmem_a(tmem + kColO + 128u * w, tmem + 128u * w + kk * 8,
                                           smem_desc_sw128(sV + kk * 16 * 128, kKVBlock, 1024), idesc_o,
                                           (j > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&pv_done[w]);
                };
                // Issue whatever is ready, for either query tile, so that the tensor core
                // always holds the next product of one tile while the other's softmax runs:
                //   S_w(t) once K(t) has landed and O_w += P_w(t - 1) V(t - 1) is complete;
                //   O_w += P_w(t) V(t) once P_w(t) is stored and V(t) has landed;
                //   K(t) into slot t % 2 once both S(t - 2) are done (their P V issued);
                //   V(t) into slot t % 2 once both P(t - 2) V(t - 2) are complete.
                // Each barrier is polled only where it cannot be two phases ahead.
                // Phase of the barrier that completes tile t in slot t % 2: tile t is
                // the (t / 2)-th of its slot; with a paged prefix, chunk tiles count
                // from the first chunk tile (prefix tiles complete k_dq / v_dq instead).
                auto kv_phase = [&](int t) { return (uint32_t)((((kPaged && t >= nt_pre) ? t - nt_pre : t) >> 1) & 1); };
                int tw[kWGs] = {0, 0};                 // next tile of query tile w
                bool at_pv[kWGs] = {false, false};     // its next product is P V (else S)
                int pv_seen[kWGs] = {0, 0};            // its P V of tiles < pv_seen are known complete
                int k_next = nt > 1 ? 2 : 1, v_next = k_next;  // next K / V tiles to request
                bool ok = true;
                uint32_t idle = 0;
                for (;;) {
                    bool progress = false, finished = true;
#pragma unroll
                    for (int w = 0; w < kWGs; w++) {
                        const int t = tw[w];
                        if (w >= nwg || t >= nt) continue;
                        finished = false;
                        if (!at_pv[w]) {
                            if (t > 0 && pv_seen[w] < t) {
                                if (!mbar_test_wait(&pv_done[w], (uint32_t)((t - 1) & 1))) continue;
                                pv_seen[w] = t;
                            }
                            uint64_t *kb = kPaged && t < nt_pre ? &k_dq[t & 1] : &k_full[t & 1];
                            if (!mbar_test_wait(kb, kv_phase(t))) continue;
                            tc_fence_after();
                            mma_s(w, t & 1);
                            at_pv[w] = true;
                        } else {
                            if (!mbar_test_wait(&p_full[w], (uint32_t)(t & 1))) continue;
                            uint64_t *vb = kPaged && t < nt_pre ? &v_dq[t & 1] : &v_full[t & 1];
                            if (!mbar_test_wait(vb, kv_phase(t))) continue;
                            tc_fence_after();
                            mma_pv(w, t, t & 1);
                            at_pv[w] = false;
                            tw[w] = t + 1;
                        }
                        progress = true;
                    }
                    if (finished) break;
                    int min_tw = tw[0], min_seen = pv_seen[0];
                    if (nwg > 1) {
                        min_tw = min(min_tw, tw[1]);
                        min_seen = min(min_seen, pv_seen[1]);
                    }
                    if (k_next < nt && min_tw >= k_next - 1) {
                        load_k(k_next, k_next & 1);
                        k_next++;
                        progress = true;
                    }
                    if (v_next < nt && min_seen >= v_next - 1) {
                        load_v(v_next, v_next & 1);
                        v_next++;
                        progress = true;
                    }
                    if (progress) {  // polls without sleeping: a sleep here lands on the critical path
                        idle = 0;
                    } else if (++idle > kWaitLimitE || *abort_flag) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) {
                    *abort_flag = 1;
                    flag_error(a.err, kErrTimeout);
                    // no copy or MMA may still be running when the CTA frees its memory
                    for (int t = max(kPaged ? nt_pre : 0, k_next - 2); t < k_next; t++)  // tensor copies only
                        mbar_wait_bounded(&k_full[t & 1], kv_phase(t), kWaitLimitE, nullptr);
                    for (int t = max(kPaged ? nt_pre : 0, v_next - 2); t < v_next; t++)
                        mbar_wait_bounded(&v_full[t & 1], kv_phase(t), kWaitLimitE, nullptr);
                    tc_commit(drain);
                    mbar_wait_bounded(drain, 0, kWaitLimitE, nullptr);
                }
            }
            __syncwarp();
        } else if (kPaged) {
            // ---------------- paged prefix: expand tile j's K (then V) from the NVFP4
            // pages into the BF16 operand layout of the slot, once it may be written
            const int dt = tid - kEThreads;  // 0 .. kDqThreads - 1
            const int32_t *bt = a.block_table + (int64_t)r * a.max_pages;
            constexpr int kBlocks = kKeys * 8;  // 16-value blocks of one K (or V) tile
            constexpr int kPer = (kBlocks + kDqThreads - 1) / kDqThreads;
            // Tile j's eight 16-token groups are bulk-copied in halves (K codes and
            // scales, V codes and scales: 1,152 B each) into raw stages by lanes 0..7
            // of the first dequantising warp as soon as a stage is free: the K halves
            // one tile ahead, the V halves two.  Groups past the prefix are not copied
            // (those keys are written as zeros); a group of an invalid page is
            // zero-filled and flagged.
            auto issue_raw = [&](int j, int which, uint8_t *dst, uint64_t *bar) {  // the first dequantising warp
                const int g = lane, tok = j * kKeys + 16 * g;
                int32_t pg = -1;
                if (g < 8 && tok < np) {
                    pg = __ldg(bt + (tok >> a.log2P));
                    if (pg < 0 || pg >= a.num_pages) {
                        flag_error(a.err, kErrPage);
                        uint4 *z = reinterpret_cast<uint4 *>(dst + g * kHalfGroup);
                        for (int i = 0; i < kHalfGroup / 16; i++) z[i] = make_uint4(0u, 0u, 0u, 0u);
                        pg = -1;
                    }
                }
                const unsigned copies = __popc(__ballot_sync(0xffffffffu, pg >= 0));
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(bar, copies * kHalfGroup);
                __syncwarp();
                if (pg >= 0)
                    bulk_g2s(dst + g * kHalfGroup,
                             a.pool + ((int64_t)pg * a.Hkv + kv) * a.slab + ((tok & (a.P - 1)) >> 4) * kGroupBytes +
                                 which * kHalfGroup,
                             kHalfGroup, bar);
            };
            uint8_t *rawk = smem + kOffRawK, *rawv = smem + kOffRawV;
            const bool issuer = warp == kEThreads / 32;
            // tiles whose halves were requested / seen landed (for the drain after an abort)
            int k_req = 0, k_seen = 0, v_req = 0, v_seen = 0;
            if (issuer) {
                for (int j = 0; j < 2 && j < nt_pre; j++) issue_raw(j, 1, rawv + j * kRawHalf, &rawv_full[j]);
                v_req = nt_pre < 2 ? nt_pre : 2;
                if (nt_pre > 0) {
                    issue_raw(0, 0, rawk, rawk_full);
                    k_req = 1;
                }
            }
            bool ok = true;
            for (int j = 0; ok && j < nt_pre; j++) {
                const int s = j & 1;
                for (int which = 0; which < 2; which++) {
                    uint64_t *landed = which ? &rawv_full[s] : rawk_full;
                    const uint32_t lph = (uint32_t)((which ? j >> 1 : j) & 1);
                    ok = __all_sync(0xffffffffu, spin_wait(landed, lph, abort_flag));
                    if (!ok) break;
                    if (which) v_seen = j + 1;
                    else k_seen = j + 1;
                    ok = __all_sync(0xffffffffu,
                                    spin_wait(which ? &v_go[s] : &k_go[s], (uint32_t)((j >> 1) & 1), abort_flag));
                    if (!ok) break;
                    const uint8_t *src = which ? rawv + s * kRawHalf : rawk;
                    uint8_t *tile = smem + (which ? kOffV : kOffK) + s * kKVTile;
                    const float g = which ? a.gv : a.gk;
                    auto expand = [&](auto unit) {  // unit: g = 1, chosen once per tile (the general form is long)
#pragma unroll 1
                        for (int i = 0; i < kPer; i++) {
                            const int b = dt + i * kDqThreads;
                            if (b >= kBlocks) continue;
                            const int key = b >> 3, blk = b & 7, tok = j * kKeys + key;
                            uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                            if (tok < np) {
                                const uint8_t *grp = src + (key >> 4) * kHalfGroup;  // codes [16][64] then scales
                                const int rr = key & 15;
                                const uint2 codes = *reinterpret_cast<const uint2 *>(grp + rr * 64 + blk * 8);
                                const uint32_t sb = grp[1024 + (which ? blk * 16 + rr : rr * 8 + blk)];
                                nvfp4_block_to_bf16<decltype(unit)::value>(codes, sb, g, o);
                            }
                            uint8_t *cb = tile + (blk >> 2) * kKVBlock;  // column block of head_dim 64 (blk / 4) ..
                            *reinterpret_cast<uint4 *>(cb + sw128_off(key, (blk & 3) * 2)) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                            *reinterpret_cast<uint4 *>(cb + sw128_off(key, (blk & 3) * 2 + 1)) =
                                make_uint4(o[4], o[5], o[6], o[7]);
                        }
                    };
                    if (g == 1.0f)
                        expand(std::true_type{});
                    else
                        expand(std::false_type{});
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the tile for the tensor core
                    mbar_arrive(which ? &v_dq[s] : &k_dq[s]);
                    // the raw half is read: the tile after next (K) or the next (V) may land in it
                    mbar_arrive(which ? &rawv_free[s] : rawk_free);
                    const int jn = which ? j + 2 : j + 1;
                    if (issuer && jn < nt_pre) {
                        ok = __all_sync(0xffffffffu, spin_wait(which ? &rawv_free[s] : rawk_free, lph, abort_flag));
                        if (!ok) break;
                        if (which) {
                            issue_raw(jn, 1, rawv + s * kRawHalf, &rawv_full[s]);
                            v_req = jn + 1;
                        } else {
                            issue_raw(jn, 0, rawk, rawk_full);
                            k_req = jn + 1;
                        }
                    }
                }
            }
            if (issuer) {  // no copy may still be writing when the CTA frees its memory
                for (int j = k_seen; j < k_req; j++) mbar_wait_bounded(rawk_full, (uint32_t)(j & 1), kWaitLimitE, nullptr);
                for (int j = v_seen; j < v_req; j++)
                    mbar_wait_bounded(&rawv_full[j & 1], (uint32_t)((j >> 1) & 1), kWaitLimitE, nullptr);
            }
            if (!ok) {
                *abort_flag = 1;
                if (lane == 0) flag_error(a.err, kErrTimeout);
            }
        }
    } else {
        if (kPaged) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftRegs));
        if ((tid >> 7) < nwg) {
            // ---------------- softmax of this thread's query row
            const int w = tid >> 7;
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lanes
            const uint32_t colS = 128u * w, colO = kColO + 128u * w;
            const int R = row0 + w * kQRows + (tid & 127);
            const bool row_ok = R < rows;
            const int token = row_ok ? R / a.G : 0;
            float m_run = kNegInfE, l_run = 0.f;
            bool ok = true;
            for (int j = 0; j < nt; j++) {
                // S_w(j) done; its commit also covers O_w += P_w(j - 1) V(j - 1)
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s_done[w], (uint32_t)(j & 1), kWaitLimitE, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const bool pre = j < nt_pre;
                const int base = pre ? j * kKeys : (j - nt_pre) * kKeys;
                const int visible = (pre ? np : token + 1) - base;   // keys [0, visible) of the tile are seen
                const bool edge = __any_sync(0xffffffffu, visible < kKeys);  // mask on edge tiles only
                // the row's 64 scores of half h (masked scores are -inf)
                auto load_half = [&](int h, float (&sc)[64]) {
                    uint32_t sr[2][32];
                    tc_ld32(tmem + lane_base + colS + 64 * h, sr[0]);
                    tc_ld32(tmem + lane_base + colS + 64 * h + 32, sr[1]);
                    tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 64; c++) sc[c] = __uint_as_float(sr[c >> 5][c & 31]);
                    if (edge) {
#pragma unroll
                        for (int c = 0; c < 64; c++)
                            if (64 * h + c >= visible) sc[c] = kNegInfE;
                    }
                };
                // P = 2^(s * scale - m) of one half, rounded to BF16 pairs; ls += the rounded values
                auto make_p = [&](const float (&sc)[64], float neg_m, uint32_t (&pw)[32], float (&ls)[4]) {
#pragma unroll
                    for (int c = 0; c < 32; c++) {
                        const float2 e = fma2(make_float2(sc[2 * c], sc[2 * c + 1]), a.score_log2, neg_m);
                        const __nv_bfloat162 pr = __floats2bfloat162_rn(ex2(e.x), ex2(e.y));
                        pw[c] = *reinterpret_cast<const uint32_t *>(&pr);
                        add_bf16x2(ls[2 * (c & 1)], ls[2 * (c & 1) + 1], pw[c]);
                    }
                };
                auto half_max = [&](const float (&sc)[64]) {
                    float m8[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) m8[e] = max3(sc[e], sc[8 + e], sc[16 + e]);
#pragma unroll
                    for (int e = 0; e < 8; e++) m8[e] = max3(m8[e], sc[24 + e], sc[32 + e]);
#pragma unroll
                    for (int e = 0; e < 8; e++) m8[e] = max3(m8[e], sc[40 + e], sc[48 + e]);
#pragma unroll
                    for (int e = 0; e < 8; e++) m8[e] = fmaxf(m8[e], sc[56 + e]);
                    return max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                };
                // One pass with the running max as it stands (the lazy rescale lets it
                // lag the true max by up to 2^8): P of half 0 stays in registers until
                // half 1 shows whether the max must move; only then does it go over the
                // scores in TMEM.  If it must (the first tile, rarely later), O and the
                // row sum are rescaled and P is formed again from the scores in TMEM.
                uint32_t pw0[32], pw1[32];
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
                float smax;
                {
                    float sc[64];
                    load_half(0, sc);
                    smax = half_max(sc);
                    make_p(sc, -m_run, pw0, ls);
                    load_half(1, sc);
                    smax = fmaxf(smax, half_max(sc));
                    const float mx = smax * a.score_log2;  // the scale is positive
                    const bool need = mx > m_run + kRescale;
                    if (!__any_sync(0xffffffffu, need)) {
                        make_p(sc, -m_run, pw1, ls);
                    } else {
                        const float m_new = need ? fmaxf(m_run, mx) : m_run;
                        const float alpha = need ? (m_run == kNegInfE ? 0.f : ex2(m_run - m_new)) : 1.f;
                        if (j > 0) {  // O_w holds tiles 0 .. j - 1 (complete): rescale this warp's rows
#pragma unroll
                            for (int cblk = 0; cblk < 4; cblk++) {
                                uint32_t ov[32];
                                tc_ld32(tmem + lane_base + colO + 32 * cblk, ov);
                                tc_wait_ld();
#pragma unroll
                                for (int e = 0; e < 32; e++) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                                tc_st32(tmem + lane_base + colO + 32 * cblk, ov);
                            }
                            tc_wait_st();
                        }
                        l_run *= alpha;
                        m_run = m_new;
                        ls[0] = ls[1] = ls[2] = ls[3] = 0.f;
                        make_p(sc, -m_run, pw1, ls);
                        load_half(0, sc);
                        make_p(sc, -m_run, pw0, ls);
                    }
                }
                l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                tc_st32(tmem + lane_base + colS, pw0);       // over scores 0 .. 31 (read already)
                tc_st32(tmem + lane_base + colS + 32, pw1);  // over scores 32 .. 63
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(&p_full[w]);
            }
            // O_w is complete after O_w += P_w(nt - 1) V(nt - 1); the previous one is
            // done already (S_w(nt - 1) waited for it), so one parity wait suffices
            if (ok)
                ok = __all_sync(0xffffffffu,
                                mbar_wait_bounded(&pv_done[w], (uint32_t)((nt - 1) & 1), kWaitLimitE, abort_flag));
            if (!ok) {
                *abort_flag = 1;
                if (lane == 0) flag_error(a.err, kErrTimeout);
            } else {
                // ---- O / l -> BF16 row of the output
                tc_fence_after();
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                uint4 *dst =
                    reinterpret_cast<uint4 *>(a.out + (((int64_t)q0 + token) * a.Hq + kv * a.G + R % a.G) * kHeadDim);
#pragma unroll
                for (int cblk = 0; cblk < 4; cblk++) {
                    uint32_t ov[32];
                    tc_ld32(tmem + lane_base + colO + 32 * cblk, ov);
                    tc_wait_ld();
                    if (row_ok) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; q4++) {
                            uint32_t wv[4];
#pragma unroll
                            for (int e = 0; e < 4; e++) {
                                const __nv_bfloat162 hv = __floats2bfloat162_rn(
                                    __uint_as_float(ov[8 * q4 + 2 * e]) * inv, __uint_as_float(ov[8 * q4 + 2 * e + 1]) * inv);
                                wv[e] = *reinterpret_cast<const uint32_t *>(&hv);
                            }
                            dst[4 * cblk + q4] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                        }
                    }
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

// [rows][Hkv][128] BF16 at `base` as a 3-D map with 64 x 1 x 128 boxes.
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

namespace {

template <bool kPaged>
cudaError_t launch_extend_kernel(const ExtendMaps &maps, const ExtendArgs &a, int num_reqs, int max_q_len,
                                 int num_kv_heads, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(reinterpret_cast<const void *>(&extend_kernel<kPaged>),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kPaged ? kESmemPaged : kESmem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int64_t qtiles = ceil_div64((int64_t)max_q_len * a.G, kCtaRows);
    dim3 grid((unsigned)qtiles, (unsigned)num_kv_heads, (unsigned)num_reqs);
    extend_kernel<kPaged><<<grid, kPaged ? kEThreadsPaged : kEThreads, kPaged ? kESmemPaged : kESmem, stream>>>(maps, a);
    return cudaGetLastError();
}

ExtendArgs common_args(const void *q, const int32_t *cu_q, int max_q_len, int num_q_heads, int num_kv_heads,
                       float sm_scale, void *out, unsigned *err) {
    ExtendArgs a = {};
    a.q = static_cast<const uint16_t *>(q);
    a.cu_q = cu_q;
    a.Hq = num_q_heads;
    a.Hkv = num_kv_heads;
    a.G = num_q_heads / num_kv_heads;
    a.max_q_len = max_q_len;
    a.score_log2 = (float)((double)sm_scale * 1.4426950408889634);
    a.out = static_cast<uint16_t *>(out);
    a.err = err;
    return a;
}

}  // namespace

cudaError_t launch_extend(const void *q, const void *k_prefix, const void *v_prefix, const int32_t *cu_prefix,
                          int64_t total_prefix, const void *k_chunk, const void *v_chunk, const int32_t *cu_q,
                          int64_t total_q, int num_reqs, int max_q_len, int num_q_heads, int num_kv_heads,
                          float sm_scale, void *out, unsigned *err, cudaStream_t stream) {
    ExtendMaps maps;
    if (!make_kv_map(&maps.k_pre, k_prefix, total_prefix, num_kv_heads) ||
        !make_kv_map(&maps.v_pre, v_prefix, total_prefix, num_kv_heads) ||
        !make_kv_map(&maps.k_new, k_chunk, total_q, num_kv_heads) ||
        !make_kv_map(&maps.v_new, v_chunk, total_q, num_kv_heads))
        return cudaErrorInvalidValue;
    ExtendArgs a = common_args(q, cu_q, max_q_len, num_q_heads, num_kv_heads, sm_scale, out, err);
    a.cu_prefix = cu_prefix;
    return launch_extend_kernel<false>(maps, a, num_reqs, max_q_len, num_kv_heads, stream);
}

cudaError_t launch_extend_paged(const nvfp4kv_cache &c, const void *q, const int32_t *block_table, int max_pages,
                                const int32_t *prefix_lens, const void *k_chunk, const void *v_chunk,
                                const int32_t *cu_q, int64_t total_q, int num_reqs, int max_q_len, int num_q_heads,
                                float sm_scale, void *out, unsigned *err, cudaStream_t stream) {
    ExtendMaps maps;  // the prefix maps are never used: they alias the chunk
    if (!make_kv_map(&maps.k_new, k_chunk, total_q, c.num_kv_heads) ||
        !make_kv_map(&maps.v_new, v_chunk, total_q, c.num_kv_heads))
        return cudaErrorInvalidValue;
    maps.k_pre = maps.k_new;
    maps.v_pre = maps.v_new;
    ExtendArgs a = common_args(q, cu_q, max_q_len, num_q_heads, c.num_kv_heads, sm_scale, out, err);
    a.pool = static_cast<const uint8_t *>(c.pool);
    a.num_pages = c.num_pages;
    a.slab = (int64_t)144 * c.page_size;
    a.P = c.page_size;
    a.log2P = __builtin_ctz((unsigned)c.page_size);
    a.max_pages = max_pages;
    a.block_table = block_table;
    a.prefix_lens = prefix_lens;
    a.gk = c.k_global_scale;
    a.gv = c.v_global_scale;
    return launch_extend_kernel<true>(maps, a, num_reqs, max_q_len, c.num_kv_heads, stream);
}

}  // namespace nvfp4kv
