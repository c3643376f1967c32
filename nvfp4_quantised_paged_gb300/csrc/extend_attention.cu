// extend_attention.cu -- attention of a new chunk over [cached prefix || chunk], causal in the chunk.
//
// Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV
// Cache", section A2, path 2 (chunked prefill / extend): the attention takes
// two KV sources, the cached prefix -- gathered from the NVFP4 pages and
// dequantised into a workspace shared across layers (prefix_dequant.cu
// writes it, in BF16) -- and the current chunk's own K/V.  Chunk token i
// attends to the whole prefix and to chunk tokens 0..i.
//
// GB300 design: a flash-attention forward with BF16 mma.sync (m16n8k16,
// FP32 accumulation).  One CTA = 4 warps = 64 query rows of one (request,
// kv head), row = chunk token * G + query head of the group, so the G heads
// that share a KV head share every K/V tile.  K/V tiles of 64 keys (16 KB
// each) are double-buffered in shared memory by cp.async (rows past the end
// zero-filled) in a 16-byte-chunk XOR swizzle that makes the ldmatrix reads
// conflict-free; S = Q K^T takes K through ldmatrix, P.V takes V through
// ldmatrix.trans, and the S accumulators become the P operand in registers.
// Base-2 online softmax with a lazily updated running max (rescale only when
// a score exceeds it by 2^8).  Prefix tiles come first, then the chunk tiles
// up to the CTA's last token, masked causally.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4kv {

namespace {

constexpr int kEWarps = 4;
constexpr int kEThreads = 32 * kEWarps;
constexpr int kQRows = 16 * kEWarps;      // query rows per CTA
constexpr int kKeys = 64;                 // keys per K/V tile
constexpr int kRowBytes = kHeadDim * 2;   // one BF16 row
constexpr int kTileBytes = kKeys * kRowBytes;
constexpr int kStageBytes = 2 * kTileBytes;  // K tile | V tile
constexpr int kESmem = 2 * kStageBytes;      // double buffer
constexpr float kRescale = 8.0f;
constexpr float kNegInfE = -__builtin_huge_valf();
constexpr uint32_t kOnesBf16x2 = 0x3f803f80u;

struct ExtendArgs {
    const uint16_t *q;                 // BF16 [total_q][Hq][128]
    const uint16_t *k_pre, *v_pre;     // BF16 [total_prefix][Hkv][128]
    const uint16_t *k_new, *v_new;     // BF16 [total_q][Hkv][128]
    const int32_t *cu_prefix, *cu_q;   // [num_reqs + 1]
    int Hq, Hkv, G, max_q_len;
    float score_log2;                  // sm_scale * log2(e)
    uint16_t *out;                     // BF16 [total_q][Hq][128]
    unsigned *err;
};

// Byte offset of 16-byte chunk `chunk` (0..15) of row `row` in a swizzled tile.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, FP32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(kEThreads, 3) extend_kernel(ExtendArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int r = blockIdx.z, kv = blockIdx.y;
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
    const int row_end = min(row0 + kQRows, rows);
    const int t_last = (row_end - 1) / a.G;  // last chunk token of this CTA
    const int nt_pre = (np + kKeys - 1) / kKeys;
    const int nt = nt_pre + t_last / kKeys + 1;

    // this thread's two query rows (g and g + 8 of its warp's 16)
    const int ra = row0 + 16 * warp + g, rb = ra + 8;
    const bool va = ra < rows, vb = rb < rows;
    const int ta = va ? ra / a.G : 0, tb = vb ? rb / a.G : 0;

    // ---- Q fragments (A operand, 8 k-steps over head_dim)
    uint32_t qf[8][4];
    {
        const uint32_t *qa = reinterpret_cast<const uint32_t *>(
            a.q + ((int64_t)(q0 + ta) * a.Hq + kv * a.G + ra % a.G) * kHeadDim);
        const uint32_t *qb = reinterpret_cast<const uint32_t *>(
            a.q + ((int64_t)(q0 + tb) * a.Hq + kv * a.G + rb % a.G) * kHeadDim);
#pragma unroll
        for (int ks = 0; ks < 8; ks++) {
            qf[ks][0] = va ? __ldg(qa + 8 * ks + c) : 0u;
            qf[ks][1] = vb ? __ldg(qb + 8 * ks + c) : 0u;
            qf[ks][2] = va ? __ldg(qa + 8 * ks + 4 + c) : 0u;
            qf[ks][3] = vb ? __ldg(qb + 8 * ks + 4 + c) : 0u;
        }
    }

    const uint32_t sbase = smem_u32(smem);
    // cp.async of tile i into stage s: 1024 16-byte chunks of K and of V, 8 + 8 per thread
    auto issue = [&](int i, int s) {
        const bool pre = i < nt_pre;
        const int base = pre ? i * kKeys : (i - nt_pre) * kKeys;
        const int limit = pre ? np : L;
        const uint16_t *kb = pre ? a.k_pre : a.k_new;
        const uint16_t *vsrc = pre ? a.v_pre : a.v_new;
        const int64_t row_origin = pre ? p0 : q0;
#pragma unroll
        for (int it = 0; it < 8; it++) {
            const int idx = tid + it * kEThreads;  // 0..1023
            const int key = idx >> 4, chunk = idx & 15;
            const bool ok = base + key < limit;
            // rows past the end are zero-filled; their (unread) source is the tensor base
            const int64_t grow = ok ? ((row_origin + base + key) * a.Hkv + kv) * kHeadDim + chunk * 8 : 0;
            const uint32_t dst = sbase + s * kStageBytes + swz(key, chunk);
            cp_async16(dst, kb + grow, ok);
            cp_async16(dst + kTileBytes, vsrc + grow, ok);
        }
    };

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    // row sums of the BF16-rounded probabilities, from an all-ones B operand:
    // ol[0] (row g) and ol[2] (row g + 8), so numerator and denominator see
    // the same rounded weights
    float ol[4] = {0.f, 0.f, 0.f, 0.f};
    float m_a = kNegInfE, m_b = kNegInfE;

    issue(0, 0);
    cp_async_commit();
    for (int i = 0; i < nt; i++) {
        if (i + 1 < nt) issue(i + 1, (i + 1) & 1);
        cp_async_commit();
        cp_async_wait1();
        __syncthreads();
        const uint32_t kt = sbase + (i & 1) * kStageBytes, vt = kt + kTileBytes;
        const bool pre = i < nt_pre;
        const int base = pre ? i * kKeys : (i - nt_pre) * kKeys;

        // ---- S = Q K^T (16 rows x 64 keys per warp)
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
                ldsm_x4(kt + swz(key, 2 * ks + (m & 1)), b0, b1, b2, b3);
                mma_bf16_16816(s[2 * j], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
                mma_bf16_16816(s[2 * j + 1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
            }
        }

        // ---- mask, online softmax (base 2)
        float mx_a = kNegInfE, mx_b = kNegInfE;
#pragma unroll
        for (int n = 0; n < 8; n++) {
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int key = base + 8 * n + 2 * c + e;
                const bool oka = pre ? key < np : key <= ta;
                const bool okb = pre ? key < np : key <= tb;
                s[n][e] = oka ? s[n][e] * a.score_log2 : kNegInfE;
                s[n][2 + e] = okb ? s[n][2 + e] * a.score_log2 : kNegInfE;
                mx_a = fmaxf(mx_a, s[n][e]);
                mx_b = fmaxf(mx_b, s[n][2 + e]);
            }
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const bool need = mx_a > m_a + kRescale || mx_b > m_b + kRescale;
        if (__any_sync(0xffffffffu, need)) {
            const float na = fmaxf(m_a, mx_a), nb = fmaxf(m_b, mx_b);
            const float fa = na == kNegInfE ? 1.f : ex2(m_a - na), fb = nb == kNegInfE ? 1.f : ex2(m_b - nb);
            m_a = na;
            m_b = nb;
            ol[0] *= fa;
            ol[1] *= fa;
            ol[2] *= fb;
            ol[3] *= fb;
#pragma unroll
            for (int d = 0; d < 16; d++) {
                o[d][0] *= fa;
                o[d][1] *= fa;
                o[d][2] *= fb;
                o[d][3] *= fb;
            }
        }
        uint32_t pa[4][4];  // P as the A operand of 4 k-steps of 16 keys
#pragma unroll
        for (int n = 0; n < 8; n++) {
            const float p0 = ex2(s[n][0] - m_a), p1 = ex2(s[n][1] - m_a);
            const float p2 = ex2(s[n][2] - m_b), p3 = ex2(s[n][3] - m_b);
            pa[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0, p1);
            pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2, p3);
        }

        // ---- O += P V (16 rows x 128 dims per warp)
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {
#pragma unroll
            for (int nd = 0; nd < 16; nd += 2) {
                const int m = lane >> 3;
                const int key = 16 * kk + (m & 1) * 8 + (lane & 7);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vt + swz(key, nd + (m >> 1)), b0, b1, b2, b3);
                mma_bf16_16816(o[nd], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
                mma_bf16_16816(o[nd + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
            }
            mma_bf16_16816(ol, pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], kOnesBf16x2, kOnesBf16x2);
        }
        __syncthreads();  // the stage is refilled by the next iteration's copies
    }

    // ---- normalise and store
    const float l_a = ol[0], l_b = ol[2];
    const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
    uint32_t *oa = reinterpret_cast<uint32_t *>(a.out + ((int64_t)(q0 + ta) * a.Hq + kv * a.G + ra % a.G) * kHeadDim);
    uint32_t *ob = reinterpret_cast<uint32_t *>(a.out + ((int64_t)(q0 + tb) * a.Hq + kv * a.G + rb % a.G) * kHeadDim);
#pragma unroll
    for (int d = 0; d < 16; d++) {
        if (va) oa[4 * d + c] = pack_bf16(o[d][0] * ia, o[d][1] * ia);
        if (vb) ob[4 * d + c] = pack_bf16(o[d][2] * ib, o[d][3] * ib);
    }
}

}  // namespace

cudaError_t launch_extend(const void *q, const void *k_prefix, const void *v_prefix, const int32_t *cu_prefix,
                          const void *k_chunk, const void *v_chunk, const int32_t *cu_q, int num_reqs, int max_q_len,
                          int num_q_heads, int num_kv_heads, float sm_scale, void *out, unsigned *err,
                          cudaStream_t stream) {
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
    ExtendArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.k_pre = static_cast<const uint16_t *>(k_prefix);
    a.v_pre = static_cast<const uint16_t *>(v_prefix);
    a.k_new = static_cast<const uint16_t *>(k_chunk);
    a.v_new = static_cast<const uint16_t *>(v_chunk);
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
    extend_kernel<<<grid, kEThreads, kESmem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace nvfp4kv
