// quantize_append.cu -- BF16 K/V rows -> NVFP4 (or FP8) rows in the paged pool.
//
// Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV
// Cache", section A2, paths 1 and 2 (the KV of a prefill or of a new chunk is
// quantised and written into the persistent paged cache), format of section A3
// and Fig. 1 (E2M1 values, one E4M3 scale per 16 values, FP32 tensor scale).
//
// A 16-value block is 32 bytes of BF16 in (two 16-byte loads) and 8 bytes of
// packed codes + 1 scale byte out; eight consecutive threads cover one
// head_dim row, so reads are fully coalesced and the 64-byte code row is
// written by one 8-thread group.  Each thread quantises three blocks a grid
// apart, their loads issued first.  The kernel is HBM-bound: per token and KV
// head it reads 512 B of BF16 and writes 144 B.
//
// Rounding (must match the CPU oracle bit for bit):
//   q     = amax / (6 g)                         FP32, correctly rounded
//   scale = cvt.rn.satfinite.e4m3 (q)            nearest-even, saturating
//   y_i   = x_i / (scale g)                      see below
//   code  = cvt.rn.satfinite.e2m1 (y_i)          nearest-even, saturating
// For g = 1 the kernel forms q as amax * fl32(1/6): the FP32 results differ
// from the quotient for some amax, but the E4M3 scale never does (all 32,640
// finite non-negative BF16 values checked on the host).  It forms y_i as
// x_i * rcp(scale) with the hardware's approximate reciprocal, rounds y_i to
// FP16 (11 significant bits) and converts that to E2M1.  x_i has at most 8
// significant bits and the scale at most 4, so every exact quotient that is
// not exactly an E2M1 rounding midpoint lies more than 2^-8 (relative) away
// from every midpoint, far outside the ~2^-22 error of the reciprocal product
// plus the 2^-11 of the FP16 rounding, which therefore neither crosses a
// midpoint nor lands on one; an exact midpoint has at most 3 significant bits
// and the FP16 rounding lands on it exactly (quotients beyond the FP16 range
// become infinity, which saturates to 6 like the quotient itself).  Hence the
// codes equal those of the exactly rounded quotient (the GPU tests check every
// BF16 value against every scale).  For g != 1 the codes are the
// exact roundings too (quantize.cuh: an FP32 estimate, then exact midpoint
// checks by fused multiply-add).
#include "common.cuh"
#include "kernels.h"
#include "quantize.cuh"

namespace nvfp4kv {

namespace {

struct AppendArgs {
    uint8_t *pool;
    int64_t num_slots;  // num_pages * P
    int P;
    int log2P;
    int Hkv;
    int log2Hkv;        // log2(Hkv) when Hkv is a power of two, else -1
    int64_t slab;       // bytes per (page, kv_head)
    const uint4 *k;     // BF16 rows viewed as 16-byte vectors
    const uint4 *v;
    int64_t num_tokens;
    int64_t stride16;   // token stride in 16-byte units
    const int64_t *slots;
    float gk, gv;
    int dtype;
    unsigned *err;
};

constexpr int kBlocksPerThread = 3;  // 16-value blocks per thread, their loads issued together

// Work item -> (token, kv_head, which, block), block fastest.  Thread i takes
// items i, i + n, i + 2n (n = threads in the grid), so every round of loads is
// coalesced across the warp, and issues all of their loads before the first
// quantisation: three blocks' worth of reads in flight per thread hide the HBM
// latency that one block's could not (72.4 -> 68.3 us on 65,536 random slots).
template <bool kUnitScale>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
    pdl_launch_dependents();  // a dependent decode plan may launch early; it waits for this kernel
    // the host guarantees num_tokens * Hkv * 16 < 2^31
    const uint32_t items = (uint32_t)(a.num_tokens * a.Hkv * 16);
    const uint32_t n = gridDim.x * blockDim.x;
    const uint32_t id0 = blockIdx.x * blockDim.x + threadIdx.x;
    // Scale bytes are stored "evict last" in L2: with scattered slots the other
    // tokens of a scale sector arrive at random times in the call, and a sector
    // evicted partly written costs a read of the rest from DRAM.  On 65,536
    // tokens x 8 heads into random slots of a 2,048-page pool, 66 -> 61.5 us
    // (57.5 against 55.6 us with page-ordered slots).
    const uint64_t scale_policy = l2_policy_evict_last();
    uint4 x0[kBlocksPerThread], x1[kBlocksPerThread];
    int64_t slot[kBlocksPerThread];
#pragma unroll
    for (int j = 0; j < kBlocksPerThread; j++) {
        const uint32_t id = id0 + (uint32_t)j * n;
        slot[j] = -1;
        if (id >= items) continue;
        const int blk = (int)(id & 7);
        const int which = (int)((id >> 3) & 1);
        const uint32_t th = id >> 4;
        const uint32_t t32 = a.log2Hkv >= 0 ? th >> a.log2Hkv : th / (uint32_t)a.Hkv;
        const int h = (int)(th - t32 * (uint32_t)a.Hkv);
        const uint4 *src = (which ? a.v : a.k) + (int64_t)t32 * a.stride16 + h * (kHeadDim / 8) + blk * 2;
        x0[j] = __ldg(src);
        x1[j] = __ldg(src + 1);
        slot[j] = __ldg(a.slots + t32);
    }
#pragma unroll
    for (int j = 0; j < kBlocksPerThread; j++) {
        const uint32_t id = id0 + (uint32_t)j * n;
        if (id >= items || slot[j] < 0) continue;
        const int blk = (int)(id & 7);
        const int which = (int)((id >> 3) & 1);
        const uint32_t th = id >> 4;
        const uint32_t t32 = a.log2Hkv >= 0 ? th >> a.log2Hkv : th / (uint32_t)a.Hkv;
        const int h = (int)(th - t32 * (uint32_t)a.Hkv);
        if (slot[j] >= a.num_slots) {
            if (blk == 0 && which == 0 && h == 0) flag_error(a.err, kErrSlot);
            continue;
        }
        const int64_t page = slot[j] >> a.log2P;
        store_block_values<kUnitScale, true>(a.pool + (page * a.Hkv + h) * a.slab, a.dtype,
                                             (int)(slot[j] & (a.P - 1)), which, blk, x0[j], x1[j],
                                             which ? a.gv : a.gk, scale_policy);
    }
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
    a.log2Hkv = (c.num_kv_heads & (c.num_kv_heads - 1)) == 0 ? __builtin_ctz((unsigned)c.num_kv_heads) : -1;
    a.slab = (int64_t)(c.dtype == NVFP4KV_DTYPE_NVFP4 ? 144 : 256) * c.page_size;
    a.k = static_cast<const uint4 *>(k);
    a.v = static_cast<const uint4 *>(v);
    a.num_tokens = num_tokens;
    a.stride16 = token_stride / 8;
    a.slots = slot_mapping;
    a.gk = c.k_global_scale;
    a.gv = c.v_global_scale;
    a.dtype = c.dtype;
    a.err = err;
    const int64_t items = num_tokens * c.num_kv_heads * 2 * 8;
    const int block = 256;
    const int64_t grid = ceil_div64(ceil_div64(items, kBlocksPerThread), block);
    const bool unit = c.k_global_scale == 1.0f && c.v_global_scale == 1.0f;
    if (unit)
        append_kernel<true><<<(unsigned)grid, block, 0, stream>>>(a);
    else
        append_kernel<false><<<(unsigned)grid, block, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace nvfp4kv
