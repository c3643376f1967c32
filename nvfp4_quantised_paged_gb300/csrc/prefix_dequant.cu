// prefix_dequant.cu -- cached NVFP4 (or FP8) prefix pages -> contiguous BF16 workspace.
//
// Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV
// Cache", section A2, path 2 (chunked prefill / extend): the cached prefix's
// entries are gathered through the page table and dequantised into a
// workspace shared across layers, which the new chunk's KV then joins.  The
// page writes an FP8 workspace; this kernel writes BF16, which holds every
// dequantised value exactly for a tensor scale of 1.
//
// One thread per 16-value block: reads 8 code bytes + 1 scale byte (NVFP4) or
// 16 bytes (FP8), writes 32 bytes of BF16.  HBM-bound, dominated by writes
// (per token and KV head 144 B in, 512 B out).
#include "common.cuh"
#include "kernels.h"
#include "quantize.cuh"

namespace nvfp4kv {

namespace {

struct PrefixArgs {
    const uint8_t *pool;
    int64_t num_pages;
    int P;
    int log2P;
    int Hkv;
    int64_t slab;
    int dtype;
    float gk, gv;
    const int32_t *block_table;
    int max_pages;
    const int32_t *prefix_lens;
    const int32_t *cu;
    int num_reqs;
    int64_t total;
    uint4 *k_ws;
    uint4 *v_ws;
    unsigned *err;
};


__global__ void __launch_bounds__(256) prefix_dequant_kernel(PrefixArgs a) {
    // the host guarantees total * Hkv * 16 < 2^31
    const uint32_t id = blockIdx.x * blockDim.x + threadIdx.x;
    if (id >= (uint32_t)(a.total * a.Hkv * 16)) return;
    const int blk = (int)(id & 7);
    const int which = (int)((id >> 3) & 1);
    const uint32_t th = id >> 4;
    const uint32_t row = th / (uint32_t)a.Hkv;
    const int h = (int)(th - row * (uint32_t)a.Hkv);
    // request r: the last r with cu[r] <= row
    int lo = 0, hi = a.num_reqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((uint32_t)__ldg(a.cu + mid) <= row) lo = mid;
        else hi = mid - 1;
    }
    const int r = lo;
    const int64_t t = (int64_t)row - __ldg(a.cu + r);
    const int32_t n = __ldg(a.prefix_lens + r);
    if (t < 0 || t >= n) {
        if (blk == 0 && which == 0 && h == 0) flag_error(a.err, kErrCuPrefix);
        return;
    }
    if (t >= (int64_t)a.max_pages * a.P) {
        if (blk == 0 && which == 0 && h == 0) flag_error(a.err, kErrSeqLen);
        return;
    }
    const int64_t page = __ldg(a.block_table + (int64_t)r * a.max_pages + (t >> a.log2P));
    if (page < 0 || page >= a.num_pages) {
        if (blk == 0 && which == 0 && h == 0) flag_error(a.err, kErrPage);
        return;
    }
    const int rp = (int)(t & (a.P - 1));
    const int rr = rp & 15;  // row inside its 16-token group
    const uint8_t *slab = a.pool + (page * a.Hkv + h) * a.slab;
    const float g = which ? a.gv : a.gk;
    uint32_t o[8];
    if (a.dtype == NVFP4KV_DTYPE_NVFP4) {
        const uint8_t *grp = slab + (rp >> 4) * 2304;
        const uint2 codes = __ldg(reinterpret_cast<const uint2 *>(grp + (which ? 1152 : 0) + rr * 64 + blk * 8));
        const uint32_t sbyte = __ldg(grp + (which ? 2176 + blk * 16 + rr : 1024 + rr * 8 + blk));
        if (g == 1.0f)
            nvfp4_block_to_bf16<true>(codes, sbyte, g, o);
        else
            nvfp4_block_to_bf16<false>(codes, sbyte, g, o);
    } else {
        const uint4 c = __ldg(
            reinterpret_cast<const uint4 *>(slab + (rp >> 4) * 4096 + (which ? 2048 : 0) + rr * 128 + blk * 16));
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
        if (g == 1.0f) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                o[2 * i] = f16x2_to_bf16x2_scaled<true>(e4m3x2_to_f16x2(w[i] & 0xffffu), g);
                o[2 * i + 1] = f16x2_to_bf16x2_scaled<true>(e4m3x2_to_f16x2(w[i] >> 16), g);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                o[2 * i] = f16x2_to_bf16x2_scaled<false>(e4m3x2_to_f16x2(w[i] & 0xffffu), g);
                o[2 * i + 1] = f16x2_to_bf16x2_scaled<false>(e4m3x2_to_f16x2(w[i] >> 16), g);
            }
        }
    }
    uint4 *dst = (which ? a.v_ws : a.k_ws) + ((int64_t)row * a.Hkv + h) * (kHeadDim / 8) + blk * 2;
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace

cudaError_t launch_prefix_dequant(const nvfp4kv_cache &c, const int32_t *block_table, int max_pages,
                                  const int32_t *prefix_lens, const int32_t *cu, int num_reqs, int64_t total,
                                  void *k_ws, void *v_ws, unsigned *err, cudaStream_t stream) {
    PrefixArgs a;
    a.pool = static_cast<const uint8_t *>(c.pool);
    a.num_pages = c.num_pages;
    a.P = c.page_size;
    a.log2P = __builtin_ctz((unsigned)c.page_size);
    a.Hkv = c.num_kv_heads;
    a.slab = (int64_t)(c.dtype == NVFP4KV_DTYPE_NVFP4 ? 144 : 256) * c.page_size;
    a.dtype = c.dtype;
    a.gk = c.k_global_scale;
    a.gv = c.v_global_scale;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.prefix_lens = prefix_lens;
    a.cu = cu;
    a.num_reqs = num_reqs;
    a.total = total;
    a.k_ws = static_cast<uint4 *>(k_ws);
    a.v_ws = static_cast<uint4 *>(v_ws);
    a.err = err;
    const int64_t threads = total * c.num_kv_heads * 16;
    const int block = 256;
    prefix_dequant_kernel<<<(unsigned)ceil_div64(threads, block), block, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace nvfp4kv
