// decode_noalloc.cu -- paged decode attention for callers that cannot allocate.
//
// Some callers cannot allocate device memory themselves: code hosted by a
// framework that owns every device allocation, or a latency-critical path
// where cudaMalloc (which may synchronise the device) is not acceptable.
// nvfp4_paged_decode_attention needs a caller-provided workspace for its
// split-KV partials and work plan; this entry point runs the same kernels with
// that scratch taken from a fixed array of this library instead.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// the library holds its NVFP4KV_NOALLOC_SCRATCH_BYTES until the process exits.
// All calls share it, so calls that overlap on the GPU (for example on two
// streams without ordering between them) race on it.  Nothing in it needs to
// start at zero: every byte a call reads was written earlier in that call.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

using namespace nvfp4kv;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NVFP4KV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of the array on the current device, looked up once per
// device (host code sees only a stand-in for the symbol, not its address).
cudaError_t scratch_address(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int nvfp4_paged_decode_attention_noalloc(const nvfp4kv_cache *cache, const void *q, int batch,
                                                    int num_q_heads, const int32_t *block_table,
                                                    int max_pages_per_seq, const int32_t *seq_lens, float sm_scale,
                                                    void *out, int num_splits, cudaStream_t stream) {
    if (!cache || batch < 0 || num_q_heads < 1 || cache->num_kv_heads < 1 || num_q_heads % cache->num_kv_heads ||
        num_splits < 0)
        return NVFP4KV_EINVAL;
    if (batch == 0) return NVFP4KV_OK;
    const size_t need = nvfp4kv_decode_workspace_bytes(cache, batch, num_q_heads, num_splits);
    if (need == 0) return NVFP4KV_EINVAL;  // invalid descriptor or shape (same checks as the workspace query)
    if (need > (size_t)NVFP4KV_NOALLOC_SCRATCH_BYTES) return NVFP4KV_EUNSUPPORTED;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return NVFP4KV_ECUDA;
    return nvfp4_paged_decode_attention(cache, q, batch, num_q_heads, block_table, max_pages_per_seq, seq_lens,
                                        sm_scale, out, scratch, need, num_splits, stream);
}
