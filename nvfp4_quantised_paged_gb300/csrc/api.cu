// api.cu -- the C ABI of libnvfp4kv.so: host-side validation and dispatch.
//
// Every entry point validates its arguments on the host before launching, so
// a rejected call launches nothing.  Indices that live in device memory are
// checked by the kernels, which record problems in a per-device error word
// (a __device__ variable of this file) instead of trapping.
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace {

using namespace nvfp4kv;

__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
unsigned *g_err_ptr[kMaxDevices];

// Device address of this device's error word (looked up once per device).
unsigned *error_word(cudaError_t *status) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
    if (e != cudaSuccess) {
        *status = e;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_err_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_error_word);
        if (e != cudaSuccess) {
            *status = e;
            return nullptr;
        }
        g_err_ptr[dev] = static_cast<unsigned *>(p);
    }
    *status = cudaSuccess;
    return g_err_ptr[dev];
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A tensor scale is a positive normal FP32 number (the exact-rounding argument of
// the g != 1 quantiser needs g >= 2^-126).
bool normal_positive(float x) { return isfinite(x) && x >= 0x1p-126f; }

// Validates the cache descriptor; returns NVFP4KV_OK or a negative status.
int check_cache(const nvfp4kv_cache *c) {
    if (!c) return NVFP4KV_EINVAL;
    if (c->dtype != NVFP4KV_DTYPE_NVFP4 && c->dtype != NVFP4KV_DTYPE_FP8_E4M3) return NVFP4KV_EUNSUPPORTED;
    if (c->head_dim != kHeadDim) return NVFP4KV_EUNSUPPORTED;
    if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64 && c->page_size != 128)
        return NVFP4KV_EUNSUPPORTED;
    if (c->num_kv_heads < 1 || c->num_pages < 1) return NVFP4KV_EINVAL;
    if (!normal_positive(c->k_global_scale) || !normal_positive(c->v_global_scale)) return NVFP4KV_EINVAL;
    if (!c->pool || !aligned(c->pool, 256)) return NVFP4KV_EINVAL;
    return NVFP4KV_OK;
}

size_t slab_of(const nvfp4kv_cache *c) {
    return (size_t)(c->dtype == NVFP4KV_DTYPE_NVFP4 ? 144 : 256) * (size_t)c->page_size;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4KV_OK : NVFP4KV_ECUDA; }

// Benchmark hook state (nvfp4kv_profile_decode).
std::vector<cudaEvent_t> g_prof_before, g_prof_after;
size_t g_prof_next = 0;
size_t g_prof_every = 1;

}  // namespace

namespace {

int decode_entry(const nvfp4kv_cache *cache, const void *k_new, const void *v_new, int64_t new_stride, const void *q,
                 int batch, int num_q_heads, const int32_t *block_table, int max_pages_per_seq,
                 const int32_t *seq_lens, float sm_scale, void *out, void *workspace, size_t workspace_bytes,
                 int num_splits, cudaStream_t stream, const int32_t *shared_pages = nullptr, int shared_len = 0) {
    int rc = check_cache(cache);
    if (rc) return rc;
    if (batch < 0 || num_q_heads < 1 || num_q_heads % cache->num_kv_heads || num_splits < 0) return NVFP4KV_EINVAL;
    if (num_q_heads / cache->num_kv_heads > 16) return NVFP4KV_EUNSUPPORTED;
    if (!isfinite(sm_scale)) return NVFP4KV_EINVAL;
    if (batch == 0) return NVFP4KV_OK;
    if (!q || !block_table || !seq_lens || !out || !workspace) return NVFP4KV_EINVAL;
    if (max_pages_per_seq < 1) return NVFP4KV_EINVAL;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 256) || !aligned(block_table, 4) ||
        !aligned(seq_lens, 4))
        return NVFP4KV_EINVAL;
    if (k_new || v_new) {
        if (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return NVFP4KV_EINVAL;
        if (new_stride < (int64_t)cache->num_kv_heads * kHeadDim || new_stride % 8) return NVFP4KV_EINVAL;
    }
    if (shared_pages) {
        if (cache->dtype != NVFP4KV_DTYPE_NVFP4) return NVFP4KV_EUNSUPPORTED;
        if (!aligned(shared_pages, 4) || shared_len <= 0 || shared_len % 64 || shared_len % cache->page_size ||
            (int64_t)shared_len > (int64_t)max_pages_per_seq * cache->page_size)
            return NVFP4KV_EINVAL;
    }
    const int G = num_q_heads / cache->num_kv_heads;
    cudaError_t e = cudaSuccess;
    const int grid = num_splits ? num_splits : decode_auto_grid(*cache, G, &e);
    if (e != cudaSuccess || grid <= 0) return NVFP4KV_ECUDA;
    size_t need = decode_workspace_bytes(*cache, batch, num_q_heads, grid);
    if (shared_pages) need += cascade_extra_bytes(*cache, batch, num_q_heads, shared_len);
    if (workspace_bytes < need) return NVFP4KV_EINVAL;
    unsigned *err = error_word(&e);
    if (!err) return NVFP4KV_ECUDA;
    cudaEvent_t before = nullptr, after = nullptr;
    if (!g_prof_before.empty()) {
        const size_t call = g_prof_next++;
        if (call % g_prof_every == 0) {
            const size_t i = (call / g_prof_every) % g_prof_before.size();
            before = g_prof_before[i];
            after = g_prof_after[i];
        }
    }
    return from_cuda(launch_decode(*cache, q, batch, num_q_heads, block_table, max_pages_per_seq, seq_lens, sm_scale,
                                   out, workspace, grid, err, stream, before, after, k_new, v_new, new_stride,
                                   shared_pages, shared_len));
}

}  // namespace

extern "C" {

int nvfp4kv_version(void) { return 100; }

const char *nvfp4kv_status_string(int status) {
    switch (status) {
        case NVFP4KV_OK: return "ok";
        case NVFP4KV_EINVAL: return "invalid argument";
        case NVFP4KV_EUNSUPPORTED: return "unsupported configuration";
        case NVFP4KV_ECUDA: return "CUDA error";
        case NVFP4KV_EDEVICE_CHECK: return "a kernel skipped an out-of-range index (device error word set)";
        default: return "unknown status";
    }
}

size_t nvfp4kv_slab_bytes(const nvfp4kv_cache *cache) {
    if (!cache) return 0;
    nvfp4kv_cache c = *cache;
    if (!c.pool) c.pool = reinterpret_cast<void *>(256);  // layout query needs no pool
    return check_cache(&c) == NVFP4KV_OK ? slab_of(&c) : 0;
}

size_t nvfp4kv_pool_bytes(const nvfp4kv_cache *cache) {
    const size_t slab = nvfp4kv_slab_bytes(cache);
    return slab ? slab * (size_t)cache->num_pages * (size_t)cache->num_kv_heads : 0;
}

int nvfp4_kv_quantize_append(const nvfp4kv_cache *cache, const void *k, const void *v, int64_t num_tokens,
                             int64_t token_stride, const int64_t *slot_mapping, cudaStream_t stream) {
    int rc = check_cache(cache);
    if (rc) return rc;
    if (num_tokens < 0) return NVFP4KV_EINVAL;
    if (num_tokens == 0) return NVFP4KV_OK;
    if (!k || !v || !slot_mapping) return NVFP4KV_EINVAL;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8)) return NVFP4KV_EINVAL;
    if (token_stride < (int64_t)cache->num_kv_heads * kHeadDim || token_stride % 8) return NVFP4KV_EINVAL;
    if (num_tokens * cache->num_kv_heads * 16 >= ((int64_t)1 << 31)) return NVFP4KV_EUNSUPPORTED;
    cudaError_t e;
    unsigned *err = error_word(&e);
    if (!err) return NVFP4KV_ECUDA;
    return from_cuda(launch_quantize_append(*cache, k, v, num_tokens, token_stride, slot_mapping, err, stream));
}

int nvfp4_extend_attention(const void *q, const void *k_prefix, const void *v_prefix, const int32_t *cu_prefix_lens,
                           int64_t total_prefix_tokens, const void *k_chunk, const void *v_chunk,
                           const int32_t *cu_q_lens, int64_t total_q_tokens, int num_reqs, int max_q_len,
                           int num_q_heads, int num_kv_heads, float sm_scale, void *out, cudaStream_t stream) {
    if (num_reqs < 0 || max_q_len < 0 || num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads ||
        total_prefix_tokens < 0 || total_q_tokens < 0)
        return NVFP4KV_EINVAL;
    if (total_prefix_tokens >= ((int64_t)1 << 31) || total_q_tokens >= ((int64_t)1 << 31))
        return NVFP4KV_EUNSUPPORTED;
    if (!isfinite(sm_scale)) return NVFP4KV_EINVAL;
    if (num_reqs == 0 || max_q_len == 0) return NVFP4KV_OK;
    if (!q || !k_chunk || !v_chunk || !out || !cu_prefix_lens || !cu_q_lens || !k_prefix || !v_prefix)
        return NVFP4KV_EINVAL;
    if (!aligned(q, 16) || !aligned(k_chunk, 16) || !aligned(v_chunk, 16) || !aligned(out, 16) ||
        !aligned(k_prefix, 16) || !aligned(v_prefix, 16) || !aligned(cu_prefix_lens, 4) || !aligned(cu_q_lens, 4))
        return NVFP4KV_EINVAL;
    const int64_t G = num_q_heads / num_kv_heads;
    if ((int64_t)max_q_len * G >= ((int64_t)1 << 31) || num_kv_heads > 65535 || num_reqs > 65535)
        return NVFP4KV_EUNSUPPORTED;
    cudaError_t e;
    unsigned *err = error_word(&e);
    if (!err) return NVFP4KV_ECUDA;
    return from_cuda(launch_extend(q, k_prefix, v_prefix, cu_prefix_lens, total_prefix_tokens, k_chunk, v_chunk,
                                   cu_q_lens, total_q_tokens, num_reqs, max_q_len, num_q_heads, num_kv_heads, sm_scale,
                                   out, err, stream));
}

int nvfp4_extend_attention_paged(const nvfp4kv_cache *cache, const void *q, const int32_t *block_table,
                                 int max_pages_per_seq, const int32_t *prefix_lens, const void *k_chunk,
                                 const void *v_chunk, const int32_t *cu_q_lens, int64_t total_q_tokens, int num_reqs,
                                 int max_q_len, int num_q_heads, float sm_scale, void *out, cudaStream_t stream) {
    int rc = check_cache(cache);
    if (rc) return rc;
    if (cache->dtype != NVFP4KV_DTYPE_NVFP4) return NVFP4KV_EUNSUPPORTED;
    if (num_reqs < 0 || max_q_len < 0 || num_q_heads < 1 || num_q_heads % cache->num_kv_heads ||
        total_q_tokens < 0 || max_pages_per_seq < 1)
        return NVFP4KV_EINVAL;
    if (total_q_tokens >= ((int64_t)1 << 31)) return NVFP4KV_EUNSUPPORTED;
    if (!isfinite(sm_scale)) return NVFP4KV_EINVAL;
    if (num_reqs == 0 || max_q_len == 0) return NVFP4KV_OK;
    if (!q || !block_table || !prefix_lens || !k_chunk || !v_chunk || !cu_q_lens || !out) return NVFP4KV_EINVAL;
    if (!aligned(q, 16) || !aligned(k_chunk, 16) || !aligned(v_chunk, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(prefix_lens, 4) || !aligned(cu_q_lens, 4))
        return NVFP4KV_EINVAL;
    const int64_t G = num_q_heads / cache->num_kv_heads;
    if ((int64_t)max_q_len * G >= ((int64_t)1 << 31) || cache->num_kv_heads > 65535 || num_reqs > 65535 ||
        (int64_t)max_pages_per_seq * cache->page_size >= ((int64_t)1 << 31))
        return NVFP4KV_EUNSUPPORTED;
    cudaError_t e;
    unsigned *err = error_word(&e);
    if (!err) return NVFP4KV_ECUDA;
    return from_cuda(launch_extend_paged(*cache, q, block_table, max_pages_per_seq, prefix_lens, k_chunk, v_chunk,
                                         cu_q_lens, total_q_tokens, num_reqs, max_q_len, num_q_heads, sm_scale, out,
                                         err, stream));
}

int nvfp4kv_calibrate_global_scales(const void *k, const void *v, int64_t num_tokens, int num_kv_heads,
                                    int64_t token_stride, float *scales, cudaStream_t stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || !scales || !aligned(scales, 8)) return NVFP4KV_EINVAL;
    if (num_tokens > 0) {
        if (!k || !v || !aligned(k, 16) || !aligned(v, 16)) return NVFP4KV_EINVAL;
        if (token_stride < (int64_t)num_kv_heads * kHeadDim || token_stride % 8) return NVFP4KV_EINVAL;
    }
    return from_cuda(launch_calibrate(k, v, num_tokens, num_kv_heads, token_stride, scales, stream));
}

int nvfp4kv_decode_auto_splits(const nvfp4kv_cache *cache, int num_q_heads) {
    if (check_cache(cache) || num_q_heads < 1 || num_q_heads % cache->num_kv_heads) return 0;
    const int G = num_q_heads / cache->num_kv_heads;
    if (G > 16) return 0;
    return decode_auto_grid(*cache, G, nullptr);
}

int nvfp4kv_decode_launch_count(const nvfp4kv_cache *cache, int batch, int num_q_heads, int num_splits,
                                int shared_len) {
    if (check_cache(cache) || batch < 1 || num_q_heads < 1 || num_q_heads % cache->num_kv_heads || num_splits < 0 ||
        shared_len < 0 || num_q_heads / cache->num_kv_heads > 16)
        return 0;
    // (plan,) (shared prefix,) decode, reduction: a small batch without a shared prefix is planned in the decode CTAs
    return decode_plans_in_cta(batch, shared_len > 0) ? 2 : shared_len > 0 ? 4 : 3;
}

size_t nvfp4kv_decode_workspace_bytes(const nvfp4kv_cache *cache, int batch, int num_q_heads, int num_splits) {
    if (check_cache(cache) || batch < 0 || num_q_heads < 1 || num_q_heads % cache->num_kv_heads || num_splits < 0)
        return 0;
    const int G = num_q_heads / cache->num_kv_heads;
    if (G > 16) return 0;
    const int grid = num_splits ? num_splits : decode_auto_grid(*cache, G, nullptr);
    if (grid <= 0) return 0;
    return decode_workspace_bytes(*cache, batch, num_q_heads, grid);
}

int nvfp4_paged_decode_attention(const nvfp4kv_cache *cache, const void *q, int batch, int num_q_heads,
                                 const int32_t *block_table, int max_pages_per_seq, const int32_t *seq_lens,
                                 float sm_scale, void *out, void *workspace, size_t workspace_bytes, int num_splits,
                                 cudaStream_t stream) {
    return decode_entry(cache, nullptr, nullptr, 0, q, batch, num_q_heads, block_table, max_pages_per_seq, seq_lens,
                        sm_scale, out, workspace, workspace_bytes, num_splits, stream);
}

size_t nvfp4kv_cascade_workspace_bytes(const nvfp4kv_cache *cache, int batch, int num_q_heads, int num_splits,
                                       int shared_len) {
    const size_t base = nvfp4kv_decode_workspace_bytes(cache, batch, num_q_heads, num_splits);
    if (!base || shared_len <= 0 || shared_len % 64) return base;
    return base + cascade_extra_bytes(*cache, batch, num_q_heads, shared_len);
}

int nvfp4_cascade_decode_attention(const nvfp4kv_cache *cache, const void *q, int batch, int num_q_heads,
                                   const int32_t *shared_pages, int shared_len, const int32_t *block_table,
                                   int max_pages_per_seq, const int32_t *seq_lens, float sm_scale, void *out,
                                   void *workspace, size_t workspace_bytes, int num_splits, cudaStream_t stream) {
    if (!shared_pages) return NVFP4KV_EINVAL;
    return decode_entry(cache, nullptr, nullptr, 0, q, batch, num_q_heads, block_table, max_pages_per_seq, seq_lens,
                        sm_scale, out, workspace, workspace_bytes, num_splits, stream, shared_pages, shared_len);
}

int nvfp4_paged_decode_attention_append(const nvfp4kv_cache *cache, const void *k_new, const void *v_new,
                                        int64_t new_stride, const void *q, int batch, int num_q_heads,
                                        const int32_t *block_table, int max_pages_per_seq, const int32_t *seq_lens,
                                        float sm_scale, void *out, void *workspace, size_t workspace_bytes,
                                        int num_splits, cudaStream_t stream) {
    if (!k_new || !v_new) return NVFP4KV_EINVAL;
    return decode_entry(cache, k_new, v_new, new_stride, q, batch, num_q_heads, block_table, max_pages_per_seq,
                        seq_lens, sm_scale, out, workspace, workspace_bytes, num_splits, stream);
}

int nvfp4_prefix_dequant(const nvfp4kv_cache *cache, const int32_t *block_table, int max_pages_per_seq,
                         const int32_t *prefix_lens, const int32_t *cu_prefix_lens, int num_reqs,
                         int64_t total_prefix_tokens, void *k_ws, void *v_ws, cudaStream_t stream) {
    int rc = check_cache(cache);
    if (rc) return rc;
    if (num_reqs < 0 || total_prefix_tokens < 0) return NVFP4KV_EINVAL;
    if (num_reqs == 0 || total_prefix_tokens == 0) return NVFP4KV_OK;
    if (!block_table || !prefix_lens || !cu_prefix_lens || !k_ws || !v_ws || max_pages_per_seq < 1)
        return NVFP4KV_EINVAL;
    if (!aligned(k_ws, 16) || !aligned(v_ws, 16)) return NVFP4KV_EINVAL;
    if (total_prefix_tokens * cache->num_kv_heads * 16 >= ((int64_t)1 << 31)) return NVFP4KV_EUNSUPPORTED;
    cudaError_t e;
    unsigned *err = error_word(&e);
    if (!err) return NVFP4KV_ECUDA;
    return from_cuda(launch_prefix_dequant(*cache, block_table, max_pages_per_seq, prefix_lens, cu_prefix_lens,
                                           num_reqs, total_prefix_tokens, k_ws, v_ws, err, stream));
}

int nvfp4kv_profile_decode(const cudaEvent_t *before, const cudaEvent_t *after, int count, int every) {
    g_prof_before.clear();
    g_prof_after.clear();
    g_prof_next = 0;
    g_prof_every = 1;
    if (count < 0 || every < 1) return NVFP4KV_EINVAL;
    g_prof_every = (size_t)every;
    if (count == 0 || !before || !after) return NVFP4KV_OK;
    for (int i = 0; i < count; i++) {
        if (!before[i] || !after[i]) {
            g_prof_before.clear();
            g_prof_after.clear();
            return NVFP4KV_EINVAL;
        }
        g_prof_before.push_back(before[i]);
        g_prof_after.push_back(after[i]);
    }
    return NVFP4KV_OK;
}

int nvfp4kv_selftest_bounded_wait(int arrive, unsigned poll_limit, int *result, cudaStream_t stream) {
    if (!result || !aligned(result, 4) || poll_limit == 0 || poll_limit > (1u << 24)) return NVFP4KV_EINVAL;
    cudaError_t e;
    unsigned *err = error_word(&e);
    if (!err) return NVFP4KV_ECUDA;
    return from_cuda(launch_bounded_wait_selftest(arrive, poll_limit, result, err, stream));
}

int nvfp4kv_check_device_errors(cudaStream_t stream) {
    cudaError_t e;
    unsigned *err = error_word(&e);
    if (!err) return NVFP4KV_ECUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NVFP4KV_ECUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return NVFP4KV_ECUDA;
    if (word) {
        const unsigned zero = 0;
        if (cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return NVFP4KV_ECUDA;
        return NVFP4KV_EDEVICE_CHECK;
    }
    return NVFP4KV_OK;
}

}  // extern "C"
