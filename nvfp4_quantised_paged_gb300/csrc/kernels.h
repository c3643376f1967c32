// kernels.h -- internal launchers of the NVFP4 KV cache kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <vector_types.h>

#include "nvfp4kv.h"

namespace nvfp4kv {

cudaError_t launch_quantize_append(const nvfp4kv_cache &c, const void *k, const void *v, int64_t num_tokens,
                                   int64_t token_stride, const int64_t *slot_mapping, unsigned *err,
                                   cudaStream_t stream);

cudaError_t launch_prefix_dequant(const nvfp4kv_cache &c, const int32_t *block_table, int max_pages,
                                  const int32_t *prefix_lens, const int32_t *cu, int num_reqs, int64_t total,
                                  void *k_ws, void *v_ws, unsigned *err, cudaStream_t stream);

// Number of decode CTAs an auto split uses (SM count x resident CTAs per SM).
int decode_auto_grid(const nvfp4kv_cache &c, int group, cudaError_t *status);

// Whether a decode call plans its split inside the decode CTAs (a small batch
// without a shared prefix) instead of launching the plan kernel first.
bool decode_plans_in_cta(int batch, bool shared_prefix);

// Workspace bytes for a decode call with `grid` CTAs.
size_t decode_workspace_bytes(const nvfp4kv_cache &c, int batch, int num_q_heads, int grid);

// before / after: optional events recorded around the decode kernel launch.
// k_new / v_new (nullptr: no fused append): BF16 rows [batch][new_stride]
// quantised into position seq_lens[b] - 1 of each sequence before attending.
cudaError_t launch_decode(const nvfp4kv_cache &c, const void *q, int batch, int num_q_heads,
                          const int32_t *block_table, int max_pages, const int32_t *seq_lens, float sm_scale,
                          void *out, void *workspace, int grid, unsigned *err, cudaStream_t stream,
                          cudaEvent_t before, cudaEvent_t after, const void *k_new = nullptr,
                          const void *v_new = nullptr, int64_t new_stride = 0,
                          const int32_t *shared_pages = nullptr, int shared_len = 0);

// Number of slices the shared prefix is cut into (each leaves one partial per
// row), and the extra workspace bytes of a cascade call.
int cascade_splits(const nvfp4kv_cache &c, int batch, int num_q_heads, int shared_len);
size_t cascade_extra_bytes(const nvfp4kv_cache &c, int batch, int num_q_heads, int shared_len);

// Partials (m, l, acc) of every sequence's query heads over the shared prefix
// (shared_len tokens in pages shared_pages[]), `splits` slices of it, one
// partial per (slice, sequence, kv head, head).
cudaError_t launch_shared_prefix(const nvfp4kv_cache &c, const void *q, int batch, int num_q_heads,
                                 const int32_t *shared_pages, int shared_len, int splits, float sm_scale,
                                 float2 *casc_ml, float *casc_acc, unsigned *err, cudaStream_t stream);

// Attention of each request's chunk over [its BF16 prefix rows || its chunk], causal in the chunk.
cudaError_t launch_extend(const void *q, const void *k_prefix, const void *v_prefix, const int32_t *cu_prefix,
                          int64_t total_prefix, const void *k_chunk, const void *v_chunk, const int32_t *cu_q,
                          int64_t total_q, int num_reqs, int max_q_len, int num_q_heads, int num_kv_heads,
                          float sm_scale, void *out, unsigned *err, cudaStream_t stream);

// The same with request r's prefix read from the NVFP4 pool through row r of
// the block table (prefix_lens[r] tokens) and expanded to BF16 in the kernel.
cudaError_t launch_extend_paged(const nvfp4kv_cache &c, const void *q, const int32_t *block_table, int max_pages,
                                const int32_t *prefix_lens, const void *k_chunk, const void *v_chunk,
                                const int32_t *cu_q, int64_t total_q, int num_reqs, int max_q_len, int num_q_heads,
                                float sm_scale, void *out, unsigned *err, cudaStream_t stream);

// g_K, g_V = amax / (6 * 448) of K and V (1.0 for an all-zero tensor) into scales[0..1].
cudaError_t launch_calibrate(const void *k, const void *v, int64_t num_tokens, int num_kv_heads, int64_t token_stride,
                             float *scales, cudaStream_t stream);

// One warp waits, at most poll_limit polls, on an mbarrier phase that completes
// only if `arrive`; writes 1 to *result (and kErrTimeout to *err) if it gave up.
cudaError_t launch_bounded_wait_selftest(int arrive, uint32_t poll_limit, int *result, unsigned *err,
                                         cudaStream_t stream);

}  // namespace nvfp4kv
