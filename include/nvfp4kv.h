/*
 * nvfp4kv.h -- C ABI of the NVFP4 paged KV cache library (libnvfp4kv.so).
 *
 * The library implements the three cache paths of "Accelerating Long-Context
 * and Agentic Inference with NVFP4 KV Cache" (section A2) on one GB300 GPU
 * (sm_103a), as hand-written CUDA:
 *
 *   nvfp4_kv_quantize_append      -- new K/V written into the paged cache
 *                                    (path 1 "initial prefill" writes its
 *                                    FP8/BF16 KV this way; path 2 appends the
 *                                    new chunk this way).
 *   nvfp4_paged_decode_attention  -- path 3 "decode": the kernel reads packed
 *                                    4-bit values and block scales, dequantises
 *                                    them on chip (Fig. 3) and never writes
 *                                    dequantised KV back to HBM.
 *   nvfp4_prefix_dequant          -- path 2 "chunked prefill / extend": the
 *                                    cached prefix is expanded into a reusable
 *                                    workspace shared across layers.
 *
 * Format (section A3 and Fig. 1): each run of 16 consecutive values along
 * head_dim is one block with an FP8 E4M3 scale; values are 4-bit E2M1; an
 * FP32 tensor scale multiplies everything (fixed at 1.0 on the page, A7).
 * 16 values take 8 bytes + 1 scale byte, (8 + 1) / 16 = 0.5625 of FP8
 * (section A2, storage ratio formula).  An FP8 E4M3 cache (the page's
 * fp8_e4m3 baseline, A4) is supported for comparison.
 *
 * Conventions for every call:
 *   - All buffers are caller-owned DEVICE memory unless stated otherwise.  The
 *     library never allocates device memory; calls that need scratch take a
 *     caller-sized workspace.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream) and do
 *     not synchronise.  Arguments are validated on the host before any launch;
 *     a rejected call launches nothing and returns a negative status.
 *   - Indices a call reads from device memory (slot mapping, block table
 *     entries, lengths) are range-checked on the device.  An out-of-range index
 *     is skipped (never dereferenced) and recorded in a per-device error word
 *     that nvfp4kv_check_device_errors() reports.  No kernel traps or asserts.
 *   - head_dim is 128.  page_size P is 16, 32, 64 or 128 tokens.
 *   - Per device, the library keeps the device addresses of its own
 *     __device__ variables (the error word, the no-alloc scratch array) and
 *     kernel attributes it has set, from the first call on that device.  They
 *     belong to the device's primary context: after cudaDeviceReset (or any
 *     teardown of the primary context) the library must not be called again
 *     in that process.
 *
 * Pool layout, one slab per (page, kv_head), slabs ordered page-major:
 *   pool = uint8[num_pages][num_kv_heads][slab_bytes]
 *   A slab is P/16 groups of 16 consecutive token rows; group j (rows 16j ..
 *   16j+15) starts at byte j * group_bytes and holds, for its rows r = 0..15:
 *   NVFP4 group (2304 bytes, slab = 144 * P):
 *     K codes  uint8[16][64]  byte i of row r = element 2i (low nibble) and
 *                             element 2i+1 (high nibble) of that token's K row
 *     K scales uint8[16][8]   E4M3 scale of block b (elements 16b..16b+15)
 *     V codes  uint8[16][64]  as K codes
 *     V scales uint8[8][16]   block-major: scale of block b of row r at [b][r]
 *   FP8 group (4096 bytes, slab = 256 * P):  K uint8[16][128] | V uint8[16][128]
 *   Token position t of a sequence is row t % P of page block_table[t / P].
 *   A nibble is an E2M1 code: bit 3 sign, bits 2..0 magnitude index into
 *   {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 */
#ifndef NVFP4KV_H
#define NVFP4KV_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define NVFP4KV_API __attribute__((visibility("default")))
#else
#define NVFP4KV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum {
    NVFP4KV_OK = 0,
    NVFP4KV_EINVAL = -1,        /* a pointer, size, shape or alignment is invalid */
    NVFP4KV_EUNSUPPORTED = -2,  /* valid request outside what this build implements */
    NVFP4KV_ECUDA = -3,         /* a CUDA runtime call or kernel launch failed */
    NVFP4KV_EDEVICE_CHECK = -4  /* a kernel found an out-of-range index (see conventions) */
} nvfp4kv_status;

typedef enum {
    NVFP4KV_DTYPE_NVFP4 = 0,    /* E2M1 values + E4M3 scale per 16 */
    NVFP4KV_DTYPE_FP8_E4M3 = 1  /* one E4M3 code per value */
} nvfp4kv_dtype;

/* Describes a caller-owned page pool.  The library reads it, never frees it. */
typedef struct {
    void *pool;             /* device, uint8[num_pages][num_kv_heads][slab_bytes], 256-byte aligned */
    int64_t num_pages;      /* >= 1 */
    int32_t page_size;      /* P: 16, 32, 64 or 128 tokens */
    int32_t num_kv_heads;   /* >= 1 */
    int32_t head_dim;       /* must be 128 */
    int32_t dtype;          /* nvfp4kv_dtype */
    float k_global_scale;   /* FP32 tensor scale of K, a positive normal FP32 number (>= 2^-126; 1.0 on the page) */
    float v_global_scale;   /* FP32 tensor scale of V, a positive normal FP32 number */
} nvfp4kv_cache;

/* Bytes of one (page, kv_head) slab: 144*P (NVFP4) or 256*P (FP8); 0 if the
 * descriptor is invalid. */
NVFP4KV_API size_t nvfp4kv_slab_bytes(const nvfp4kv_cache *cache);

/* Bytes of the whole pool (num_pages * num_kv_heads * slab); 0 if invalid. */
NVFP4KV_API size_t nvfp4kv_pool_bytes(const nvfp4kv_cache *cache);

/*
 * Quantise BF16 K and V rows and write them into the pool.
 * Source: section A2, path 1 (KV quantised to NVFP4 and written to the
 * persistent cache) and path 2 (the new chunk's KV quantised and appended).
 *
 *   k, v          device BF16 [num_tokens][token_stride]; the row of kv head h
 *                 is elements h*128 .. h*128+127 of the token.  16-byte aligned.
 *   token_stride  elements between consecutive tokens; >= num_kv_heads*128 and
 *                 a multiple of 8.
 *   slot_mapping  device int64 [num_tokens]: slot = page * P + row.  A negative
 *                 slot skips the token; a slot >= num_pages * P is skipped and
 *                 flagged in the device error word.
 * Per block of 16 values x_i (g = the tensor scale of K or V):
 *   scale  = E4M3(amax_i |x_i| / (6 g)),  round to nearest even, saturating;
 *   code_i = E2M1(x_i / (scale g)),       round to nearest even, saturating;
 *            a block whose scale is 0 stores signed zeros.
 * Each scale and code is the rounding of the exact quotient, for every tensor
 * scale g (the kernel decides the cases an FP32 quotient would get wrong with
 * exact fused multiply-add comparisons against the rounding midpoints).
 * FP8 pools store E4M3(x_i / g) per value, rounded the same way.  Two tokens writing the same slot
 * in one call is a caller error (the result is one of the two rows).
 * num_tokens == 0 is a no-op.
 */
NVFP4KV_API int nvfp4_kv_quantize_append(const nvfp4kv_cache *cache, const void *k, const void *v, int64_t num_tokens,
                             int64_t token_stride, const int64_t *slot_mapping, cudaStream_t stream);

/*
 * Calibrate the per-tensor FP32 global scales of K and V.
 * Source: section A4 (outlook): the page's benchmarks fix the FP32 tensor
 * scale at 1.0 and name its calibration as the way to avoid overflow and
 * underflow of the block scales.  The rule used is the two-level NVFP4 one:
 *   g = amax / (6 * 448)   (FP32 IEEE division; g = 1 when amax = 0),
 * amax = the largest finite |x| over all num_tokens x num_kv_heads x 128 BF16
 * values of the tensor (Inf and NaN are ignored), so the block holding amax
 * gets the largest E4M3 scale and no block scale saturates.
 *
 *   k, v          device BF16 [num_tokens][token_stride], layout as for
 *                 nvfp4_kv_quantize_append (16-byte aligned; unused if
 *                 num_tokens == 0).
 *   scales        device float[2], 8-byte aligned, written with {g_K, g_V}
 *                 (also used as scratch while the call runs on `stream`).
 * Pass the results as k_global_scale / v_global_scale of the cache
 * descriptor before appending.  A tensor whose largest finite magnitude is
 * below 2^-126 * 2688 (about 3.2e-35) gets a subnormal g, which the cache
 * descriptor does not accept (a tensor scale is a positive normal FP32
 * number): keep g = 1 for such a tensor.  Returns NVFP4KV_EINVAL for a bad
 * argument.
 */
NVFP4KV_API int nvfp4kv_calibrate_global_scales(const void *k, const void *v, int64_t num_tokens, int num_kv_heads,
                                                int64_t token_stride, float *scales, cudaStream_t stream);

/* Workspace bytes nvfp4_paged_decode_attention needs for this shape and
 * num_splits on the current device (0 if the arguments are invalid). */
NVFP4KV_API size_t nvfp4kv_decode_workspace_bytes(const nvfp4kv_cache *cache, int batch, int num_q_heads, int num_splits);

/* Number of work partitions an auto-split (num_splits = 0) call uses on the
 * current device for this cache. */
NVFP4KV_API int nvfp4kv_decode_auto_splits(const nvfp4kv_cache *cache, int num_q_heads);

/* Kernel launches one nvfp4_paged_decode_attention (shared_len = 0) or
 * nvfp4_cascade_decode_attention (shared_len > 0) call of this shape makes:
 * the decode kernel and the log-sum-exp reduction (2) for a batch of at most
 * 96 sequences, which every decode CTA plans itself from seq_lens; the plan
 * kernel as well (3) for a larger batch; the plan and the shared-prefix kernel
 * as well (4) for a cascade call.  The fused append variant makes as many.
 * 0 if the arguments are invalid (or batch = 0: nothing is launched). */
NVFP4KV_API int nvfp4kv_decode_launch_count(const nvfp4kv_cache *cache, int batch, int num_q_heads, int num_splits,
                                            int shared_len);

/*
 * Paged GQA decode attention over the cache, one query token per sequence.
 * Source: section A2, path 3 and Fig. 3 (packed K/V tiles and block scales
 * staged in shared memory, unpacked in registers, scaled, matrix products on
 * the dequantised values, tensor scales applied as product scaling).
 *
 *   q            device BF16 [batch][num_q_heads][128], 16-byte aligned
 *   block_table  device int32 [batch][max_pages_per_seq]; only the first
 *                ceil(seq_lens[b] / P) entries of row b are read
 *   seq_lens     device int32 [batch]; 0 <= seq_lens[b] <= max_pages_per_seq*P
 *                (a larger value is clamped and flagged)
 *   out          device BF16 [batch][num_q_heads][128], 16-byte aligned
 *   workspace    device, >= nvfp4kv_decode_workspace_bytes(...) bytes,
 *                256-byte aligned; holds split-KV partials and the work plan
 *   num_splits   number of work partitions the KV range is cut into (each
 *                becomes one CTA; partials are merged by a log-sum-exp
 *                reduction kernel); 0 = auto, a multiple of the SM count.
 * Query head h attends KV head h / G, G = num_q_heads / num_kv_heads <= 16.
 *   out[b][h] = sum_t softmax_t(sm_scale * g_K * q_h . k_t) * g_V * v_t
 * over t < seq_lens[b], with k_t, v_t the dequantised cache rows.  A sequence
 * of length 0 yields zeros.
 */
NVFP4KV_API int nvfp4_paged_decode_attention(const nvfp4kv_cache *cache, const void *q, int batch, int num_q_heads,
                                 const int32_t *block_table, int max_pages_per_seq, const int32_t *seq_lens,
                                 float sm_scale, void *out, void *workspace, size_t workspace_bytes, int num_splits,
                                 cudaStream_t stream);

/*
 * Cascade decode: decode attention for sequences that all begin with the same
 * shared_len tokens, stored once in the pages shared_pages[0 ..
 * shared_len/P - 1] (and listed first in every sequence's block table).
 * Source: section A4 (agentic workloads share a long common prefix, kept once
 * by the radix cache) and section A2, path 3.  The shared pages are read and
 * dequantised once per kv head and multiplied with the queries of all
 * sequences together; each sequence's remaining tokens are decoded as in
 * nvfp4_paged_decode_attention, and the two partial softmaxes are merged by
 * log-sum-exp.  The result equals nvfp4_paged_decode_attention on the same
 * arguments up to floating-point summation order.
 *
 *   shared_pages  device int32 [shared_len / P] page ids.
 *   shared_len    tokens of the shared prefix: > 0, a multiple of 64 and of P.
 *   workspace     device, >= nvfp4kv_cascade_workspace_bytes(...), 256-aligned.
 * Every seq_lens[b] must be >= shared_len (a shorter one is flagged in the
 * device error word and only its shared part is attended).  NVFP4 pools only
 * (NVFP4KV_EUNSUPPORTED for FP8).  Other arguments as
 * nvfp4_paged_decode_attention.
 */
NVFP4KV_API size_t nvfp4kv_cascade_workspace_bytes(const nvfp4kv_cache *cache, int batch, int num_q_heads,
                                                   int num_splits, int shared_len);
NVFP4KV_API int nvfp4_cascade_decode_attention(const nvfp4kv_cache *cache, const void *q, int batch,
                                               int num_q_heads, const int32_t *shared_pages, int shared_len,
                                               const int32_t *block_table, int max_pages_per_seq,
                                               const int32_t *seq_lens, float sm_scale, void *out,
                                               void *workspace, size_t workspace_bytes, int num_splits,
                                               cudaStream_t stream);

/*
 * Decode step with the new token appended in the same launch.
 * Source: section A2, path 3 (decode reads the NVFP4 cache in-kernel) with
 * path 1's quantise-and-write of the new token's K/V fused in front of it.
 * For every sequence b with seq_lens[b] >= 1, row b of k_new / v_new (the
 * token at position seq_lens[b] - 1, already counted in seq_lens) is
 * quantised exactly as nvfp4_kv_quantize_append would, and written through
 * the block table to position seq_lens[b] - 1; then attention runs as in
 * nvfp4_paged_decode_attention.  The result, pool and output alike, equals
 * nvfp4_kv_quantize_append with slot_mapping[b] = slot(seq_lens[b] - 1)
 * followed by nvfp4_paged_decode_attention.
 *
 *   k_new, v_new  device BF16 [batch][new_stride], kv head h at elements
 *                 h*128 .. h*128+127 of a row; 16-byte aligned.
 *   new_stride    elements between rows; >= num_kv_heads*128, a multiple of 8.
 * Other arguments, workspace and errors as nvfp4_paged_decode_attention; a
 * block-table entry out of range for the new token skips its write and is
 * flagged in the device error word.
 */
NVFP4KV_API int nvfp4_paged_decode_attention_append(const nvfp4kv_cache *cache, const void *k_new, const void *v_new,
                                                    int64_t new_stride, const void *q, int batch, int num_q_heads,
                                                    const int32_t *block_table, int max_pages_per_seq,
                                                    const int32_t *seq_lens, float sm_scale, void *out,
                                                    void *workspace, size_t workspace_bytes, int num_splits,
                                                    cudaStream_t stream);

/* Size of the library's static scratch array used by
 * nvfp4_paged_decode_attention_noalloc (64 MiB on every GPU that loads the
 * library, held until the process exits). */
#define NVFP4KV_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * Paged decode attention for callers that cannot allocate device memory (a
 * host framework that owns every allocation, or a latency-critical path where
 * cudaMalloc's possible device synchronisation is not acceptable).  No
 * counterpart on the page: it is nvfp4_paged_decode_attention with the
 * workspace taken from a static __device__ array of the library instead of
 * the caller; arguments and results are the same, minus the workspace.
 *   - Allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 *   - Needs nvfp4kv_decode_workspace_bytes(cache, batch, num_q_heads,
 *     num_splits) <= NVFP4KV_NOALLOC_SCRATCH_BYTES; a larger request returns
 *     NVFP4KV_EUNSUPPORTED and launches nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it for the
 *     life of the process; make that first call before any stream capture.
 *     A cudaDeviceReset (or anything else that destroys the device's primary
 *     context) invalidates the kept address: do not call this entry point on
 *     a device after resetting it.
 *   - Every call shares the one array, which keeps the last call's contents:
 *     calls that overlap on the GPU (e.g. on unordered streams) race.  No part
 *     of the array needs to start at zero.
 */
NVFP4KV_API int nvfp4_paged_decode_attention_noalloc(const nvfp4kv_cache *cache, const void *q, int batch,
                                                     int num_q_heads, const int32_t *block_table,
                                                     int max_pages_per_seq, const int32_t *seq_lens, float sm_scale,
                                                     void *out, int num_splits, cudaStream_t stream);

/*
 * Dequantise cached prefixes into a contiguous BF16 workspace.
 * Source: section A2, path 2 (cached prefix entries gathered, dequantised into
 * a layer-shared workspace that the new chunk's KV joins before attention).
 * The page writes an FP8 workspace; this library writes BF16, which holds
 * every dequantised NVFP4 value exactly (at most 5 significant bits).
 *
 *   block_table     device int32 [num_reqs][max_pages_per_seq]
 *   prefix_lens     device int32 [num_reqs]
 *   cu_prefix_lens  device int32 [num_reqs + 1], cu[0] = 0, cu[r+1] = cu[r] + prefix_lens[r]
 *   total_prefix_tokens  host copy of cu[num_reqs] (sizes the launch)
 *   k_ws, v_ws      device BF16 [total_prefix_tokens][num_kv_heads][128],
 *                   16-byte aligned; row cu[r] + t receives prefix token t of
 *                   request r:  value = the exact product e2m1 * e4m3 * g
 *                   rounded once to BF16, nearest-even (exact for g = 1);
 *                   FP8 pools: e4m3 * g rounded the same way.
 */
NVFP4KV_API int nvfp4_prefix_dequant(const nvfp4kv_cache *cache, const int32_t *block_table, int max_pages_per_seq,
                         const int32_t *prefix_lens, const int32_t *cu_prefix_lens, int num_reqs,
                         int64_t total_prefix_tokens, void *k_ws, void *v_ws, cudaStream_t stream);

/*
 * Extend attention: each request's new chunk attends to [its cached prefix ||
 * the chunk itself], causally within the chunk.
 * Source: section A2, path 2 (chunked prefill / extend): the attention
 * consumes the cached prefix as the layer-shared workspace holds it (written
 * by nvfp4_prefix_dequant) and the current chunk's K/V.  Chunk token i of
 * request r sees all prefix tokens of r and chunk tokens 0..i:
 *   out[t][h] = sum_j softmax_j(sm_scale * q[t][h] . k_j) v_j
 * over those keys, with query head h reading KV head h / G.
 *
 *   q               device BF16 [total_q][num_q_heads][128]; request r's
 *                   chunk is rows cu_q_lens[r] .. cu_q_lens[r+1]-1.
 *   k_prefix, v_prefix  device BF16 [total_prefix][num_kv_heads][128]; request
 *                   r's prefix is rows cu_prefix_lens[r] .. cu_prefix_lens[r+1]-1
 *                   (the nvfp4_prefix_dequant workspace layout).
 *   k_chunk, v_chunk    device BF16 [total_q][num_kv_heads][128], rows as q.
 *   cu_prefix_lens, cu_q_lens  device int32 [num_reqs + 1], non-decreasing.
 *   total_prefix_tokens, total_q_tokens  host: rows of k_prefix / v_prefix
 *                   and of q, k_chunk, v_chunk (the kernel's copies stay
 *                   inside them: rows past a request are read but masked).
 *   max_q_len       host bound on every chunk length (grid size); a longer
 *                   chunk is cut to it and flagged in the device error word.
 *   out             device BF16 [total_q][num_q_heads][128].
 * All data pointers 16-byte aligned.  Computes in BF16 x BF16 -> FP32 on the
 * tensor cores (probabilities rounded to BF16).  num_reqs == 0 is a no-op.
 * Needs the driver's tensor-map encoder (NVFP4KV_ECUDA if it is missing).
 */
NVFP4KV_API int nvfp4_extend_attention(const void *q, const void *k_prefix, const void *v_prefix,
                                       const int32_t *cu_prefix_lens, int64_t total_prefix_tokens,
                                       const void *k_chunk, const void *v_chunk, const int32_t *cu_q_lens,
                                       int64_t total_q_tokens, int num_reqs, int max_q_len, int num_q_heads,
                                       int num_kv_heads, float sm_scale, void *out, cudaStream_t stream);

/*
 * Extend attention with the prefix read straight from the NVFP4 cache: path 2
 * of section A2 without the BF16 workspace.  Request r's prefix is tokens
 * 0 .. prefix_lens[r] - 1 of its pages (row r of block_table); the kernel
 * expands each 128-token tile of them to BF16 (e2m1 * e4m3 * g, rounded once,
 * as nvfp4_prefix_dequant writes it) in shared memory and attends as
 * nvfp4_extend_attention does, so the result equals nvfp4_prefix_dequant
 * followed by nvfp4_extend_attention on the same data, bit for bit.
 *
 *   cache           the NVFP4 pool (an FP8 pool gives NVFP4KV_EUNSUPPORTED);
 *                   num_kv_heads is the cache's.
 *   block_table     device int32 [num_reqs][max_pages_per_seq].
 *   prefix_lens     device int32 [num_reqs], 0 <= prefix_lens[r] <=
 *                   max_pages_per_seq * P (a larger one is clamped and flagged;
 *                   a page id outside the pool is flagged and read as zeros).
 *   q, k_chunk, v_chunk, cu_q_lens, total_q_tokens, max_q_len, out, sm_scale
 *                   as for nvfp4_extend_attention.
 */
NVFP4KV_API int nvfp4_extend_attention_paged(const nvfp4kv_cache *cache, const void *q, const int32_t *block_table,
                                             int max_pages_per_seq, const int32_t *prefix_lens, const void *k_chunk,
                                             const void *v_chunk, const int32_t *cu_q_lens, int64_t total_q_tokens,
                                             int num_reqs, int max_q_len, int num_q_heads, float sm_scale, void *out,
                                             cudaStream_t stream);

/* Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns NVFP4KV_OK, NVFP4KV_EDEVICE_CHECK (some kernel skipped an
 * out-of-range index since the last check) or NVFP4KV_ECUDA. */
NVFP4KV_API int nvfp4kv_check_device_errors(cudaStream_t stream);

/* Failure-path self-test (no counterpart on the pages; for tests of failure
 * detection).  Launches one warp on `stream` that waits on an mbarrier phase
 * with the same bounded wait the decode kernel uses on its bulk copies:
 * the phase completes only if `arrive` != 0.  After `poll_limit` unsuccessful
 * polls (1 .. 2^24) the wait gives up, the kernel writes 1 to *result (device
 * int, 4-byte aligned) and sets the timeout bit of the device error word, as a
 * decode kernel whose copy never landed would; otherwise it writes 0.  The
 * kernel then returns normally, so the context stays usable.  Returns
 * NVFP4KV_EINVAL for a bad argument, NVFP4KV_ECUDA if the launch fails. */
NVFP4KV_API int nvfp4kv_selftest_bounded_wait(int arrive, unsigned poll_limit, int *result, cudaStream_t stream);

/* Benchmark hook: while enabled, every `every`-th decode call (of
 * nvfp4_paged_decode_attention or nvfp4_paged_decode_attention_append: calls
 * 0, every, 2*every, ...; the j-th of them uses pair j % count)
 * records before[] on its stream immediately before launching the decode
 * kernel and after[] immediately after it, so the caller can time that kernel
 * alone with cudaEventElapsedTime while the calls in between run undisturbed
 * (an event between the launches keeps the decode kernel from starting early
 * under programmatic dependent launch).  The events are created and owned by
 * the caller; count = 0 (or NULL arrays) disables the hook and resets the call
 * counter; every < 1 is EINVAL.  Process-wide and not thread-safe: for
 * benchmarks only. */
NVFP4KV_API int nvfp4kv_profile_decode(const cudaEvent_t *before, const cudaEvent_t *after, int count, int every);

/* Static description of a status code. */
NVFP4KV_API const char *nvfp4kv_status_string(int status);

/* Library ABI version (major * 100 + minor). */
NVFP4KV_API int nvfp4kv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4KV_H */
