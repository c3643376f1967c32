// common.cuh -- device helpers shared by the NVFP4 KV cache kernels (sm_103a).
//
// Inline PTX wrappers for the Blackwell features the kernels use: mbarrier
// completion of 1-D bulk (TMA) copies into shared memory, the hardware E2M1 and
// E4M3 conversions, movmatrix, and the f16 tensor-core MMA.  Nothing here is
// generated or copied from a compiled library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4kv.h"

namespace nvfp4kv {

constexpr int kHeadDim = 128;
constexpr int kBlock = 16;

// Bits of the per-device error word (see nvfp4kv_check_device_errors).
enum : unsigned {
    kErrSlot = 1u,      // slot_mapping entry >= num_pages * P
    kErrPage = 2u,      // block_table entry outside [0, num_pages)
    kErrSeqLen = 4u,    // seq_len / prefix_len negative or beyond the table
    kErrTimeout = 8u,   // an mbarrier wait exceeded its iteration limit
    kErrCuPrefix = 16u  // cu_prefix_lens inconsistent with prefix_lens
};

__device__ __forceinline__ void flag_error(unsigned *err, unsigned bit) { atomicOr(err, bit); }

// ---------------------------------------------------------------- conversions

// Two E2M1 codes in one byte (element 2i low nibble) -> f16x2 (low half = low nibble).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low_bits) {
    uint32_t r;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "r"(byte_in_low_bits));
    return r;
}

// The four bytes of w, each holding two E2M1 codes -> four f16x2.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                                  uint32_t &r3) {
    asm("{ .reg .b8 a, b, c, d; mov.b32 {a, b, c, d}, %4;\n"
        "  cvt.rn.f16x2.e2m1x2 %0, a; cvt.rn.f16x2.e2m1x2 %1, b;\n"
        "  cvt.rn.f16x2.e2m1x2 %2, c; cvt.rn.f16x2.e2m1x2 %3, d; }"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(w));
}

// Two E4M3 codes (low byte -> low half) -> f16x2; exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t r;
    uint16_t h = (uint16_t)two_bytes;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
    return r;
}

// Round-to-nearest-even, saturating: (hi, lo) floats -> two E4M3 bytes (lo in the low byte).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Round-to-nearest-even, saturating: (hi, lo) floats -> one byte of two E2M1 codes (lo in the low nibble).
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float hi, float lo) {
    uint32_t r;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float hi, float lo) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Transpose an 8x8 b16 matrix held in the standard fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of phase completion.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: returns false after `limit` unsuccessful polls (the caller
// records kErrTimeout and winds down instead of spinning forever).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit,
                                                  const volatile int *abort_flag) {
    for (uint32_t i = 0; i < limit; i++) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (i > 64) __nanosleep(64);
    }
    return false;
}

// 1-D bulk copy global -> shared, completion signalled on `bar` (complete_tx).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- programmatic dependent launch
//
// A kernel launched with launch_pdl() may start while the previous kernel of
// the stream is still running, once every CTA of that kernel has executed
// pdl_launch_dependents() (or exited).  pdl_wait() blocks until the previous
// kernel has completed and its memory operations are visible, so it must
// come before the first access to anything that kernel (or earlier work)
// writes.  Without a programmatic dependency both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

inline cudaError_t launch_pdl(const void *fn, dim3 grid, unsigned block, size_t smem, cudaStream_t stream,
                              void **args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// ---------------------------------------------------------------- misc

__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace nvfp4kv
