// calibrate.cu -- per-tensor FP32 global scales of K and V from their absolute maxima.
//
// Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV
// Cache", section A4 (limitations and outlook): the benchmarks fix the
// per-tensor FP32 global scale of the NVFP4 format at 1.0, and calibrating
// it is named as the way to remove the overflow and underflow of block
// scales.  Calibration here is the plain two-level NVFP4 rule: g = amax / (6 *
// 448), so that the block holding the tensor's largest magnitude gets the
// largest E4M3 scale (448) and no block scale saturates.
//
// Two launches on the caller's stream: a grid-stride max of BF16 magnitudes
// (bit patterns compared as integers; Inf and NaN ignored) accumulated by
// atomicMax into the two output words, then one thread turning each maximum
// into g in place (IEEE division; 1.0 when the maximum is 0).
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4kv {

namespace {

constexpr float kRange = 6.0f * 448.0f;  // largest E2M1 magnitude x largest E4M3 scale

// Largest finite BF16 magnitude among the 8 values of w (as bits, 0 if none).
__device__ __forceinline__ uint32_t amax8(uint4 w) {
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint32_t lo = x[i] & 0x7fffu, hi = (x[i] >> 16) & 0x7fffu;
        lo = lo >= 0x7f80u ? 0u : lo;  // Inf / NaN
        hi = hi >= 0x7f80u ? 0u : hi;
        m = max(m, max(lo, hi));
    }
    return m;
}

// Eight CTAs per SM (32 registers): the grid below is one wave of resident CTAs.
__global__ void __launch_bounds__(256, 8) amax_kernel(const uint4 *k, const uint4 *v, int64_t num_tokens,
                                                   int64_t stride16, int row16, unsigned *out) {
    pdl_launch_dependents();
    const int64_t n = num_tokens * row16;
    // flat index i = t * row16 + j over the 16-byte vectors; (t, j) advance by
    // a fixed step without divisions, four vectors of K and of V in flight
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    const int64_t step_t = step / row16;
    const int step_j = (int)(step - step_t * row16);
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t t = i / row16;
    int j = (int)(i - t * row16);
    uint32_t mk = 0, mv = 0;
    auto advance = [&]() {
        i += step;
        t += step_t;
        j += step_j;
        if (j >= row16) {
            j -= row16;
            t++;
        }
    };
    while (i + 3 * step < n) {
        uint4 xk[4], xv[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            xk[u] = __ldg(k + t * stride16 + j);
            xv[u] = __ldg(v + t * stride16 + j);
            advance();
        }
#pragma unroll
        for (int u = 0; u < 4; u++) {
            mk = max(mk, amax8(xk[u]));
            mv = max(mv, amax8(xv[u]));
        }
    }
    for (; i < n; advance()) {
        mk = max(mk, amax8(__ldg(k + t * stride16 + j)));
        mv = max(mv, amax8(__ldg(v + t * stride16 + j)));
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) {
        mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, s));
        mv = max(mv, __shfl_xor_sync(0xffffffffu, mv, s));
    }
    if ((threadIdx.x & 31) == 0) {
        if (mk) atomicMax(out, mk);
        if (mv) atomicMax(out + 1, mv);
    }
}

__global__ void finalize_kernel(unsigned *words) {
    pdl_wait();
#pragma unroll
    for (int i = 0; i < 2; i++) {
        const float amax = __uint_as_float(words[i] << 16);  // BF16 bits -> float
        const float g = amax > 0.f ? __fdiv_rn(amax, kRange) : 1.0f;
        words[i] = __float_as_uint(g);
    }
}

constexpr int kMaxDevices = 64;
std::mutex g_wave_mu;
int64_t g_wave[kMaxDevices];  // resident amax CTAs per device (SMs x CTAs per SM), 0 until known

// One wave of resident amax CTAs, so that the grid-stride loop has no tail
// wave; looked up once per device (the occupancy query costs host time).
cudaError_t amax_wave(int64_t *wave) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_wave_mu);
    if (!g_wave[dev]) {
        int sms = 0, per_sm = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, amax_kernel, 256, 0)) != cudaSuccess) return e;
        g_wave[dev] = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    }
    *wave = g_wave[dev];
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_calibrate(const void *k, const void *v, int64_t num_tokens, int num_kv_heads, int64_t token_stride,
                             float *scales, cudaStream_t stream) {
    unsigned *words = reinterpret_cast<unsigned *>(scales);
    cudaError_t e = cudaMemsetAsync(words, 0, 2 * sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
    const int row16 = num_kv_heads * (kHeadDim / 8);
    const int64_t n = num_tokens * row16;
    int64_t wave = 0;
    if ((e = amax_wave(&wave)) != cudaSuccess) return e;
    const int64_t want = ceil_div64(n, 256);
    const unsigned grid = (unsigned)(want < wave ? (want > 0 ? want : 1) : wave);
    amax_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), num_tokens,
                                          token_stride / 8, row16, words);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    void *args[] = {&words};
    return launch_pdl(reinterpret_cast<const void *>(&finalize_kernel), 1, 1, 0, stream, args);
}

}  // namespace nvfp4kv
