// FP32 peak probe: the denominator of the compositing kernel's roofline.
//
// The compositing step (section "La règle de composition alpha") is bound by
// FP32 issue, not by memory, so its roofline is the rate of fused multiply-adds
// the SMs sustain. This kernel measures that rate on the device at hand: every
// thread runs kChains independent FMA chains (enough independent work per warp
// to hide the pipe latency), `iterations` steps each, written as inline PTX so
// that each step is exactly one fma.rn.f32 per chain, or one fma.rn.f32x2 per
// pair of chains (packed form). Values stay bounded (a * 0.99999988 + 1e-7
// moves towards a fixed point), and the chains' sum is stored only under a
// condition that the seed makes false, so no chain can be dropped.
#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kPeakThreads = 256;
constexpr int kChains = 16;

__global__ void __launch_bounds__(kPeakThreads) ffma_peak_kernel(int iterations, float seed, float* sink) {
    grid_dependency_begin();
    float a[kChains];
#pragma unroll
    for (int i = 0; i < kChains; i++) a[i] = seed + 1e-3f * (float)(threadIdx.x + i);
    const float b = 0.99999988f, c = 1e-7f;
    for (int it = 0; it < iterations; it++) {
#pragma unroll
        for (int i = 0; i < kChains; i++) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a[i]) : "f"(b), "f"(c));
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChains; i++) s += a[i];
    if (s == seed) sink[blockIdx.x * kPeakThreads + threadIdx.x] = s;
}

__global__ void __launch_bounds__(kPeakThreads) ffma2_peak_kernel(int iterations, float seed, float* sink) {
    grid_dependency_begin();
    unsigned long long a[kChains / 2];
#pragma unroll
    for (int i = 0; i < kChains / 2; i++) {
        const float lo = seed + 1e-3f * (float)(threadIdx.x + 2 * i), hi = lo + 1e-3f;
        asm("mov.b64 %0, {%1, %2};" : "=l"(a[i]) : "f"(lo), "f"(hi));
    }
    unsigned long long b, c;
    {
        const float bb = 0.99999988f, cc = 1e-7f;
        asm("mov.b64 %0, {%1, %1};" : "=l"(b) : "f"(bb));
        asm("mov.b64 %0, {%1, %1};" : "=l"(c) : "f"(cc));
    }
    for (int it = 0; it < iterations; it++) {
#pragma unroll
        for (int i = 0; i < kChains / 2; i++) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(a[i]) : "l"(b), "l"(c));
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChains / 2; i++) {
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a[i]));
        s += lo + hi;
    }
    if (s == seed) sink[blockIdx.x * kPeakThreads + threadIdx.x] = s;
}

}  // namespace
}  // namespace gs

using namespace gs;

extern "C" gs_status gs_fp32_peak_probe(int32_t blocks, int32_t iterations, int32_t packed, float* sink,
                                        int64_t* fma_count, void* stream) {
    if (blocks < 1 || blocks > (1 << 20) || iterations < 1 || !sink) return GS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    // seed -1: the sum of 16 chains that start near -1 and move slowly towards +0.83 stays far
    // from -1 for any run length a caller can time, so nothing is stored
    if (packed)
        launch_k(ffma2_peak_kernel, blocks, kPeakThreads, 0, s, iterations, -1.0f, sink);
    else
        launch_k(ffma_peak_kernel, blocks, kPeakThreads, 0, s, iterations, -1.0f, sink);
    if (fma_count) *fma_count = (int64_t)blocks * kPeakThreads * (int64_t)iterations * kChains;
    return cudaGetLastError() == cudaSuccess ? GS_OK : GS_ERR_CUDA;
}
