// Step 5 of the forward renderer: front-to-back compositing per 16x16 tile.
//
// Method: lesson page "3D Gaussian Splatting à partir de zéro", section "La
// règle de composition alpha" (C = sum alpha_i T_i c_i, T_i = prod_{j<i}
// (1 - alpha_j), alpha_i = o_i exp(-0.5 d^T Sigma'^-1 d)) and "Étape 2"
// (rasterise_2d: integer pixel grid, alpha clamped at 0.99, front-to-back
// loop over the depth order). Contributions with alpha < 1/255 are skipped
// and a pixel stops once T < 1e-4, after the Gaussian that took it there.
//
// One block per tile, one thread per pixel. The tile's sorted Gaussian list
// is walked in batches of 256: each thread gathers one projected record
// (centre, conic with the exponent's constants folded in, opacity, colour)
// into shared memory, then every thread evaluates the batch for its pixel.
// The block leaves the loop as soon as all its pixels are done
// (__syncthreads_count). The work is FP32-issue bound: per (pixel, Gaussian)
// two subtractions, the quadratic form, an ex2 on the MUFU pipe, a min and a
// compare, plus the blend for contributing pairs.
#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kRastThreads = kTile * kTile;
constexpr float kLog2e = 1.4426950408889634f;

// 2^x on the MUFU pipe (PTX ex2.approx; relative error about 2^-22).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// log2(x) on the MUFU pipe (PTX lg2.approx).
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct RastArgs {
    const float2* mean2d;
    const float4* conic_opacity;
    const float* rgb;
    const uint32_t* sorted_vals;
    const uint2* ranges;
    uint32_t n;
    int width, height, tiles_x;
    float bg0, bg1, bg2;
    float* image;
    float* final_T;
    uint32_t* n_contrib;
};

__global__ void __launch_bounds__(kRastThreads) rasterize_kernel(const RastArgs a) {
    __shared__ float4 s_q[kRastThreads];   // (mx, my, qa, qb)
    __shared__ float4 s_r[kRastThreads];   // (qc, log2 o, r, g)
    __shared__ float s_b[kRastThreads];    // b

    const int tile = blockIdx.x;
    const int tx = tile % a.tiles_x, ty = tile / a.tiles_x;
    const int px = tx * kTile + (threadIdx.x & (kTile - 1));
    const int py = ty * kTile + (threadIdx.x >> 4);
    const bool inside = px < a.width && py < a.height;
    const uint2 range = a.ranges[tile];
    const float fpx = (float)px, fpy = (float)py;

    float T = 1.0f, C0 = 0.0f, C1 = 0.0f, C2 = 0.0f;
    uint32_t last = 0;
    bool done = !inside;

    for (uint32_t base = range.x; base < range.y; base += kRastThreads) {
        if (__syncthreads_count(done) == kRastThreads) break;
        const uint32_t idx = base + threadIdx.x;
        if (idx < range.y) {
            uint32_t g = __ldg(a.sorted_vals + idx);
            // an index outside the scene can only come from a sort that was cut
            // short (its status is flagged); never read past the arrays
            if (g >= a.n) g = 0;
            const float2 m = __ldg(a.mean2d + g);
            const float4 co = __ldg(a.conic_opacity + g);
            // exponent in base 2: log2(alpha) = log2 o - (log2 e / 2)(A dx^2 + C dy^2) - log2 e B dx dy
            s_q[threadIdx.x] = make_float4(m.x, m.y, -0.5f * kLog2e * co.x, -kLog2e * co.y);
            s_r[threadIdx.x] = make_float4(-0.5f * kLog2e * co.z, fast_log2(co.w), __ldg(a.rgb + 3 * g),
                                           __ldg(a.rgb + 3 * g + 1));
            s_b[threadIdx.x] = __ldg(a.rgb + 3 * g + 2);
        }
        __syncthreads();
        const int cnt = (int)min((uint32_t)kRastThreads, range.y - base);
        if (!done) {
            for (int j = 0; j < cnt; j++) {
                const float4 q = s_q[j];
                const float4 r = s_r[j];
                const float dx = q.x - fpx, dy = q.y - fpy;
                const float e = r.y + dx * (q.z * dx + q.w * dy) + r.x * dy * dy;
                const float alpha = fminf(0.99f, fast_exp2(e));
                if (alpha < (1.0f / 255.0f)) continue;
                const float w = alpha * T;
                C0 += w * r.z;
                C1 += w * r.w;
                C2 += w * s_b[j];
                T -= w;
                last = base - range.x + j + 1;
                if (T < 1e-4f) {
                    done = true;
                    break;
                }
            }
        }
    }
    if (inside) {
        const int64_t p = (int64_t)py * a.width + px;
        a.image[3 * p] = C0 + T * a.bg0;
        a.image[3 * p + 1] = C1 + T * a.bg1;
        a.image[3 * p + 2] = C2 + T * a.bg2;
        if (a.final_T) a.final_T[p] = T;
        if (a.n_contrib) a.n_contrib[p] = last;
    }
}

}  // namespace

cudaError_t launch_rasterize(const gs_projected& p, int64_t n, const uint32_t* sorted_vals, const uint32_t* ranges,
                             const CamConst& cam, float* image, float* final_T, uint32_t* n_contrib,
                             cudaStream_t s) {
    RastArgs a;
    a.mean2d = reinterpret_cast<const float2*>(p.mean2d);
    a.conic_opacity = reinterpret_cast<const float4*>(p.conic_opacity);
    a.rgb = p.rgb;
    a.sorted_vals = sorted_vals;
    a.ranges = reinterpret_cast<const uint2*>(ranges);
    a.n = (uint32_t)n;
    a.width = cam.width;
    a.height = cam.height;
    a.tiles_x = cam.tiles_x;
    a.bg0 = cam.bg[0];
    a.bg1 = cam.bg[1];
    a.bg2 = cam.bg[2];
    a.image = image;
    a.final_T = final_T;
    a.n_contrib = n_contrib;
    const unsigned tiles = (unsigned)(cam.tiles_x * cam.tiles_y);
    if (n == 0) a.sorted_vals = nullptr;
    rasterize_kernel<<<tiles, kRastThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gs
