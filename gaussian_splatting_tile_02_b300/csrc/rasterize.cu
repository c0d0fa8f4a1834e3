// Step 5 of the forward renderer: front-to-back compositing per 16x16 tile.
//
// Method: lesson page "3D Gaussian Splatting à partir de zéro", section "La
// règle de composition alpha" (C = sum alpha_i T_i c_i, T_i = prod_{j<i}
// (1 - alpha_j), alpha_i = o_i exp(-0.5 d^T Sigma'^-1 d)) and "Étape 2"
// (rasterise_2d: integer pixel grid, alpha clamped at 0.99, front-to-back
// loop over the depth order). Contributions with alpha < 1/255 are skipped
// and a pixel stops once T < 1e-4, after the Gaussian that took it there.
//
// One block per tile, one thread per pixel; warp w covers the 8x4 pixel block
// (8 (w & 1), 4 (w >> 1)) of the tile. The tile's sorted list is walked in
// batches of 256 entries. Staging: each thread gathers one projected record
// into shared memory with the exponent's constants folded in
// (alpha = 2^(log2 o + quadratic form)) and the box that holds the region where
// alpha can reach 1/255 (o exp(-q/2) >= 1/255, i.e. q <= 2 ln(255 o), widened
// by a safety margin). Each warp then ballots which of the 256 entries' boxes
// meet its 8x4 block and evaluates only those, in list order, for its 32
// pixels: an entry whose box misses the block cannot contribute to any of its
// pixels, so skipping it changes no result. The block leaves the list as soon
// as all its pixels are done (__syncthreads_count). Per evaluated (pixel,
// entry): two subtractions, the quadratic form (5 FP32 ops), ex2 on the MUFU
// pipe, a min and a compare, plus the blend for contributing pairs.
#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kRastThreads = kTile * kTile;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kAlphaMin = 1.0f / 255.0f;

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
    __shared__ float4 s_q[kRastThreads];    // (mx, my, qa, qb)
    __shared__ float4 s_r[kRastThreads];    // (qc, log2 o, r, g)
    __shared__ float s_b[kRastThreads];     // b
    __shared__ float4 s_box[kRastThreads];  // (x lo, x hi, y lo, y hi) of the alpha >= 1/255 region

    const int tile = blockIdx.x;
    const int tx = tile % a.tiles_x, ty = tile / a.tiles_x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx0 = tx * kTile + 8 * (warp & 1), by0 = ty * kTile + 4 * (warp >> 1);
    const int px = bx0 + (lane & 7), py = by0 + (lane >> 3);
    const float fbx0 = (float)bx0, fbx1 = (float)(bx0 + 7), fby0 = (float)by0, fby1 = (float)(by0 + 3);
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
            s_q[threadIdx.x] = make_float4(m.x, m.y, -0.5f * kLog2e * co.x, -kLog2e * co.y);
            s_r[threadIdx.x] = make_float4(-0.5f * kLog2e * co.z, fast_log2(co.w), __ldg(a.rgb + 3 * g),
                                           __ldg(a.rgb + 3 * g + 1));
            s_b[threadIdx.x] = __ldg(a.rgb + 3 * g + 2);
            // box of {d : d^T conic d <= tau}, tau = 2 ln(255 o): half-extents
            // sqrt(tau Sigma'_xx) and sqrt(tau Sigma'_yy) with Sigma' = conic^-1;
            // tau is raised by 0.02 and the half-extents widened by 1% + 0.05 px,
            // far more than the rounding of the per-pixel alpha can move it.
            // The rounding of det(conic) is about 3e-8 (A + C)^2 / det relative:
            // conics with (A + C)^2 > 1e4 det keep an unbounded box (never culled).
            const float detc = co.x * co.z - co.y * co.y;
            const float tau = 2.0f * __logf(255.0f * co.w) + 0.02f;
            float4 box = make_float4(-INFINITY, INFINITY, -INFINITY, INFINITY);
            if (!(tau > 0.0f)) {  // o below 1/255 (margin included): never contributes
                box = make_float4(INFINITY, -INFINITY, INFINITY, -INFINITY);
            } else if (detc > 0.0f && (co.x + co.z) * (co.x + co.z) <= 1e4f * detc) {
                const float hx = 1.01f * sqrtf(tau * co.z / detc) + 0.05f;
                const float hy = 1.01f * sqrtf(tau * co.x / detc) + 0.05f;
                if (hx < INFINITY && hy < INFINITY) box = make_float4(m.x - hx, m.x + hx, m.y - hy, m.y + hy);
            }
            s_box[threadIdx.x] = box;
        }
        __syncthreads();
        const uint32_t cnt = min((uint32_t)kRastThreads, range.y - base);
        // which of the batch entries can touch this warp's 8x4 pixel block
        uint32_t mask[kRastThreads / 32];
#pragma unroll
        for (int i = 0; i < kRastThreads / 32; i++) {
            const uint32_t j = (uint32_t)(i * 32 + lane);
            bool hit = false;
            if (j < cnt) {
                const float4 bx = s_box[j];
                hit = bx.x <= fbx1 && bx.y >= fbx0 && bx.z <= fby1 && bx.w >= fby0;
            }
            mask[i] = __ballot_sync(0xffffffffu, hit);
        }
#pragma unroll
        for (int i = 0; i < kRastThreads / 32; i++) {
            if (__all_sync(0xffffffffu, done)) break;
            uint32_t m = mask[i];
            while (m) {
                const int j = i * 32 + __ffs(m) - 1;
                m &= m - 1;
                if (done) continue;
                const float4 q = s_q[j];
                const float4 r = s_r[j];
                const float dx = q.x - fpx, dy = q.y - fpy;
                const float e = r.y + dx * (q.z * dx + q.w * dy) + r.x * dy * dy;
                const float alpha = fminf(0.99f, fast_exp2(e));
                if (alpha < kAlphaMin) continue;
                const float w = alpha * T;
                C0 += w * r.z;
                C1 += w * r.w;
                C2 += w * s_b[j];
                T -= w;
                last = base - range.x + (uint32_t)j + 1;
                if (T < 1e-4f) done = true;
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
