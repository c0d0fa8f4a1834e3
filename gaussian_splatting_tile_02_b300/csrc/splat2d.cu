// 2D splats on the tile pipeline: the lesson page "3D Gaussian Splatting à
// partir de zéro", section "Étape 2" (rasterise_2d: Gaussians given directly by
// an image-space mean, a 2x2 covariance, a colour, an opacity in [0, 1] and a
// per-Gaussian scalar that only orders them; alpha = o exp(-0.5 d^T cov^-1 d)
// clamped at 0.99 on the integer pixel grid, composited front to back in
// increasing order of that scalar) and "Étape 3" (the trainable 2D scene).
//
// preprocess2d_kernel writes the same per-Gaussian record the projection step
// writes for 3D Gaussians, so binning, the sorts, the ranges and compositing
// (and the compositing backward) are the 3D path's kernels unchanged. Two
// differences from the 3D projection:
//  - the ordering scalar is any real number, so the record's depth field
//    holds an order-preserving 32-bit key (sign bit flipped for positive
//    values, all bits for negative ones) instead of the float's own bits;
//  - the tile rectangle comes from this fixed binary32 program (each product,
//    sum and square root rounded on its own, no FMA):
//      b = 0.5 (cov01 + cov10); det = a c - b b, culled unless 0 < det <= FLT_MAX
//      lam = 0.5 (a + c) + sqrt((0.5 (a - c))^2 + b^2); r = ceil(3 sqrt(lam))
//      culled unless u, v, r are finite and o > 0
//      x0 = max(ceil(u - r), 0), x1 = min(floor(u + r), W - 1), same for y;
//      tiles [x0>>4 .. x1>>4] x [y0>>4 .. y1>>4] if x0 <= x1 and y0 <= y1.
// The cut-offs of the tile renderer apply as in 3D: each Gaussian covers the
// tiles of its 3-sigma rectangle, alpha < 1/255 is skipped and a pixel stops
// once T < 1e-4.
#include <cuda_fp16.h>
#include <float.h>

#include "gs_internal.cuh"

namespace gs {
namespace {

__device__ __forceinline__ float mul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float add(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float sub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float sq(float a) { return __fsqrt_rn(a); }

// order-preserving map of a float to uint32 (NaN excluded by the caller)
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Pre2dArgs {
    const float2* means;
    const float* covs;        // [n][2][2]
    const float* colours;     // [n][3]
    const float* opacities;   // [n]
    const float* depths;      // [n]
    int64_t n;
    int width, height;
    float* depth_key;         // [n] the order key's bits
    uint32_t* tiles_touched;
    ushort4* rect;
    float4* raster;           // [n][3]
};

__global__ void __launch_bounds__(256) preprocess2d_kernel(const Pre2dArgs a) {
    grid_dependency_begin();
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= a.n) return;
    const float2 m = a.means[g];
    const float ca = a.covs[4 * g], c01 = a.covs[4 * g + 1], c10 = a.covs[4 * g + 2], cc = a.covs[4 * g + 3];
    const float cb = mul(0.5f, add(c01, c10));
    const float o = a.opacities[g];
    const float dz = a.depths[g];
    const float det = sub(mul(ca, cc), mul(cb, cb));
    const float hm = mul(0.5f, sub(ca, cc));
    const float lam = add(mul(0.5f, add(ca, cc)), sq(add(mul(hm, hm), mul(cb, cb))));
    const float rf = ceilf(mul(3.0f, sq(lam)));
    const float u = m.x, v = m.y;
    a.depth_key[g] = __uint_as_float(order_key(dz));
    if (!(det > 0.0f && det <= FLT_MAX) || !(fabsf(u) <= FLT_MAX && fabsf(v) <= FLT_MAX && rf <= FLT_MAX) ||
        !(o > 0.0f) || dz != dz) {
        a.tiles_touched[g] = 0;
        a.rect[g] = make_ushort4(0, 0, 0, 0);
        return;
    }
    float x0 = ceilf(sub(u, rf)), x1 = floorf(add(u, rf));
    float y0 = ceilf(sub(v, rf)), y1 = floorf(add(v, rf));
    x0 = x0 > 0.0f ? x0 : 0.0f;
    y0 = y0 > 0.0f ? y0 : 0.0f;
    const float wm1 = (float)(a.width - 1), hm1 = (float)(a.height - 1);
    x1 = x1 < wm1 ? x1 : wm1;
    y1 = y1 < hm1 ? y1 : hm1;
    uint32_t touched = 0;
    ushort4 rect = make_ushort4(0, 0, 0, 0);
    if (x0 <= x1 && y0 <= y1) {
        const int tx0 = (int)x0 >> 4, tx1 = (int)x1 >> 4, ty0 = (int)y0 >> 4, ty1 = (int)y1 >> 4;
        touched = (uint32_t)((tx1 - tx0 + 1) * (ty1 - ty0 + 1));
        rect = make_ushort4((unsigned short)tx0, (unsigned short)ty0, (unsigned short)tx1, (unsigned short)ty1);
    }
    a.tiles_touched[g] = touched;
    a.rect[g] = rect;
    if (!touched) return;
    // the compositor's record, as the 3D projection writes it: centre (exact
    // here, residual 0), log2(alpha) = log2 o - (k1 dx)^2 - (k2 dy + k3 dx)^2,
    // colour and the alpha >= 1/255 box
    const float sc = 0.84932180028801907f;   // sqrt(log2(e) / 2)
    const float ra = rsqrtf(ca);
    const float k1 = sc * ra;
    const float k2 = sc * sqrtf(ca / det);
    const float k3 = -sc * cb * ra * rsqrtf(det);
    const float oc = o < 1.0f ? o : 1.0f;
    const float tau = 2.0f * logf(255.0f * oc) + 0.02f;
    float hx = INFINITY, hy = INFINITY;
    if (!(tau > 0.0f)) {
        hx = hy = -1.0f;
    } else if ((ca + cc) * (ca + cc) <= 1e8f * det) {
        hx = 1.01f * sqrtf(tau * ca) + 0.05f;
        hy = 1.01f * sqrtf(tau * cc) + 0.05f;
    }
    const __half2 h = __halves2half2(__float2half_ru(hx), __float2half_ru(hy));
    float4* rec = a.raster + 3 * g;
    rec[0] = make_float4(u, v, 0.0f, 0.0f);
    rec[1] = make_float4(k1, k2, k3, log2f(oc));
    rec[2] = make_float4(a.colours[3 * g], a.colours[3 * g + 1], a.colours[3 * g + 2],
                         __uint_as_float(*reinterpret_cast<const uint32_t*>(&h)));
}

// dL/dconic (A, B, C) -> dL/dcov as a full 2x2 matrix, cov = conic^-1:
// dL/dcov = -Q G Q with Q = conic and G = [[gA, gB/2], [gB/2, gC]]; the
// off-diagonal gradient is split evenly over cov01 and cov10.
__global__ void __launch_bounds__(256) conic_to_cov_grad_kernel(const float* __restrict__ covs,
                                                                const uint32_t* __restrict__ tiles_touched,
                                                                const float* __restrict__ g_conic, int64_t n,
                                                                float* __restrict__ g_covs) {
    grid_dependency_begin();
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n) return;
    float* out = g_covs + 4 * g;
    if (tiles_touched[g] == 0) {
        out[0] = out[1] = out[2] = out[3] = 0.0f;
        return;
    }
    const float a = covs[4 * g], b = 0.5f * (covs[4 * g + 1] + covs[4 * g + 2]), c = covs[4 * g + 3];
    const float idet = 1.0f / (a * c - b * b);
    const float A = c * idet, B = -b * idet, C = a * idet;
    const float gA = g_conic[3 * g], gB = 0.5f * g_conic[3 * g + 1], gC = g_conic[3 * g + 2];
    const float QG00 = A * gA + B * gB, QG01 = A * gB + B * gC, QG10 = B * gA + C * gB, QG11 = B * gB + C * gC;
    const float Ga = -(QG00 * A + QG01 * B);
    const float Gb = -(QG00 * B + QG01 * C);
    const float Gc = -(QG10 * B + QG11 * C);
    out[0] = Ga;
    out[1] = Gb;
    out[2] = Gb;
    out[3] = Gc;
}

}  // namespace

cudaError_t launch_preprocess2d(const float* means, const float* covs, const float* colours, const float* opacities,
                                const float* depths, int64_t n, int width, int height, const gs_projected& p,
                                cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    Pre2dArgs a;
    a.means = reinterpret_cast<const float2*>(means);
    a.covs = covs;
    a.colours = colours;
    a.opacities = opacities;
    a.depths = depths;
    a.n = n;
    a.width = width;
    a.height = height;
    a.depth_key = p.depth;
    a.tiles_touched = p.tiles_touched;
    a.rect = reinterpret_cast<ushort4*>(p.rect);
    a.raster = reinterpret_cast<float4*>(p.raster);
    launch_k(preprocess2d_kernel, (unsigned)((n + 255) / 256), 256, 0, s, a);
    return cudaGetLastError();
}

cudaError_t launch_conic_to_cov_grad(const float* covs, const uint32_t* tiles_touched, const float* g_conic,
                                     int64_t n, float* g_covs, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    launch_k(conic_to_cov_grad_kernel, (unsigned)((n + 255) / 256), 256, 0, s, covs, tiles_touched, g_conic, n, g_covs);
    return cudaGetLastError();
}

GS_DEFINE_CHECK_SETTER(splat2d)

}  // namespace gs
