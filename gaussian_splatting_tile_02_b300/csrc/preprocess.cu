// Step 1 of the forward renderer: per-Gaussian projection.
//
// Method: lesson page "3D Gaussian Splatting à partir de zéro", sections
// "Ce qu'un Gaussien porte" (Sigma = R S S^T R^T, scale = exp(log-scale),
// opacity = sigmoid), "L'étape de projection" (mu' = project(mu),
// Sigma' = J W Sigma W^T J^T), "Étape 5" (quaternion rotation, camera-space
// depth) and "Étape 6" (SH colour along the view direction).
//
// One thread per Gaussian; the kernel is bound by the HBM stream of the
// parameters (236 B per Gaussian at SH degree 3) and its outputs.
//
// The integer results (culling, depth bits, radius, pixel and tile rectangles)
// are computed by a fixed binary32 program: every product, quotient, sum and
// square root is a separately rounded __f*_rn intrinsic (never contracted into
// an FMA), in this order:
//   p_i  = ((R_i0 m0 + R_i1 m1) + R_i2 m2) + t_i ;  z = p_2 ;  cull unless z > near
//   n2   = ((qw^2 + qx^2) + qy^2) + qz^2 ; cull unless 0 < n2 <= FLT_MAX ;
//          (w, x, y, z) = q / sqrt(n2)
//   G    = rotation of (w, x, y, z): G00 = 1 - 2(yy + zz), G01 = 2(xy - wz),
//          G02 = 2(xz + wy), G10 = 2(xy + wz), G11 = 1 - 2(xx + zz),
//          G12 = 2(yz - wx), G20 = 2(xz - wy), G21 = 2(yz + wx), G22 = 1 - 2(xx + yy)
//   s_k  = exp32(log_scale_k)   (binary32 exp below)
//   B_ij = ((R_i0 G_0j + R_i1 G_1j) + R_i2 G_2j) s_j          (B = W R S)
//   j00  = fx / z, j11 = fy / z, j02 = -((fx p0) / (z z)), j12 = -((fy p1) / (z z))
//   M_0k = j00 B_0k + j02 B_2k,  M_1k = j11 B_1k + j12 B_2k   (M = J W R S)
//   a = (M00^2 + M01^2) + M02^2,  b = (M00 M10 + M01 M11) + M02 M12,
//   c = (M10^2 + M11^2) + M12^2                               (Sigma' = M M^T)
//   det = a c - b b ; cull unless 0 < det <= FLT_MAX
//   lam = 0.5 (a + c) + sqrt((0.5 (a - c))^2 + b^2) ; r = ceil(3 sqrt(lam))
//   u = (fx p0) / z + cx,  v = (fy p1) / z + cy ; cull unless u, v, r finite
//   x0 = max(ceil(u - r), 0), x1 = min(floor(u + r), W - 1), same for y;
//   tiles [x0>>4 .. x1>>4] x [y0>>4 .. y1>>4] if x0 <= x1 and y0 <= y1.
// Sigma' = M M^T is the pages' J W Sigma W^T J^T with Sigma = (R S)(R S)^T.
// The continuous outputs (conic, opacity, colour) use ordinary fp32 arithmetic.
#include <cuda_fp16.h>
#include <float.h>

#include <map>
#include <utility>
#include <mutex>

#include "gs_internal.cuh"

namespace gs {
namespace {

__device__ __forceinline__ float mul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float add(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float sub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float dv(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ float sq(float a) { return __fsqrt_rn(a); }

// Scale activation e^l in binary32 with a fixed operation sequence (so the
// result is reproducible bit for bit): Cody and Waite's range reduction
// (Software Manual for the Elementary Functions, 1980), l = k ln2 + r with ln2
// split into the 12-bit head 2839/4096 (k * head is exact) and a rounded tail,
// then the degree-7 Taylor polynomial of e^r (|r| <= ln2/2) in Horner form,
// then the exact product with 2^k. l is clamped to [-80, 80] so that 2^k and
// the result are normal numbers. Constants: ln 2 and 1/j! rounded to binary32.
__device__ __forceinline__ float exp32(float x) {
    if (x != x) return x;
    x = x > 80.0f ? 80.0f : x;
    x = x < -80.0f ? -80.0f : x;
    const float k = rintf(mul(x, 0x1.715476p+0f));                       // x / ln2
    const float r = sub(sub(x, mul(k, 0x1.62ep-1f)), mul(k, 0x1.0bfbe8p-15f));
    float p = 0x1.a01a02p-13f;                                           // 1/7!
    p = add(0x1.6c16c2p-10f, mul(r, p));                                 // 1/6!
    p = add(0x1.111112p-7f, mul(r, p));                                  // 1/5!
    p = add(0x1.555556p-5f, mul(r, p));                                  // 1/4!
    p = add(0x1.555556p-3f, mul(r, p));                                  // 1/3!
    p = add(0.5f, mul(r, p));
    p = add(1.0f, mul(r, p));
    p = add(1.0f, mul(r, p));
    return mul(p, __int_as_float((127 + (int)k) << 23));
}

// Error-free transformations of binary32 arithmetic (Dekker's product via
// FMA, Knuth's two-sum): a*b = p + e and a+b = s + e exactly.
__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
    p = __fmul_rn(a, b);
    e = fmaf(a, b, -p);
}
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Camera-space point and projected centre carried as unevaluated sums
// hi + lo of two floats (compensated dot product in the manner of Ogita, Rump
// and Oishi, "Accurate sum and dot product", 2005), good to ~1e-13 relative:
// the projected centre is then known to ~1e-9 px where the binary32 decision
// value u carries up to ~1e-4 px of rounding at u ~ 1000.
__device__ __forceinline__ void dot3_add(const float* r, float m0, float m1, float m2, float t, float& hi,
                                         float& lo) {
    float p, s, h, e, q;
    two_prod(r[0], m0, p, s);
    two_prod(r[1], m1, h, e);
    two_sum(p, h, p, q);
    s += q + e;
    two_prod(r[2], m2, h, e);
    two_sum(p, h, p, q);
    s += q + e;
    two_sum(p, t, p, q);
    s += q;
    hi = p;
    lo = s;
}
// f * (xh + xl) / (zh + zl) + c, returned as hi + lo
__device__ __forceinline__ void project_df(float f, float xh, float xl, float zh, float zl, float c, float& hi,
                                          float& lo) {
    const float q1 = xh / zh;
    float ph, pl;
    two_prod(q1, zh, ph, pl);
    const float rr = ((xh - ph) - pl) + xl - q1 * zl;
    const float q2 = rr / zh;
    float h, l, s, e;
    two_prod(f, q1, h, l);
    l = fmaf(f, q2, l);
    two_sum(h, c, s, e);
    hi = s;
    lo = e + l;
}

// Real SH basis constants, from their closed forms: sqrt(1/4pi), sqrt(3/4pi),
// sqrt(15/4pi), sqrt(5/16pi), sqrt(15/16pi), sqrt(35/32pi), sqrt(105/4pi),
// sqrt(21/32pi), sqrt(7/16pi), sqrt(105/16pi).
constexpr float kY0 = 0.28209479177387814f;
constexpr float kY1 = 0.48860251190291992f;
constexpr float kY2a = 1.0925484305920792f;
constexpr float kY2b = 0.31539156525252005f;
constexpr float kY2c = 0.54627421529603959f;
constexpr float kY3a = 0.59004358992664352f;
constexpr float kY3b = 2.8906114426405538f;
constexpr float kY3c = 0.45704579946446572f;
constexpr float kY3d = 0.3731763325901154f;
constexpr float kY3e = 1.4453057213202769f;

// Colour along unit direction (x, y, z): sum_k Y_k c_k + 0.5, clamped at 0.
// Signs follow the printed code of "Étape 6" for bands 0..2 (band 1: -y, +z,
// -x; band 2 all +); band 3 (not printed) uses the band-1 pattern, odd m
// negative.
template <int D>
__device__ __forceinline__ float3 eval_sh(const float* co, float x, float y, float z) {
    constexpr int NK = (D + 1) * (D + 1);
    float Y[NK];
    Y[0] = kY0;
    if constexpr (D >= 1) {
        Y[1] = -kY1 * y;
        Y[2] = kY1 * z;
        Y[3] = -kY1 * x;
    }
    if constexpr (D >= 2) {
        const float xx = x * x, yy = y * y, zz = z * z;
        Y[4] = kY2a * x * y;
        Y[5] = kY2a * y * z;
        Y[6] = kY2b * (2.0f * zz - xx - yy);
        Y[7] = kY2a * x * z;
        Y[8] = kY2c * (xx - yy);
        if constexpr (D >= 3) {
            Y[9] = -kY3a * y * (3.0f * xx - yy);
            Y[10] = kY3b * x * y * z;
            Y[11] = -kY3c * y * (4.0f * zz - xx - yy);
            Y[12] = kY3d * z * (2.0f * zz - 3.0f * xx - 3.0f * yy);
            Y[13] = -kY3c * x * (4.0f * zz - xx - yy);
            Y[14] = kY3e * z * (xx - yy);
            Y[15] = -kY3a * x * (xx - 3.0f * yy);
        }
    }
    float r = 0.5f, g = 0.5f, b = 0.5f;
#pragma unroll
    for (int k = 0; k < NK; k++) {
        r = fmaf(Y[k], co[3 * k], r);
        g = fmaf(Y[k], co[3 * k + 1], g);
        b = fmaf(Y[k], co[3 * k + 2], b);
    }
    return make_float3(fmaxf(r, 0.0f), fmaxf(g, 0.0f), fmaxf(b, 0.0f));
}

// The (D + 1)^2 x 3 SH coefficients of one Gaussian into registers, from
// global memory (read-only path) or from a shared-memory stage; rows of
// 12 or 48 floats (D = 1, 3) as float4 loads.
template <int D, bool kShared>
__device__ __forceinline__ void load_sh(const float* __restrict__ c, float* co) {
    constexpr int NK3 = (D + 1) * (D + 1) * 3;
    if constexpr (D == 3 || D == 1) {
        const float4* c4 = reinterpret_cast<const float4*>(c);
#pragma unroll
        for (int i = 0; i < NK3 / 4; i++) {
            const float4 q = kShared ? c4[i] : __ldg(c4 + i);
            co[4 * i] = q.x; co[4 * i + 1] = q.y; co[4 * i + 2] = q.z; co[4 * i + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < NK3; i++) co[i] = kShared ? c[i] : __ldg(c + i);
    }
}

struct PreArgs {
    const float* means;
    const float4* quats;
    const float* log_scales;
    const float* logits;
    const float* sh;
    int64_t n;
    CamConst cam;
    float2* mean2d;
    float4* raster;
    float4* conic_opacity;
    float* rgb;
    float* depth;
    int32_t* radius;
    uint32_t* tiles_touched;
    ushort4* rect;
    // depth-order sort input, nullable: key = depth bits for Gaussians with
    // tiles (depth > near > 0, so the bits order like the depths), 0xffffffff
    // for the others (sorted last); value = index; digit histograms of the
    // keys ([4][256], accumulated)
    uint32_t* dkeys;
    uint32_t* dvals;
    uint32_t* dhist;
    // staged kernel only: where a bulk copy that did not land is reported
    StatusHeader* header;
};

// Where preprocess_one reads a Gaussian's parameters: the caller's arrays in
// global memory, or a block's shared-memory stage of them (same layouts,
// indexed from the stage's first Gaussian).
struct GlobalIn {
    const PreArgs& a;
    int64_t g;
    __device__ float mean(int k) const { return __ldg(a.means + 3 * g + k); }
    __device__ float4 quat() const { return __ldg(a.quats + g); }
    __device__ float log_scale(int k) const { return __ldg(a.log_scales + 3 * g + k); }
    __device__ float logit() const { return __ldg(a.logits + g); }
    template <int D>
    __device__ void sh(float* co) const {
        load_sh<D, false>(a.sh + g * (D + 1) * (D + 1) * 3, co);
    }
};
struct SharedIn {
    const float* means;
    const float4* quats;
    const float* log_scales;
    const float* logits;
    const float* shs;
    int i;
    uint64_t* sh_bar;     // the SH rows land on their own barrier, waited for here
    uint32_t parity;
    __device__ float mean(int k) const { return means[3 * i + k]; }
    __device__ float4 quat() const { return quats[i]; }
    __device__ float log_scale(int k) const { return log_scales[3 * i + k]; }
    __device__ float logit() const { return logits[i]; }
    template <int D>
    __device__ void sh(float* co) const {
        mbar_wait_bounded(sh_bar, parity, kBulkWaitLimit);   // a failure is recorded by the block after the chunk
        load_sh<D, true>(shs + i * (D + 1) * (D + 1) * 3, co);
    }
};

// One Gaussian seen by one camera; returns its depth-order key.
template <int D, typename In>
__device__ __forceinline__ uint32_t preprocess_one(const PreArgs& a, int64_t g, const In& in) {
    const CamConst& C = a.cam;
    const float m0 = in.mean(0), m1 = in.mean(1), m2 = in.mean(2);

    float p[3];
#pragma unroll
    for (int i = 0; i < 3; i++)
        p[i] = add(add(add(mul(C.R[3 * i], m0), mul(C.R[3 * i + 1], m1)), mul(C.R[3 * i + 2], m2)), C.t[i]);
    const float z = p[2];
    a.depth[g] = z;

    bool ok = z > C.near_z;
    float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ok) {
        q = in.quat();
    }
    const float n2 = add(add(add(mul(q.x, q.x), mul(q.y, q.y)), mul(q.z, q.z)), mul(q.w, q.w));
    ok = ok && n2 > 0.0f && n2 <= FLT_MAX;
    if (!ok) {
        if (a.radius) a.radius[g] = 0;
        a.tiles_touched[g] = 0;
        a.rect[g] = make_ushort4(0, 0, 0, 0);
        return 0xffffffffu;
    }
    const float rn = sq(n2);
    const float w = dv(q.x, rn), x = dv(q.y, rn), y = dv(q.z, rn), zq = dv(q.w, rn);
    float G[9];
    {
        const float xx = mul(x, x), yy = mul(y, y), zz = mul(zq, zq);
        const float xy = mul(x, y), xz = mul(x, zq), yz = mul(y, zq);
        const float wx = mul(w, x), wy = mul(w, y), wz = mul(w, zq);
        G[0] = sub(1.0f, mul(2.0f, add(yy, zz)));
        G[1] = mul(2.0f, sub(xy, wz));
        G[2] = mul(2.0f, add(xz, wy));
        G[3] = mul(2.0f, add(xy, wz));
        G[4] = sub(1.0f, mul(2.0f, add(xx, zz)));
        G[5] = mul(2.0f, sub(yz, wx));
        G[6] = mul(2.0f, sub(xz, wy));
        G[7] = mul(2.0f, add(yz, wx));
        G[8] = sub(1.0f, mul(2.0f, add(xx, yy)));
    }
    float s[3];
#pragma unroll
    for (int k = 0; k < 3; k++) s[k] = exp32(in.log_scale(k));
    float Arot[9], B[9];   // Arot = W R (the Gaussian's axes in camera space), B = Arot S
#pragma unroll
    for (int i = 0; i < 3; i++)
#pragma unroll
        for (int j = 0; j < 3; j++) {
            Arot[3 * i + j] = add(add(mul(C.R[3 * i], G[j]), mul(C.R[3 * i + 1], G[3 + j])), mul(C.R[3 * i + 2], G[6 + j]));
            B[3 * i + j] = mul(Arot[3 * i + j], s[j]);
        }
    const float j00 = dv(C.fx, z), j11 = dv(C.fy, z);
    const float zz2 = mul(z, z);
    const float fxp0 = mul(C.fx, p[0]), fyp1 = mul(C.fy, p[1]);
    const float j02 = -dv(fxp0, zz2), j12 = -dv(fyp1, zz2);
    float M0[3], M1[3];
#pragma unroll
    for (int k = 0; k < 3; k++) {
        M0[k] = add(mul(j00, B[k]), mul(j02, B[6 + k]));
        M1[k] = add(mul(j11, B[3 + k]), mul(j12, B[6 + k]));
    }
    const float ca = add(add(mul(M0[0], M0[0]), mul(M0[1], M0[1])), mul(M0[2], M0[2]));
    const float cb = add(add(mul(M0[0], M1[0]), mul(M0[1], M1[1])), mul(M0[2], M1[2]));
    const float cc = add(add(mul(M1[0], M1[0]), mul(M1[1], M1[1])), mul(M1[2], M1[2]));
    const float det = sub(mul(ca, cc), mul(cb, cb));
    const float hm = mul(0.5f, sub(ca, cc));
    const float mid = mul(0.5f, add(ca, cc));
    const float lam = add(mid, sq(add(mul(hm, hm), mul(cb, cb))));
    const float rf = ceilf(mul(3.0f, sq(lam)));
    const float u = add(dv(fxp0, z), C.cx);
    const float v = add(dv(fyp1, z), C.cy);
    if (!(det > 0.0f && det <= FLT_MAX) || !(fabsf(u) <= FLT_MAX && fabsf(v) <= FLT_MAX && rf <= FLT_MAX)) {
        if (a.radius) a.radius[g] = 0;
        a.tiles_touched[g] = 0;
        a.rect[g] = make_ushort4(0, 0, 0, 0);
        return 0xffffffffu;
    }
    float x0 = ceilf(sub(u, rf)), x1 = floorf(add(u, rf));
    float y0 = ceilf(sub(v, rf)), y1 = floorf(add(v, rf));
    x0 = x0 > 0.0f ? x0 : 0.0f;
    y0 = y0 > 0.0f ? y0 : 0.0f;
    const float wm1 = (float)(C.width - 1), hm1 = (float)(C.height - 1);
    x1 = x1 < wm1 ? x1 : wm1;
    y1 = y1 < hm1 ? y1 : hm1;
    uint32_t touched = 0;
    ushort4 rect = make_ushort4(0, 0, 0, 0);
    if (x0 <= x1 && y0 <= y1) {
        const int tx0 = (int)x0 >> 4, tx1 = (int)x1 >> 4, ty0 = (int)y0 >> 4, ty1 = (int)y1 >> 4;
        touched = (uint32_t)((tx1 - tx0 + 1) * (ty1 - ty0 + 1));
        rect = make_ushort4((unsigned short)tx0, (unsigned short)ty0, (unsigned short)tx1, (unsigned short)ty1);
    }
    if (a.radius) a.radius[g] = rf <= 1073741824.0f ? (int32_t)rf : 1073741824;
    a.tiles_touched[g] = touched;
    a.rect[g] = rect;
    if (a.mean2d) a.mean2d[g] = make_float2(u, v);

    // continuous values (ordinary fp32)
    // det Sigma' without cancellation: Sigma' = M M^T with M = J Arot S, so by
    // the Lagrange identity det = |M_0 x M_1|^2, and (Lu) x (Lv) = cof(L)(u x v)
    // with L = (Arot S)^T gives M_0 x M_1 = diag(s1 s2, s0 s2, s0 s1) Arot^T
    // (J_0 x J_1), J_0 x J_1 = (fx fy / z^3) p: a sum of three squares, each a
    // scaled dot product that is small only when its term does not matter.
    float det_acc;
    {
        const float kz = (C.fx * C.fy) / (z * z * z);
        const float sp[3] = {s[1] * s[2], s[0] * s[2], s[0] * s[1]};
        det_acc = 0.0f;
#pragma unroll
        for (int k = 0; k < 3; k++) {
            const float dk = sp[k] * kz * (Arot[k] * p[0] + Arot[3 + k] * p[1] + Arot[6 + k] * p[2]);
            det_acc = fmaf(dk, dk, det_acc);
        }
        if (!(det_acc > 0.0f) || !isfinite(det_acc)) det_acc = det;
    }
    const float inv_det = 1.0f / det_acc;
    const float logit = in.logit();
    const float o = 1.0f / (1.0f + expf(-logit));
    const float conA = cc * inv_det, conB = -cb * inv_det, conC = ca * inv_det;
    if (a.conic_opacity) a.conic_opacity[g] = make_float4(conA, conB, conC, o);

    float dx = m0 - C.campos[0], dy = m1 - C.campos[1], dz = m2 - C.campos[2];
    const float il = rsqrtf(dx * dx + dy * dy + dz * dz);
    dx *= il; dy *= il; dz *= il;
    float co[(D + 1) * (D + 1) * 3];
    in.template sh<D>(co);
    const float3 col = eval_sh<D>(co, dx, dy, dz);
    if (a.rgb) {
        a.rgb[3 * g] = col.x;
        a.rgb[3 * g + 1] = col.y;
        a.rgb[3 * g + 2] = col.z;
    }
    if (a.raster && touched) {
        // the compositor's record (three float4):
        //  {u, v, du, dv}: decision centre and the residual to the accurate
        //      centre, from a compensated evaluation of the projection
        //  {k1, k2, k3, log2 o}: log2(alpha) = log2 o - (k1 dx)^2 - (k2 dy + k3 dx)^2
        //  {r, g, b, half2(hx, hy)}: colour and the half-extents (rounded up) of
        //      the box holding {d : o exp(-d^T conic d / 2) >= 1/255}, i.e.
        //      sqrt(tau Sigma'_xx), sqrt(tau Sigma'_yy), tau = 2 ln(255 o),
        //      widened by margins far above the rounding of the per-pixel alpha;
        //      +inf (never culled) when Sigma' is too ill-conditioned for them,
        //      -1 (always culled) when o < 1/255 (margin included)
        float xh, xl, yh, yl, zh, zl, uh, ul, vh, vl;
        dot3_add(C.R, m0, m1, m2, C.t[0], xh, xl);
        dot3_add(C.R + 3, m0, m1, m2, C.t[1], yh, yl);
        dot3_add(C.R + 6, m0, m1, m2, C.t[2], zh, zl);
        project_df(C.fx, xh, xl, zh, zl, C.cx, uh, ul);
        project_df(C.fy, yh, yl, zh, zl, C.cy, vh, vl);
        const float tau = 2.0f * logf(255.0f * o) + 0.02f;
        float hx = INFINITY, hy = INFINITY;
        if (!(tau > 0.0f)) {
            hx = hy = -1.0f;
        } else if ((ca + cc) * (ca + cc) <= 1e8f * det_acc) {
            hx = 1.01f * sqrtf(tau * ca) + 0.05f;
            hy = 1.01f * sqrtf(tau * cc) + 0.05f;
        }
        const __half2 h = __halves2half2(__float2half_ru(hx), __float2half_ru(hy));
        float4* rec = a.raster + 3 * g;
        rec[0] = make_float4(u, v, (uh - u) + ul, (vh - v) + vl);
        // q = d^T Sigma'^-1 d = (dx / sqrt(a))^2 + ((a dy - b dx) / sqrt(a det))^2:
        // a sum of two squares (relative error ~eps sqrt(cond), where the
        // expanded conic form loses ~eps cond); scaled by sqrt(log2(e) / 2) so
        // that log2(alpha) = log2 o - t1^2 - t2^2, t1 = k1 dx, t2 = k2 dy + k3 dx
        const float sc = 0.84932180028801907f;   // sqrt(log2(e) / 2)
        const float ra = rsqrtf(ca);
        const float k1 = sc * ra;
        const float k2 = sc * sqrtf(ca * inv_det);
        const float k3 = -sc * cb * ra * rsqrtf(det_acc);
        rec[1] = make_float4(k1, k2, k3, log2f(o));
        rec[2] = make_float4(col.x, col.y, col.z, __uint_as_float(*reinterpret_cast<const uint32_t*>(&h)));
    }
    return touched ? __float_as_uint(z) : 0xffffffffu;
}

// The depth-order key of Gaussian g into the sort input and the block's digit
// histograms (8-bit digits of the 32-bit key, [4][256] in shared memory).
// The two high digits take few values across a warp (depths of nearby
// magnitude share their exponent bits), so they are counted once per distinct
// value per warp; the two low ones are near-uniform and counted per key.
// Called by whole warps (inactive lanes pass valid = false).
__device__ __forceinline__ void emit_depth_key(const PreArgs& a, int64_t g, uint32_t key, uint32_t* s_hist,
                                               bool valid = true) {
    if (valid) {
        a.dkeys[g] = key;
        a.dvals[g] = (uint32_t)g;
        atomicAdd(&s_hist[key & 255u], 1u);
        atomicAdd(&s_hist[256 + ((key >> 8) & 255u)], 1u);
    }
    const uint32_t lt = (1u << (threadIdx.x & 31)) - 1u;
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
#pragma unroll
    for (int p = 2; p < 4; p++) {
        const uint32_t d = (key >> (8 * p)) & 255u;
        const uint32_t peers = __match_any_sync(0xffffffffu, valid ? d : 0xffffffffu) & vmask;
        if (valid && (peers & lt) == 0) atomicAdd(&s_hist[p * 256 + d], (uint32_t)__popc(peers));
    }
}
__device__ __forceinline__ void flush_depth_hist(const uint32_t* s_hist, uint32_t* hist) {
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x)
        if (s_hist[i]) atomicAdd(&hist[i], s_hist[i]);
}

// Grid-stride over the Gaussians with as many blocks as fit on the GPU at
// once, so that the per-block digit histograms of the depth keys are flushed
// by few blocks.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const PreArgs a) {
    grid_dependency_begin();
    __shared__ uint32_t s_hist[4 * 256];
    if (a.dkeys)
        for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x) s_hist[i] = 0;
    __syncthreads();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // warp-uniform trip count (the key emission works on whole warps)
    for (int64_t g0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); g0 < a.n; g0 += stride) {
        const int64_t g = g0 + (threadIdx.x & 31);
        const bool valid = g < a.n;
        const uint32_t key = valid ? preprocess_one<D>(a, g, GlobalIn{a, g}) : 0u;
        if (a.dkeys) emit_depth_key(a, g, key, s_hist, valid);
    }
    if (a.dkeys) flush_depth_hist(s_hist, a.dhist);
}

// The same projection with the parameters staged through shared memory.
// Persistent blocks (six per SM) take chunks of kStage Gaussians in turn; for
// each chunk one thread issues five bulk copies (means, quaternions,
// log-scales, logits, SH rows: 236 B per Gaussian at degree 3, 30 KB per
// chunk). The first four land on one mbarrier and the SH rows on a second, so
// the decision program starts on the 44 B per Gaussian it needs while the
// 192 B of SH rows are still on their way; every thread then projects its
// Gaussian from the stage. With three chunks in flight per SM the HBM stream
// does not wait on per-thread load latency. A chunk that is not whole (the
// tail) is read from global memory directly. Waits are bounded (kBulkWaitLimit
// polls): a copy that did not land in time sets GS_FLAG_TIMEOUT, and the block
// waits once more (again bounded) for its copy before it leaves.
constexpr int kStage = 128;
template <int D>
constexpr int stage_bytes() {
    return kStage * (12 + 16 + 12 + 4 + (D + 1) * (D + 1) * 12);
}

template <int D>
__global__ void __launch_bounds__(kStage, 6) preprocess_staged_kernel(const PreArgs a) {
    grid_dependency_begin();
    extern __shared__ __align__(16) unsigned char s_stage[];
    __shared__ uint32_t s_hist[4 * 256];
    __shared__ __align__(8) uint64_t s_bar[2];   // means..logits, SH rows
    constexpr int NK3 = (D + 1) * (D + 1) * 3;
    float* s_means = reinterpret_cast<float*>(s_stage);
    float4* s_quats = reinterpret_cast<float4*>(s_stage + kStage * 12);
    float* s_ls = reinterpret_cast<float*>(s_stage + kStage * 28);
    float* s_logits = reinterpret_cast<float*>(s_stage + kStage * 40);
    float* s_sh = reinterpret_cast<float*>(s_stage + kStage * 44);
    const int tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(&s_bar[0], 1);
        mbar_init(&s_bar[1], 1);
        mbar_init_fence();
    }
    if (a.dkeys)
        for (int i = tid; i < 4 * 256; i += kStage) s_hist[i] = 0;
    __syncthreads();
    const int64_t chunks = (a.n + kStage - 1) / kStage, whole = a.n / kStage;
    auto issue = [&](int64_t c) {   // one thread, whole chunks only
        const int64_t g0 = c * kStage;
        mbar_arrive_expect_tx(&s_bar[0], (uint32_t)(kStage * 44));
        mbar_arrive_expect_tx(&s_bar[1], (uint32_t)(kStage * NK3 * 4));
        bulk_copy_g2s(s_means, a.means + 3 * g0, kStage * 12, &s_bar[0]);
        bulk_copy_g2s(s_quats, a.quats + g0, kStage * 16, &s_bar[0]);
        bulk_copy_g2s(s_ls, a.log_scales + 3 * g0, kStage * 12, &s_bar[0]);
        bulk_copy_g2s(s_logits, a.logits + g0, kStage * 4, &s_bar[0]);
        bulk_copy_g2s(s_sh, a.sh + NK3 * g0, kStage * NK3 * 4, &s_bar[1]);
    };
    uint32_t parity = 0;
    int64_t c = blockIdx.x;
    if (tid == 0 && c < whole) issue(c);
    for (; c < chunks; c += gridDim.x) {
        const bool staged = c < whole;   // the same for the whole block
        if (staged) {
            const bool landed = mbar_wait_bounded(&s_bar[0], parity, kBulkWaitLimit);
            if (__syncthreads_or(!landed)) {
                if (tid == 0) raise_flag(a.header, GS_FLAG_TIMEOUT, 3u);
                mbar_wait_bounded(&s_bar[0], parity, kBulkWaitLimit);
                mbar_wait_bounded(&s_bar[1], parity, kBulkWaitLimit);
                return;
            }
        }
        const int64_t g = c * kStage + tid;
        const bool valid = g < a.n;
        uint32_t key = 0u;
        if (valid) {
            if (staged)
                key = preprocess_one<D>(a, g, SharedIn{s_means, s_quats, s_ls, s_logits, s_sh, tid, &s_bar[1], parity});
            else
                key = preprocess_one<D>(a, g, GlobalIn{a, g});
        }
        if (a.dkeys) emit_depth_key(a, g, key, s_hist, valid);
        if (staged) {
            // the SH rows have landed (culled Gaussians never read them) before the stage is reused
            const bool landed = mbar_wait_bounded(&s_bar[1], parity, kBulkWaitLimit);
            parity ^= 1u;
            if (__syncthreads_or(!landed)) {
                if (tid == 0) raise_flag(a.header, GS_FLAG_TIMEOUT, 3u);
                mbar_wait_bounded(&s_bar[1], parity ^ 1u, kBulkWaitLimit);
                return;
            }
        }
        __syncthreads();   // every read of the stage is done before the next copy lands in it
        const int64_t next = c + gridDim.x;
        if (tid == 0 && next < whole) {
            fence_proxy_async_shared();
            issue(next);
        }
    }
    if (a.dkeys) flush_depth_hist(s_hist, a.dhist);
}

// Several cameras in one pass over the parameters: each thread projects its
// Gaussian for every view in turn, so the 236 B of parameters come from HBM
// once (the repeated loads of the same thread hit L1/L2) and each view's
// record is written to that view's arrays.
struct PreBatchArgs {
    PreArgs v[kMaxBatchViews];
    int views;
};

template <int D>
__global__ void __launch_bounds__(256) preprocess_batch_kernel(const PreBatchArgs a) {
    grid_dependency_begin();
    __shared__ uint32_t s_hist[kMaxBatchViews * 4 * 256];   // per view
    const int nv = a.views;
    for (int k = threadIdx.x; k < nv * 1024; k += blockDim.x) s_hist[k] = 0;
    __syncthreads();
    const int64_t n = a.v[0].n, stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); g0 < n; g0 += stride) {
        const int64_t g = g0 + (threadIdx.x & 31);
        const bool valid = g < n;
        for (int i = 0; i < nv; i++) {
            const uint32_t key = valid ? preprocess_one<D>(a.v[i], g, GlobalIn{a.v[i], g}) : 0u;
            if (a.v[i].dkeys) emit_depth_key(a.v[i], g, key, s_hist + i * 1024, valid);
        }
    }
    for (int i = 0; i < nv; i++)
        if (a.v[i].dkeys) flush_depth_hist(s_hist + i * 1024, a.v[i].dhist);
}

PreArgs pre_args(const gs_gaussians& g, const CamConst& cam, const gs_projected& out, const DepthKeysOut* dk) {
    PreArgs a;
    a.means = g.means;
    a.quats = reinterpret_cast<const float4*>(g.quats);
    a.log_scales = g.log_scales;
    a.logits = g.opacity_logits;
    a.sh = g.sh;
    a.n = g.n;
    a.cam = cam;
    a.mean2d = reinterpret_cast<float2*>(out.mean2d);
    a.raster = reinterpret_cast<float4*>(out.raster);
    a.conic_opacity = reinterpret_cast<float4*>(out.conic_opacity);
    a.rgb = out.rgb;
    a.depth = out.depth;
    a.radius = out.radius;
    a.tiles_touched = out.tiles_touched;
    a.rect = reinterpret_cast<ushort4*>(out.rect);
    a.dkeys = dk ? dk->keys : nullptr;
    a.dvals = dk ? dk->vals : nullptr;
    a.dhist = dk ? dk->hist : nullptr;
    a.header = nullptr;
    return a;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Grid of the staged kernel: its resident blocks (three per SM), with the
// dynamic shared memory of its stage allowed once per device.
template <int D>
cudaError_t launch_staged(const PreArgs& a, cudaStream_t s) {
    static std::mutex mu;
    static std::map<int, int64_t> grid;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int64_t cap = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = grid.find(dev);
        if (it == grid.end()) {
            e = cudaFuncSetAttribute(preprocess_staged_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     stage_bytes<D>());
            if (e != cudaSuccess) return e;
            int sms = 0, per_sm = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, preprocess_staged_kernel<D>, kStage,
                                                              stage_bytes<D>());
            if (e != cudaSuccess) return e;
            it = grid.emplace(dev, (int64_t)(per_sm > 0 ? per_sm : 1) * sms).first;
        }
        cap = it->second;
    }
    const int64_t need = (a.n + kStage - 1) / kStage;
    launch_k(preprocess_staged_kernel<D>, (unsigned)(need < cap ? need : cap), kStage, stage_bytes<D>(), s, a);
    return cudaGetLastError();
}

// blocks of 256 that fit on the current GPU at once for this kernel
// (occupancy computed once per device and kernel; every instantiation has its
// own cache entry). Only the grid size depends on it: the kernels are
// grid-stride loops.
template <typename K>
unsigned resident_blocks(K kernel, int64_t n) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int64_t> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    const auto key = std::make_pair(dev, reinterpret_cast<const void*>(kernel));
    int64_t cap = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it == cache.end()) {
            int sms = 0, per_sm = 0;
            if (dev < 0 || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess) per_sm = 0;
            it = cache.emplace(key, (int64_t)(per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 148)).first;
        }
        cap = it->second;
    }
    const int64_t need = (n + 255) / 256;
    return (unsigned)(need < cap ? need : cap);
}

}  // namespace

cudaError_t launch_preprocess_batch(const gs_gaussians& g, const CamConst* cams, const gs_projected* outs,
                                    const DepthKeysOut* dks, int views, cudaStream_t s) {
    if (g.n == 0 || views <= 0) return cudaSuccess;
    if (views > kMaxBatchViews) return cudaErrorInvalidValue;
    PreBatchArgs a;
    for (int i = 0; i < views; i++) a.v[i] = pre_args(g, cams[i], outs[i], dks ? dks + i : nullptr);
    a.views = views;
    switch (g.sh_degree) {
        case 0:
            launch_k(preprocess_batch_kernel<0>, resident_blocks(preprocess_batch_kernel<0>, g.n), 256, 0, s, a);
            break;
        case 1:
            launch_k(preprocess_batch_kernel<1>, resident_blocks(preprocess_batch_kernel<1>, g.n), 256, 0, s, a);
            break;
        case 2:
            launch_k(preprocess_batch_kernel<2>, resident_blocks(preprocess_batch_kernel<2>, g.n), 256, 0, s, a);
            break;
        default:
            launch_k(preprocess_batch_kernel<3>, resident_blocks(preprocess_batch_kernel<3>, g.n), 256, 0, s, a);
            break;
    }
    return cudaGetLastError();
}

cudaError_t launch_preprocess(const gs_gaussians& g, const CamConst& cam, const gs_projected& out,
                              cudaStream_t s, const DepthKeysOut* dk, StatusHeader* status) {
    if (g.n == 0) return cudaSuccess;
    PreArgs a = pre_args(g, cam, out, dk);
    if (status && aligned16(g.means) && aligned16(g.quats) && aligned16(g.log_scales) &&
        aligned16(g.opacity_logits) && aligned16(g.sh)) {
        a.header = status;
        switch (g.sh_degree) {
            case 0: return launch_staged<0>(a, s);
            case 1: return launch_staged<1>(a, s);
            case 2: return launch_staged<2>(a, s);
            default: return launch_staged<3>(a, s);
        }
    }
    switch (g.sh_degree) {
        case 0:
            launch_k(preprocess_kernel<0>, resident_blocks(preprocess_kernel<0>, g.n), 256, 0, s, a);
            break;
        case 1:
            launch_k(preprocess_kernel<1>, resident_blocks(preprocess_kernel<1>, g.n), 256, 0, s, a);
            break;
        case 2:
            launch_k(preprocess_kernel<2>, resident_blocks(preprocess_kernel<2>, g.n), 256, 0, s, a);
            break;
        default:
            launch_k(preprocess_kernel<3>, resident_blocks(preprocess_kernel<3>, g.n), 256, 0, s, a);
            break;
    }
    return cudaGetLastError();
}

GS_DEFINE_CHECK_SETTER(preprocess)

}  // namespace gs
