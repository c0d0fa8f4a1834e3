// Backward pass of the forward renderer: gradients of a loss L(image) with
// respect to the Gaussian parameters, given dL/dimage.
//
// Method: lesson page "3D Gaussian Splatting à partir de zéro", section
// "Rastérisation, non rayée": every stage of the renderer is differentiable,
// which is what lets the parameters be fitted by gradient descent. The pages
// print no backward formulas; these kernels compute the derivative of the
// forward function of the other kernels (preprocess.cu, rasterize.cu) by the
// chain rule, with the forward's discrete decisions (culling, tile lists,
// the 1/255 skip, the 1e-4 stop) held fixed, as they are piecewise constant.
//
// Step 5 backward (rasterize_backward_kernel). Per pixel, the forward composite
// is out = sum_i alpha_i T_i c_i + T_N bg with T_i = prod_{j<i} (1 - alpha_j).
// Walking the contributors from the last to the first:
//     T_i   = T_{i+1} / (1 - alpha_i)                 (T_N = final T)
//     dL/dc_i     += alpha_i T_i g                     (g = dL/dout)
//     dL/dalpha_i  = T_i (c_i - a_i) . g,  a_i = (sum_{j>i} alpha_j T_j c_j + T_N bg) / T_{i+1}
//     a_{i-1}      = alpha_i c_i + (1 - alpha_i) a_i  (a = bg after the last)
// and, unless alpha_i sits at the 0.99 cap, alpha = o exp(-sigma),
// sigma = (A dx^2 + 2 B dx dy + C dy^2) / 2 with d = pixel - centre:
//     dL/do += dL/dalpha alpha / o,  dL/dsigma = -alpha dL/dalpha,
//     dL/d(A, B, C) += dL/dsigma (dx^2 / 2, dx dy, dy^2 / 2),
//     dL/d(u, v)    += -dL/dsigma (A dx + B dy, B dx + C dy).
// alpha is recomputed from the same packed record with the same operations as
// the forward kernel, so every skip decision and every alpha is bit-identical.
// The tile, warp and lane layout, the per-warp ballot of entries whose alpha
// box meets the warp's 8x8 block, and the list staging are the forward's; the
// list is walked from the last contributor of the tile backwards. A lane's two
// pixels are carried as pairs in packed fp32 arithmetic (PTX .f32x2): a pixel
// that does not take the entry blends alpha = 0, which leaves its T and its
// suffix colour a unchanged and adds no gradient, so both pixels run the same
// instructions without branching. Per entry, the warp sums its lanes'
// contributions (a reduce-scatter of the 9 values over the lanes) and nine
// lanes add them into the batch's shared-memory sums for that entry, where the
// block's other warps add theirs; once the whole block has walked the batch,
// one thread per entry adds the nine sums to the Gaussian's gradient with
// global atomics (one set per tile instead of one per warp).
//
// Step 1 backward (preprocess_backward_kernel): one thread per Gaussian maps
// dL/d(u, v), dL/d(conic), dL/do, dL/dc to the parameters through
//     rgb = max(0, sum_k Y_k(dir) sh_k + 0.5), dir = normalize(mu - campos)
//     o = sigmoid(logit)
//     (u, v) = (fx x/z + cx, fy y/z + cy), x_c = W mu + t
//     conic = Sigma'^-1,  Sigma' = J W Sigma W^T J^T,  J = J(x_c)
//     Sigma = M M^T, M = R(q / |q|) diag(exp(log_scale)).
#include <cuda_fp16.h>

#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kBwdThreads = 128;   // the forward's tile layout: 4 warps of 8x8 pixels, two per lane
constexpr float kLog2AlphaMin = -7.99435343685886f;   // log2(1/255)
constexpr float kTwoOverLog2e = 1.3862943611198906f;  // 2 ln 2 = 2 / log2(e)

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

typedef unsigned long long f2x;   // two fp32 in one 64-bit register pair (PTX .f32x2)
__device__ __forceinline__ f2x pk2(float lo, float hi) {
    f2x r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 up2(f2x v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ f2x mul2(f2x a, f2x b) {
    f2x r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2x fma2(f2x a, f2x b, f2x c) {
    f2x r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ f2x sub2(f2x a, f2x b) {
    f2x r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float hsum(f2x v) {
    const float2 p = up2(v);
    return p.x + p.y;
}

// Sums 9 per-lane values over the warp as a reduce-scatter: at each butterfly
// step a lane keeps one half of its slots and receives the partner's partial
// sums of that half (8 + 4 + 2 + 1 + 1 = 16 shuffles for 16 slots, 7 of them
// zero). Returns the complete sum of slot slot_of(lane) on even lanes.
__device__ __forceinline__ float warp_reduce_scatter9(const float (&in)[9], int lane) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 9; i++) v[i] = in[i];
#pragma unroll
    for (int i = 9; i < 16; i++) v[i] = 0.0f;
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
        const bool up = (lane & (2 * w)) != 0;
#pragma unroll
        for (int i = 0; i < w; i++) {
            const float send = up ? v[i] : v[i + w];
            const float keep = up ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * w);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}
__device__ __forceinline__ int slot_of(int lane) {
    return ((lane >> 1) & 1) | (((lane >> 2) & 1) << 1) | (((lane >> 3) & 1) << 2) | (((lane >> 4) & 1) << 3);
}

struct BwdArgs {
    const float4* raster;
    const uint32_t* order;
    const uint32_t* sorted_vals;
    const uint2* ranges;
    uint32_t n;
    int width, height, tiles_x;
    float bg0, bg1, bg2;
    const float* final_T;
    const uint32_t* n_contrib;
    const float* grad_image;
    float* g_mean2d;   // [n][2]
    float* g_conic;    // [n][3]
    float* g_opacity;  // [n]
    float* g_rgb;      // [n][3]
};

// Per (pixel, entry) state of the backward walk for one pixel.
struct PixelState {
    float T, a0, a1, a2, g0, g1, g2;
    uint32_t last;
};

__global__ void __launch_bounds__(kBwdThreads) rasterize_backward_kernel(const BwdArgs a) {
    grid_dependency_begin();
    __shared__ float4 s_q[2][kBwdThreads];    // (mx, my, k1, k2), centre tile-local
    __shared__ float4 s_r[2][kBwdThreads];    // (k3, log2 o, r, g)
    __shared__ float2 s_c[2][kBwdThreads];    // (b, 1/o)
    __shared__ float4 s_box[2][kBwdThreads];  // alpha >= 1/255 box, tile-local
    __shared__ float4 w_q[kBwdThreads / 32][32];
    __shared__ float4 w_r[kBwdThreads / 32][32];
    __shared__ float4 w_c[kBwdThreads / 32][32];   // (b, 1/o, list position as bits, unused)
    // the batch's gradient sums, [batch entry][9], added to by every warp that
    // takes the entry and flushed to global memory once per batch (double-buffered
    // so that one batch's flush overlaps the next batch's walk)
    __shared__ float s_acc[2][kBwdThreads * 9];
    __shared__ uint32_t s_g[2][kBwdThreads];   // the batch entries' Gaussians
    __shared__ uint32_t s_max;

    const int tile = a.order ? (int)a.order[blockIdx.x] : (int)blockIdx.x;
    const int tx = tile % a.tiles_x, ty = tile / a.tiles_x;
    const float tile_x0 = (float)(tx * kTile), tile_y0 = (float)(ty * kTile);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int lbx0 = 8 * (warp & 1), lby0 = 8 * (warp >> 1);
    const int lx = lbx0 + (lane & 7), ly = lby0 + (lane >> 3);
    const int px = tx * kTile + lx, py = ty * kTile + ly;
    const float fbx0 = (float)lbx0, fbx1 = (float)(lbx0 + 7), fby0 = (float)lby0, fby1 = (float)(lby0 + 7);
    const uint2 range = a.ranges[tile];
    const float fpx = (float)lx, fpy = (float)ly, fpy2 = (float)(ly + 4);

    auto load_pixel = [&](int x, int y, PixelState& s) {
        s.a0 = a.bg0;
        s.a1 = a.bg1;
        s.a2 = a.bg2;
        if (x < a.width && y < a.height) {
            const int64_t p = (int64_t)y * a.width + x;
            s.T = a.final_T[p];
            s.last = a.n_contrib[p];
            s.g0 = a.grad_image[3 * p];
            s.g1 = a.grad_image[3 * p + 1];
            s.g2 = a.grad_image[3 * p + 2];
        } else {
            s.T = 1.0f;
            s.last = 0;
            s.g0 = s.g1 = s.g2 = 0.0f;
        }
    };
    PixelState P1, P2;
    load_pixel(px, py, P1);
    load_pixel(px, py + 4, P2);
    f2x TT = pk2(P1.T, P2.T), AA0 = pk2(P1.a0, P2.a0), AA1 = pk2(P1.a1, P2.a1), AA2 = pk2(P1.a2, P2.a2);
    const f2x GG0 = pk2(P1.g0, P2.g0), GG1 = pk2(P1.g1, P2.g1), GG2 = pk2(P1.g2, P2.g2);

    if (threadIdx.x == 0) s_max = 0;
    for (int i = threadIdx.x; i < 2 * kBwdThreads * 9; i += kBwdThreads) (&s_acc[0][0])[i] = 0.0f;
    __syncthreads();
    {
        const uint32_t m = __reduce_max_sync(0xffffffffu, max(P1.last, P2.last));
        if (lane == 0) atomicMax(&s_max, m);
    }
    __syncthreads();
    // list positions [0, len) matter (an inverted range -- only a sort cut
    // short gives one, and it is flagged -- counts as empty)
    GS_CHECK(range.y >= range.x && s_max <= range.y - range.x);
    const uint32_t len = range.y > range.x ? min(s_max, range.y - range.x) : 0u;

    auto fetch = [&](uint32_t pos, float4& r0, float4& r1, float4& r2, uint32_t& gi) {
        uint32_t g = __ldg(a.sorted_vals + range.x + pos);
        GS_CHECK(g < a.n);
        gi = g;               // an out-of-scene index gets no gradient
        if (g >= a.n) g = 0;   // only a sort cut short (flagged) can give this
        r0 = __ldg(a.raster + 3 * g);
        r1 = __ldg(a.raster + 3 * g + 1);
        r2 = __ldg(a.raster + 3 * g + 2);
    };
    auto store = [&](int buf, const float4& r0, const float4& r1, const float4& r2, uint32_t gi) {
        s_g[buf][threadIdx.x] = gi;
        const float mx = (r0.x - tile_x0) + r0.z, my = (r0.y - tile_y0) + r0.w;
        const uint32_t hb = __float_as_uint(r2.w);
        const __half2 h = *reinterpret_cast<const __half2*>(&hb);
        const float hx = __low2float(h), hy = __high2float(h);
        s_q[buf][threadIdx.x] = make_float4(mx, my, r1.x, r1.y);
        s_r[buf][threadIdx.x] = make_float4(r1.z, r1.w, r2.x, r2.y);
        s_c[buf][threadIdx.x] = make_float2(r2.z, fast_exp2(-r1.w));
        s_box[buf][threadIdx.x] = make_float4(mx - hx, mx + hx, my - hy, my + hy);
    };

    // batches from the back: batch b holds positions [lo_b, hi_b), hi_b = len - 128 b
    const uint32_t nbatch = (len + kBwdThreads - 1) / kBwdThreads;
    auto lo_of = [&](uint32_t b) -> uint32_t {
        const uint32_t hi = len - b * kBwdThreads;
        return hi > (uint32_t)kBwdThreads ? hi - kBwdThreads : 0u;
    };
    if (nbatch > 0) {
        const uint32_t lo = lo_of(0);
        if (lo + threadIdx.x < len) {
            float4 r0, r1, r2;
            uint32_t gi;
            fetch(lo + threadIdx.x, r0, r1, r2, gi);
            store(0, r0, r1, r2, gi);
        }
    }
    __syncthreads();

    // one thread per entry of a finished batch: its nine sums to the global arrays
    auto flush = [&](int bf, uint32_t cnt) {
        const int t = threadIdx.x;
        if ((uint32_t)t >= cnt) return;
        float* acc = &s_acc[bf][t * 9];
        float v[9];
        bool any = false;
#pragma unroll
        for (int q = 0; q < 9; q++) {
            v[q] = acc[q];
            any |= v[q] != 0.0f;
            acc[q] = 0.0f;
        }
        const uint32_t g = s_g[bf][t];
        if (!any || g >= a.n) return;
        atomicAdd(a.g_mean2d + 2 * g, v[0]);
        atomicAdd(a.g_mean2d + 2 * g + 1, v[1]);
        atomicAdd(a.g_conic + 3 * g, v[2]);
        atomicAdd(a.g_conic + 3 * g + 1, v[3]);
        atomicAdd(a.g_conic + 3 * g + 2, v[4]);
        atomicAdd(a.g_opacity + g, v[5]);
        atomicAdd(a.g_rgb + 3 * g, v[6]);
        atomicAdd(a.g_rgb + 3 * g + 1, v[7]);
        atomicAdd(a.g_rgb + 3 * g + 2, v[8]);
    };

    uint32_t prev_cnt = 0;
    for (uint32_t b = 0; b < nbatch; b++) {
        const int buf = b & 1;
        const uint32_t lo = lo_of(b), hi = len - b * kBwdThreads;
        const uint32_t cnt = hi - lo;
        const bool have_next = b + 1 < nbatch;
        float4 n0, n1, n2;
        uint32_t ng = 0;
        if (have_next) {
            const uint32_t nlo = lo_of(b + 1);
            if (nlo + threadIdx.x < lo) fetch(nlo + threadIdx.x, n0, n1, n2, ng);
        }
        // the previous batch's sums (every warp has passed the barrier after it)
        if (b > 0) flush(buf ^ 1, prev_cnt);
        // the list positions of this batch, last group first
#pragma unroll 1
        for (int i = kBwdThreads / 32 - 1; i >= 0; i--) {
            const uint32_t j = (uint32_t)(i * 32 + lane);
            bool hit = false;
            if (j < cnt) {
                const float4 bx = s_box[buf][j];
                hit = bx.x <= fbx1 && bx.y >= fbx0 && bx.z <= fby1 && bx.w >= fby0;
            }
            const uint32_t m = __ballot_sync(0xffffffffu, hit);
            if (m == 0) continue;
            if (hit) {
                const int pos = __popc(m & lt_mask);
                w_q[warp][pos] = s_q[buf][j];
                w_r[warp][pos] = s_r[buf][j];
                const float2 c = s_c[buf][j];
                const uint32_t lp = lo + j;
                w_c[warp][pos] = make_float4(c.x, c.y, __uint_as_float(lp), 0.0f);
            }
            __syncwarp();
            const int nh = __popc(m);
            for (int k = nh - 1; k >= 0; k--) {
                const float4 q = w_q[warp][k];
                const float4 r = w_r[warp][k];
                const float4 c = w_c[warp][k];
                const uint32_t lp = __float_as_uint(c.z);
                // the forward's exponent, operation for operation; the
                // offsets themselves enter the conic gradients
                const float dx = q.x - fpx, dy = q.y - fpy, dy2 = q.y - fpy2;
                const float2 A = entry_origin_terms(q.x, q.y, q.z, q.w, r.x);
                float t1, t2, t22, e, e2;
                pixel_pair_exponents(A.x, A.y, q.z, q.w, r.x, r.y, -fpx, -fpy, t1, t2, t22, e, e2);
                const bool c1 = lp < P1.last && e >= kLog2AlphaMin;
                const bool c2 = lp < P2.last && e2 >= kLog2AlphaMin;
                if (!__any_sync(0xffffffffu, c1 || c2)) continue;
                // both pixels in pairs; a pixel that does not take this entry blends alpha = 0,
                // which leaves its state as it is and adds nothing
                const float raw1 = c1 ? fast_exp2(e) : 0.0f, raw2 = c2 ? fast_exp2(e2) : 0.0f;
                const float al1 = fminf(0.99f, raw1), al2 = fminf(0.99f, raw2);
                const f2x AL = pk2(al1, al2);
                const float2 tt = up2(TT);
                const float ti1 = c1 ? __fdividef(tt.x, 1.0f - al1) : tt.x;   // 1 - alpha >= 0.01
                const float ti2 = c2 ? __fdividef(tt.y, 1.0f - al2) : tt.y;
                const f2x TI = pk2(ti1, ti2);
                const f2x W = mul2(AL, TI);
                const f2x D0 = sub2(pk2(r.z, r.z), AA0), D1 = sub2(pk2(r.w, r.w), AA1), D2 = sub2(pk2(c.x, c.x), AA2);
                const f2x DLDA = mul2(TI, fma2(D2, GG2, fma2(D1, GG1, mul2(D0, GG0))));
                AA0 = fma2(AL, D0, AA0);
                AA1 = fma2(AL, D1, AA1);
                AA2 = fma2(AL, D2, AA2);
                TT = TI;
                // below the 0.99 cap: dL/dsigma = -alpha dL/dalpha
                const f2x ADA = mul2(DLDA, AL);
                const f2x DLDS = mul2(ADA, pk2(raw1 < 0.99f ? -1.0f : 0.0f, raw2 < 0.99f ? -1.0f : 0.0f));
                const f2x TT2 = pk2(t2, t22), DDY = pk2(dy, dy2);
                const float zt1 = q.z * t1;
                const f2x KD = mul2(DLDS, pk2(kTwoOverLog2e, kTwoOverLog2e));
                const float gu = hsum(mul2(KD, fma2(pk2(r.x, r.x), TT2, pk2(zt1, zt1))));
                const float gv = hsum(mul2(KD, mul2(pk2(q.w, q.w), TT2)));
                const float hdx2 = 0.5f * dx * dx;
                const float gA = hsum(mul2(DLDS, pk2(hdx2, hdx2)));
                const float gB = hsum(mul2(DLDS, mul2(pk2(dx, dx), DDY)));
                const float gC = hsum(mul2(DLDS, mul2(pk2(0.5f, 0.5f), mul2(DDY, DDY))));
                const float go = hsum(mul2(ADA, pk2(raw1 < 0.99f ? c.y : 0.0f, raw2 < 0.99f ? c.y : 0.0f)));
                const float gr = hsum(mul2(W, GG0)), gg = hsum(mul2(W, GG1)), gb = hsum(mul2(W, GG2));
                const float part[9] = {gu, gv, gA, gB, gC, go, gr, gg, gb};
                const float sum = warp_reduce_scatter9(part, lane);
                const int slot = slot_of(lane);
                // into the batch's sums for this entry (the block's other warps add theirs)
                if (!(lane & 1) && slot < 9) atomicAdd(&s_acc[buf][(lp - lo) * 9 + slot], sum);
            }
            __syncwarp();
        }
        if (have_next) {
            const uint32_t nlo = lo_of(b + 1);
            if (nlo + threadIdx.x < lo) store(buf ^ 1, n0, n1, n2, ng);
        }
        __syncthreads();
        prev_cnt = cnt;
    }
    if (nbatch > 0) flush((nbatch - 1) & 1, prev_cnt);
}

// ------------------------------------------------------------------ step 1 backward

// Real SH basis constants (closed forms sqrt(1/4pi), sqrt(3/4pi), sqrt(15/4pi),
// sqrt(5/16pi), sqrt(15/16pi), sqrt(35/32pi), sqrt(105/4pi), sqrt(21/32pi),
// sqrt(7/16pi), sqrt(105/16pi)), the same basis and signs as the forward.
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

// Y_k(x, y, z) and its gradient for k < NK.
template <int NK>
__device__ __forceinline__ void sh_basis_grad(float x, float y, float z, float* Y, float3* dY) {
    Y[0] = kY0;
    dY[0] = make_float3(0.f, 0.f, 0.f);
    if constexpr (NK > 1) {
        Y[1] = -kY1 * y;  dY[1] = make_float3(0.f, -kY1, 0.f);
        Y[2] = kY1 * z;   dY[2] = make_float3(0.f, 0.f, kY1);
        Y[3] = -kY1 * x;  dY[3] = make_float3(-kY1, 0.f, 0.f);
    }
    if constexpr (NK > 4) {
        const float xx = x * x, yy = y * y, zz = z * z;
        Y[4] = kY2a * x * y;                 dY[4] = make_float3(kY2a * y, kY2a * x, 0.f);
        Y[5] = kY2a * y * z;                 dY[5] = make_float3(0.f, kY2a * z, kY2a * y);
        Y[6] = kY2b * (2.f * zz - xx - yy);  dY[6] = make_float3(-2.f * kY2b * x, -2.f * kY2b * y, 4.f * kY2b * z);
        Y[7] = kY2a * x * z;                 dY[7] = make_float3(kY2a * z, 0.f, kY2a * x);
        Y[8] = kY2c * (xx - yy);             dY[8] = make_float3(2.f * kY2c * x, -2.f * kY2c * y, 0.f);
        if constexpr (NK > 9) {
            Y[9] = -kY3a * y * (3.f * xx - yy);
            dY[9] = make_float3(-6.f * kY3a * x * y, -3.f * kY3a * (xx - yy), 0.f);
            Y[10] = kY3b * x * y * z;
            dY[10] = make_float3(kY3b * y * z, kY3b * x * z, kY3b * x * y);
            Y[11] = -kY3c * y * (4.f * zz - xx - yy);
            dY[11] = make_float3(2.f * kY3c * x * y, -kY3c * (4.f * zz - xx - 3.f * yy), -8.f * kY3c * y * z);
            Y[12] = kY3d * z * (2.f * zz - 3.f * xx - 3.f * yy);
            dY[12] = make_float3(-6.f * kY3d * x * z, -6.f * kY3d * y * z, kY3d * (6.f * zz - 3.f * xx - 3.f * yy));
            Y[13] = -kY3c * x * (4.f * zz - xx - yy);
            dY[13] = make_float3(-kY3c * (4.f * zz - 3.f * xx - yy), 2.f * kY3c * x * y, -8.f * kY3c * x * z);
            Y[14] = kY3e * z * (xx - yy);
            dY[14] = make_float3(2.f * kY3e * x * z, -2.f * kY3e * y * z, kY3e * (xx - yy));
            Y[15] = -kY3a * x * (xx - 3.f * yy);
            dY[15] = make_float3(-3.f * kY3a * (xx - yy), 6.f * kY3a * x * y, 0.f);
        }
    }
}

struct PreBwdArgs {
    const float* means;
    const float* quats;
    const float* log_scales;
    const float* logits;
    const float* sh;
    const uint32_t* tiles_touched;
    int64_t n;
    CamConst cam;
    const float* g_mean2d;
    const float* g_conic;
    const float* g_opacity;
    const float* g_rgb;
    float* d_means;
    float* d_quats;
    float* d_log_scales;
    float* d_logits;
    float* d_sh;
};

// One Gaussian; row holds its SH coefficients on entry and their gradients on
// return.
template <int D>
__device__ __forceinline__ void gaussian_backward(const PreBwdArgs& a, int64_t g, float* row) {
    constexpr int NK = (D + 1) * (D + 1);
    const CamConst& C = a.cam;
    if (__ldg(a.tiles_touched + g) == 0) {
        // culled or off-screen: the image does not depend on this Gaussian
        for (int i = 0; i < 3; i++) a.d_means[3 * g + i] = 0.f;
        for (int i = 0; i < 4; i++) a.d_quats[4 * g + i] = 0.f;
        for (int i = 0; i < 3; i++) a.d_log_scales[3 * g + i] = 0.f;
        a.d_logits[g] = 0.f;
        for (int i = 0; i < NK * 3; i++) row[i] = 0.f;
        return;
    }
    const float m[3] = {__ldg(a.means + 3 * g), __ldg(a.means + 3 * g + 1), __ldg(a.means + 3 * g + 2)};
    float dm[3] = {0.f, 0.f, 0.f};

    // colour: rgb = max(0, sum_k Y_k(dir) sh_k + 0.5), dir = (mu - campos) / |mu - campos|
    {
        float d[3] = {m[0] - C.campos[0], m[1] - C.campos[1], m[2] - C.campos[2]};
        const float len = sqrtf(d[0] * d[0] + d[1] * d[1] + d[2] * d[2]);
        const float il = 1.0f / len;
        const float x = d[0] * il, y = d[1] * il, z = d[2] * il;
        float Y[NK];
        float3 dY[NK];
        sh_basis_grad<NK>(x, y, z, Y, dY);
        float raw[3] = {0.5f, 0.5f, 0.5f};
        for (int k = 0; k < NK; k++)
            for (int c = 0; c < 3; c++) raw[c] = fmaf(Y[k], row[3 * k + c], raw[c]);
        float gc[3];
        for (int c = 0; c < 3; c++) gc[c] = raw[c] > 0.f ? __ldg(a.g_rgb + 3 * g + c) : 0.f;
        float gd[3] = {0.f, 0.f, 0.f};
        for (int k = 0; k < NK; k++) {
            float s = 0.f;
            for (int c = 0; c < 3; c++) {
                s = fmaf(row[3 * k + c], gc[c], s);
                row[3 * k + c] = Y[k] * gc[c];
            }
            gd[0] = fmaf(dY[k].x, s, gd[0]);
            gd[1] = fmaf(dY[k].y, s, gd[1]);
            gd[2] = fmaf(dY[k].z, s, gd[2]);
        }
        // through the normalisation: (I - dir dir^T) / |d|
        const float dot = gd[0] * x + gd[1] * y + gd[2] * z;
        dm[0] += (gd[0] - dot * x) * il;
        dm[1] += (gd[1] - dot * y) * il;
        dm[2] += (gd[2] - dot * z) * il;
    }
    // opacity
    {
        const float o = 1.0f / (1.0f + expf(-__ldg(a.logits + g)));
        a.d_logits[g] = __ldg(a.g_opacity + g) * o * (1.0f - o);
    }
    // camera space
    float xc[3];
    for (int i = 0; i < 3; i++) xc[i] = C.R[3 * i] * m[0] + C.R[3 * i + 1] * m[1] + C.R[3 * i + 2] * m[2] + C.t[i];
    const float z = xc[2], iz = 1.0f / z, iz2 = iz * iz;
    float dxc[3];
    {
        const float gu = __ldg(a.g_mean2d + 2 * g), gv = __ldg(a.g_mean2d + 2 * g + 1);
        dxc[0] = gu * C.fx * iz;
        dxc[1] = gv * C.fy * iz;
        dxc[2] = -(gu * C.fx * xc[0] + gv * C.fy * xc[1]) * iz2;
    }
    // Sigma = M M^T, M = R S
    const float4 q4 = reinterpret_cast<const float4*>(a.quats)[g];
    const float qn = sqrtf(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
    const float iq = 1.0f / qn;
    const float w = q4.x * iq, x = q4.y * iq, y = q4.z * iq, zq = q4.w * iq;
    const float Rq[9] = {1.f - 2.f * (y * y + zq * zq), 2.f * (x * y - w * zq), 2.f * (x * zq + w * y),
                         2.f * (x * y + w * zq), 1.f - 2.f * (x * x + zq * zq), 2.f * (y * zq - w * x),
                         2.f * (x * zq - w * y), 2.f * (y * zq + w * x), 1.f - 2.f * (x * x + y * y)};
    const float s[3] = {expf(__ldg(a.log_scales + 3 * g)), expf(__ldg(a.log_scales + 3 * g + 1)),
                        expf(__ldg(a.log_scales + 3 * g + 2))};
    float M[9];
    for (int i = 0; i < 3; i++)
        for (int j = 0; j < 3; j++) M[3 * i + j] = Rq[3 * i + j] * s[j];
    float Sig[9];
    for (int i = 0; i < 3; i++)
        for (int j = 0; j < 3; j++) Sig[3 * i + j] = M[3 * i] * M[3 * j] + M[3 * i + 1] * M[3 * j + 1] + M[3 * i + 2] * M[3 * j + 2];
    // T = J W (2x3)
    const float J00 = C.fx * iz, J02 = -C.fx * xc[0] * iz2, J11 = C.fy * iz, J12 = -C.fy * xc[1] * iz2;
    float T[6];
    for (int j = 0; j < 3; j++) {
        T[j] = J00 * C.R[j] + J02 * C.R[6 + j];
        T[3 + j] = J11 * C.R[3 + j] + J12 * C.R[6 + j];
    }
    // Sigma' = T Sig T^T
    float TS[6];
    for (int i = 0; i < 2; i++)
        for (int j = 0; j < 3; j++)
            TS[3 * i + j] = T[3 * i] * Sig[j] + T[3 * i + 1] * Sig[3 + j] + T[3 * i + 2] * Sig[6 + j];
    const float sa = TS[0] * T[0] + TS[1] * T[1] + TS[2] * T[2];
    const float sb = TS[0] * T[3] + TS[1] * T[4] + TS[2] * T[5];
    const float sc = TS[3] * T[3] + TS[4] * T[4] + TS[5] * T[5];
    const float det = sa * sc - sb * sb;
    const float idet = 1.0f / det;
    const float A = sc * idet, B = -sb * idet, Cc = sa * idet;
    // dL/dSigma' = -Q G Q, G = [[gA, gB/2], [gB/2, gC]], Q = conic
    const float gA = __ldg(a.g_conic + 3 * g), gB = 0.5f * __ldg(a.g_conic + 3 * g + 1), gC = __ldg(a.g_conic + 3 * g + 2);
    const float QG00 = A * gA + B * gB, QG01 = A * gB + B * gC, QG10 = B * gA + Cc * gB, QG11 = B * gB + Cc * gC;
    const float Ga = -(QG00 * A + QG01 * B);              // [0][0]
    const float Gb = -(QG00 * B + QG01 * Cc);             // [0][1] = [1][0]
    const float Gc = -(QG10 * B + QG11 * Cc);             // [1][1]
    // dL/dSig = T^T Gs T (3x3); dL/dT = 2 Gs T Sig (2x3)
    float dSig[9];
    for (int i = 0; i < 3; i++)
        for (int j = 0; j < 3; j++)
            dSig[3 * i + j] = T[i] * (Ga * T[j] + Gb * T[3 + j]) + T[3 + i] * (Gb * T[j] + Gc * T[3 + j]);
    float dT[6];
    for (int j = 0; j < 3; j++) {
        dT[j] = 2.f * (Ga * TS[j] + Gb * TS[3 + j]);
        dT[3 + j] = 2.f * (Gb * TS[j] + Gc * TS[3 + j]);
    }
    // T = J W: dL/dJ = dT W^T; J depends on x_c
    float dJ[6];
    for (int i = 0; i < 2; i++)
        for (int k = 0; k < 3; k++)
            dJ[3 * i + k] = dT[3 * i] * C.R[3 * k] + dT[3 * i + 1] * C.R[3 * k + 1] + dT[3 * i + 2] * C.R[3 * k + 2];
    const float iz3 = iz2 * iz;
    dxc[0] += dJ[2] * (-C.fx * iz2);
    dxc[1] += dJ[5] * (-C.fy * iz2);
    dxc[2] += dJ[0] * (-C.fx * iz2) + dJ[2] * (2.f * C.fx * xc[0] * iz3) + dJ[4] * (-C.fy * iz2) +
              dJ[5] * (2.f * C.fy * xc[1] * iz3);
    // x_c = W mu + t
    for (int j = 0; j < 3; j++) dm[j] += C.R[j] * dxc[0] + C.R[3 + j] * dxc[1] + C.R[6 + j] * dxc[2];
    for (int j = 0; j < 3; j++) a.d_means[3 * g + j] = dm[j];
    // Sigma = M M^T: dL/dM = 2 dSig M (dSig symmetric)
    float dM[9];
    for (int i = 0; i < 3; i++)
        for (int j = 0; j < 3; j++)
            dM[3 * i + j] = 2.f * (dSig[3 * i] * M[j] + dSig[3 * i + 1] * M[3 + j] + dSig[3 * i + 2] * M[6 + j]);
    // M = R diag(s)
    float dR[9];
    for (int i = 0; i < 3; i++)
        for (int j = 0; j < 3; j++) dR[3 * i + j] = dM[3 * i + j] * s[j];
    for (int j = 0; j < 3; j++)
        a.d_log_scales[3 * g + j] = (dM[j] * Rq[j] + dM[3 + j] * Rq[3 + j] + dM[6 + j] * Rq[6 + j]) * s[j];
    // R(w, x, y, z) of the unit quaternion
    const float dw = 2.f * (-zq * dR[1] + y * dR[2] + zq * dR[3] - x * dR[5] - y * dR[6] + x * dR[7]);
    const float dx = 2.f * (y * dR[1] + zq * dR[2] + y * dR[3] - 2.f * x * dR[4] - w * dR[5] + zq * dR[6] +
                            w * dR[7] - 2.f * x * dR[8]);
    const float dy = 2.f * (-2.f * y * dR[0] + x * dR[1] + w * dR[2] + x * dR[3] + zq * dR[5] - w * dR[6] +
                            zq * dR[7] - 2.f * y * dR[8]);
    const float dz = 2.f * (-2.f * zq * dR[0] - w * dR[1] + x * dR[2] + w * dR[3] - 2.f * zq * dR[4] + y * dR[5] +
                            x * dR[6] + y * dR[7]);
    // q^ = q / |q|: dL/dq = (dL/dq^ - (dL/dq^ . q^) q^) / |q|
    const float dd = dw * w + dx * x + dy * y + dz * zq;
    a.d_quats[4 * g] = (dw - dd * w) * iq;
    a.d_quats[4 * g + 1] = (dx - dd * x) * iq;
    a.d_quats[4 * g + 2] = (dy - dd * y) * iq;
    a.d_quats[4 * g + 3] = (dz - dd * zq) * iq;
}

// The block's SH coefficients (and then their gradients) pass through shared
// memory, so that global reads and writes of the 48 floats per Gaussian are
// coalesced across the block; one padding word per Gaussian keeps the
// per-thread rows (stride NC + 1) in distinct banks.
constexpr int kPreBwdThreads = 128;

template <int D>
__global__ void __launch_bounds__(kPreBwdThreads) preprocess_backward_kernel(const PreBwdArgs a) {
    grid_dependency_begin();
    constexpr int NK = (D + 1) * (D + 1);
    constexpr int NC = NK * 3, NS = NC + 1;
    __shared__ float s_sh[kPreBwdThreads * NS];
    const int64_t g0 = (int64_t)blockIdx.x * kPreBwdThreads;
    const int cnt = (int)(a.n - g0 < kPreBwdThreads ? a.n - g0 : kPreBwdThreads);
    for (int i = threadIdx.x; i < cnt * NC; i += kPreBwdThreads)
        s_sh[(i / NC) * NS + i % NC] = __ldg(a.sh + g0 * NC + i);
    __syncthreads();
    const int64_t g = g0 + threadIdx.x;
    float* row = s_sh + threadIdx.x * NS;
    if (threadIdx.x < cnt) gaussian_backward<D>(a, g, row);
    __syncthreads();
    for (int i = threadIdx.x; i < cnt * NC; i += kPreBwdThreads)
        a.d_sh[g0 * NC + i] = s_sh[(i / NC) * NS + i % NC];
}

}  // namespace

cudaError_t launch_rasterize_backward(const gs_projected& p, int64_t n, const uint32_t* sorted_vals,
                                      const uint32_t* ranges, const uint32_t* tile_order, const CamConst& cam,
                                      const float* final_T, const uint32_t* n_contrib, const float* grad_image,
                                      const gs_projected_grad& grad, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(grad.mean2d, 0, sizeof(float) * 2 * (size_t)n, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(grad.conic, 0, sizeof(float) * 3 * (size_t)n, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(grad.opacity, 0, sizeof(float) * (size_t)n, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(grad.rgb, 0, sizeof(float) * 3 * (size_t)n, s);
    if (e != cudaSuccess) return e;
    BwdArgs a;
    a.raster = reinterpret_cast<const float4*>(p.raster);
    a.order = tile_order;
    a.sorted_vals = sorted_vals;
    a.ranges = reinterpret_cast<const uint2*>(ranges);
    a.n = (uint32_t)n;
    a.width = cam.width;
    a.height = cam.height;
    a.tiles_x = cam.tiles_x;
    a.bg0 = cam.bg[0];
    a.bg1 = cam.bg[1];
    a.bg2 = cam.bg[2];
    a.final_T = final_T;
    a.n_contrib = n_contrib;
    a.grad_image = grad_image;
    a.g_mean2d = grad.mean2d;
    a.g_conic = grad.conic;
    a.g_opacity = grad.opacity;
    a.g_rgb = grad.rgb;
    const unsigned tiles = (unsigned)(cam.tiles_x * cam.tiles_y);
    launch_k(rasterize_backward_kernel, tiles, kBwdThreads, 0, s, a);
    return cudaGetLastError();
}

cudaError_t launch_preprocess_backward(const gs_gaussians& g, const CamConst& cam, const uint32_t* tiles_touched,
                                       const gs_projected_grad& gin, const gs_gaussians_grad& gout,
                                       cudaStream_t s) {
    if (g.n == 0) return cudaSuccess;
    PreBwdArgs a;
    a.means = g.means;
    a.quats = g.quats;
    a.log_scales = g.log_scales;
    a.logits = g.opacity_logits;
    a.sh = g.sh;
    a.tiles_touched = tiles_touched;
    a.n = g.n;
    a.cam = cam;
    a.g_mean2d = gin.mean2d;
    a.g_conic = gin.conic;
    a.g_opacity = gin.opacity;
    a.g_rgb = gin.rgb;
    a.d_means = gout.means;
    a.d_quats = gout.quats;
    a.d_log_scales = gout.log_scales;
    a.d_logits = gout.opacity_logits;
    a.d_sh = gout.sh;
    const unsigned blocks = (unsigned)((g.n + kPreBwdThreads - 1) / kPreBwdThreads);
    switch (g.sh_degree) {
        case 0: launch_k(preprocess_backward_kernel<0>, blocks, kPreBwdThreads, 0, s, a); break;
        case 1: launch_k(preprocess_backward_kernel<1>, blocks, kPreBwdThreads, 0, s, a); break;
        case 2: launch_k(preprocess_backward_kernel<2>, blocks, kPreBwdThreads, 0, s, a); break;
        default: launch_k(preprocess_backward_kernel<3>, blocks, kPreBwdThreads, 0, s, a); break;
    }
    return cudaGetLastError();
}

GS_DEFINE_CHECK_SETTER(backward)

}  // namespace gs
