// Step 5 of the forward renderer: front-to-back compositing per 16x16 tile.
//
// Method: lesson page "3D Gaussian Splatting à partir de zéro", section "La
// règle de composition alpha" (C = sum alpha_i T_i c_i, T_i = prod_{j<i}
// (1 - alpha_j), alpha_i = o_i exp(-0.5 d^T Sigma'^-1 d)) and "Étape 2"
// (rasterise_2d: integer pixel grid, alpha clamped at 0.99, front-to-back
// loop over the depth order). Contributions with alpha < 1/255 are skipped
// and a pixel stops once T < 1e-4, after the Gaussian that took it there.
//
// One 128-thread block per tile; warp w covers the 8x8 pixel block
// (8 (w & 1), 8 (w >> 1)) of the tile and each lane two of its pixels, (x, y)
// and (x, y + 4), which share the entry's loads, dx and the dx term of the
// quadratic form. The tile's sorted list is walked in batches of 128 entries,
// double-buffered in shared memory: while the block evaluates batch b, each
// thread already holds in registers the packed record (three float4 written by
// the projection step) of its entry of batch b + 1, and stores it to the other
// buffer afterwards, so the gathers overlap the arithmetic. For each group of
// 32 batch entries a warp ballots those whose alpha >= 1/255 box (part of the
// record) meets its 8x8 block, copies their records into a per-warp list and
// evaluates that list in order with a uniform loop: an entry whose box misses
// the block cannot contribute to any of its pixels, so skipping it changes no
// result. The block leaves the list once all its pixels are done.
//
// Coordinates are relative to the tile's first pixel: a centre enters as
// (u - x0) + residual (an exact subtraction, then one rounding at small
// magnitude), so the centre keeps ~1e-6 px where a binary32 centre near
// x = 1000 carries ~1e-4 px. The quadratic form is a sum of two squares,
// log2(alpha) = log2 o - (k1 dx)^2 - (k2 dy + k3 dx)^2, which keeps its
// accuracy for elongated footprints. Its linear terms are expanded around the
// tile origin once per batch entry (k1 mx and k3 mx + k2 my), so a lane's two
// pixels cost seven FMAs per entry and two compares; ex2 (MUFU pipe), the
// 0.99 cap and the blend only for the pairs past the 1/255 test.
#include <cuda_fp16.h>

#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kRastThreads = 128;   // 4 warps, each an 8x8 pixel block, two pixels per lane
constexpr float kLog2AlphaMin = -7.99435343685886f;   // log2(1/255)

// 2^x on the MUFU pipe (PTX ex2.approx; relative error about 2^-22).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Launch order of the tiles: longest lists first, bucketed by floor(log2
// length) (order within a bucket unspecified), so that the heaviest tiles
// start in the first wave instead of trailing the last one. One block: the
// tiles are counted into shared counters per (bucket, warp), one exclusive
// scan over those pairs in launch order (bucket descending, then warp) turns
// the counters into start positions, and a second round hands out each tile's
// position. Rows are kept in launch order: row clz(len) holds bucket
// 32 - clz(len), row 32 the empty tiles. Most tiles of a frame share one or
// two buckets, so a warp's lanes are first grouped by row with six ballots
// (the row's bits) and one lane per group updates the counter.
constexpr int kOrderThreads = 1024, kOrderItems = 8, kOrderRows = 33;

// lanes of the warp holding the same 6-bit value v (63 = none)
__device__ __forceinline__ uint32_t same_row_lanes(uint32_t v) {
    uint32_t m = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < 6; b++) {
        const uint32_t bit = (v >> b) & 1u;
        const uint32_t bal = __ballot_sync(0xffffffffu, bit);
        m &= bit ? bal : ~bal;
    }
    return m;
}

__global__ void __launch_bounds__(kOrderThreads) tile_order_kernel(const uint2* __restrict__ ranges, int tiles,
                                                                   uint32_t* __restrict__ order) {
    grid_dependency_begin();
    __shared__ uint32_t s_cnt[kOrderRows][32];   // [row][warp]
    __shared__ uint32_t s_row[kOrderRows];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    for (int i = threadIdx.x; i < kOrderRows * 32; i += kOrderThreads) s_cnt[i >> 5][i & 31] = 0;
    __syncthreads();
    auto row_of = [&](int t) -> uint32_t {
        if (t >= tiles) return 63u;
        const uint2 r = __ldg(ranges + t);
        const uint32_t len = r.y > r.x ? r.y - r.x : 0u;
        return len ? (uint32_t)__clz(len) : 32u;
    };
    constexpr int kChunk = kOrderItems * kOrderThreads;
    const bool one_chunk = tiles <= kChunk;
    uint32_t rw[kOrderItems];
    for (int t0 = 0; t0 < tiles; t0 += kChunk) {
#pragma unroll
        for (int i = 0; i < kOrderItems; i++) rw[i] = row_of(t0 + i * kOrderThreads + (int)threadIdx.x);
#pragma unroll
        for (int i = 0; i < kOrderItems; i++) {
            const uint32_t m = same_row_lanes(rw[i]);
            if (rw[i] != 63u && (m & lt) == 0) s_cnt[rw[i]][warp] += (uint32_t)__popc(m);
            __syncwarp();
        }
    }
    __syncthreads();
    // exclusive scan over (row, warp): warp w scans row w (warp 0 also row 32)
    for (int row = warp; row < kOrderRows; row += 32) {
        const uint32_t c = s_cnt[row][lane];
        uint32_t v = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        s_cnt[row][lane] = v - c;
        if (lane == 31) s_row[row] = v;
    }
    __syncthreads();
    for (int row = warp; row < kOrderRows; row += 32) {
        uint32_t before = 0;
        for (int k = lane; k < row; k += 32) before += s_row[k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
        s_cnt[row][lane] += before;
    }
    __syncthreads();
    for (int t0 = 0; t0 < tiles; t0 += kChunk) {
#pragma unroll
        for (int i = 0; i < kOrderItems; i++) {
            const int t = t0 + i * kOrderThreads + (int)threadIdx.x;
            const uint32_t r = one_chunk ? rw[i] : row_of(t);
            const uint32_t m = same_row_lanes(r);
            const int leader = __ffs(m) - 1;
            uint32_t base = 0;
            if (r != 63u && lane == leader) {
                base = s_cnt[r][warp];
                s_cnt[r][warp] = base + (uint32_t)__popc(m);
            }
            base = __shfl_sync(0xffffffffu, base, leader);
            if (r != 63u) order[base + __popc(m & lt)] = (uint32_t)t;
            __syncwarp();
        }
    }
}

// The same launch order from many blocks (the render path, where the frame's
// workspace has room for the table): one thread per tile.
//   tile_order_count_kernel  : per block, the tiles of each row (bucket); the
//                              last block to finish turns the [block][row]
//                              table into start positions, in launch order
//                              (row ascending, then block).
//   tile_order_scatter_kernel: each tile's position = its (block, row) start +
//                              the tiles of that row in earlier warps + its
//                              rank among its warp's lanes of the same row.
constexpr int kOrderMultiThreads = 256, kOrderMultiWarps = kOrderMultiThreads / 32;
// the last block scans the [block][row] table with at most kOrderMaxPer entries per
// thread: up to 24 * 256 / 33 = 186 blocks of 256 tiles (47,616 tiles; 3840x2160 has
// 32,400); larger grids use the one-block order
constexpr int kOrderMaxPer = 24;
constexpr int kOrderMaxBlocks = kOrderMaxPer * kOrderMultiThreads / kOrderRows;

__device__ __forceinline__ uint32_t tile_row(const uint2* __restrict__ ranges, int tiles, int t) {
    if (t >= tiles) return 63u;
    const uint2 r = __ldg(ranges + t);
    const uint32_t len = r.y > r.x ? r.y - r.x : 0u;
    return len ? (uint32_t)__clz(len) : 32u;
}

__global__ void __launch_bounds__(kOrderMultiThreads) tile_order_count_kernel(const uint2* __restrict__ ranges,
                                                                              int tiles, uint32_t* __restrict__ table,
                                                                              uint32_t* __restrict__ done) {
    grid_dependency_begin();
    __shared__ uint32_t s_cnt[kOrderRows][kOrderMultiWarps];
    __shared__ uint32_t s_wt[kOrderMultiWarps];
    __shared__ bool s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kOrderRows * kOrderMultiWarps; i += kOrderMultiThreads)
        s_cnt[i / kOrderMultiWarps][i % kOrderMultiWarps] = 0;
    __syncthreads();
    const uint32_t row = tile_row(ranges, tiles, blockIdx.x * kOrderMultiThreads + tid);
    const uint32_t m = same_row_lanes(row);
    if (row != 63u && (m & ((1u << lane) - 1u)) == 0) s_cnt[row][warp] = (uint32_t)__popc(m);
    __syncthreads();
    const int nb = gridDim.x;
    if (tid < kOrderRows) {
        uint32_t t = 0;
#pragma unroll
        for (int w = 0; w < kOrderMultiWarps; w++) t += s_cnt[tid][w];
        table[blockIdx.x * kOrderRows + tid] = t;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(done, 1u) == (uint32_t)nb - 1u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // exclusive scan over f = row * nb + block (launch order) of the table: each thread
    // takes a run of `per` consecutive f (its loads all issued at once), then one block scan
    const int total = kOrderRows * nb;
    const int per = (total + kOrderMultiThreads - 1) / kOrderMultiThreads;
    // (launch_tile_order_multi keeps total within kOrderMaxPer runs per thread)
    uint32_t x[kOrderMaxPer];
    uint32_t sum = 0;
    const int f0 = tid * per;
#pragma unroll
    for (int k = 0; k < kOrderMaxPer; k++) {
        const int f = f0 + k;
        x[k] = (k < per && f < total) ? ld_volatile_u32(table + (f % nb) * kOrderRows + f / nb) : 0u;
        sum += x[k];
    }
    uint32_t v = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) s_wt[warp] = v;
    __syncthreads();
    uint32_t run = v - sum;
    for (int w = 0; w < warp; w++) run += s_wt[w];
#pragma unroll
    for (int k = 0; k < kOrderMaxPer; k++) {
        const int f = f0 + k;
        if (k < per && f < total) {
            table[(f % nb) * kOrderRows + f / nb] = run;
            run += x[k];
        }
    }
}

__global__ void __launch_bounds__(kOrderMultiThreads) tile_order_scatter_kernel(const uint2* __restrict__ ranges,
                                                                                int tiles,
                                                                                const uint32_t* __restrict__ table,
                                                                                uint32_t* __restrict__ order) {
    grid_dependency_begin();
    __shared__ uint32_t s_cnt[kOrderRows][kOrderMultiWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kOrderRows * kOrderMultiWarps; i += kOrderMultiThreads)
        s_cnt[i / kOrderMultiWarps][i % kOrderMultiWarps] = 0;
    __syncthreads();
    const int t = blockIdx.x * kOrderMultiThreads + tid;
    const uint32_t row = tile_row(ranges, tiles, t);
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t m = same_row_lanes(row);
    if (row != 63u && (m & lt) == 0) s_cnt[row][warp] = (uint32_t)__popc(m);
    __syncthreads();
    if (row == 63u) return;
    uint32_t pos = table[blockIdx.x * kOrderRows + row] + (uint32_t)__popc(m & lt);
    for (int w = 0; w < warp; w++) pos += s_cnt[row][w];
    order[pos] = (uint32_t)t;
}

struct RastArgs {
    const float4* raster;   // [n][3]
    const uint32_t* order;  // launch order of the tiles, or null for index order
    const uint32_t* sorted_vals;
    const uint2* ranges;
    uint32_t n;
    int width, height, tiles_x;
    float bg0, bg1, bg2;
    float* image;
    float* final_T;
    uint32_t* n_contrib;
};

// kAux: the per-pixel list position of the last contributor is tracked (for
// n_contrib); without it the blend is the same arithmetic minus that bookkeeping.
template <bool kAux>
__global__ void __launch_bounds__(kRastThreads, 8) rasterize_kernel(const RastArgs a) {
    grid_dependency_begin();
    __shared__ float4 s_q[2][kRastThreads];    // (A1, A2, k1, k2): origin terms of the exponent
    __shared__ float4 s_r[2][kRastThreads];    // (k3, log2 o, r, g)
    __shared__ float s_b[2][kRastThreads];     // b
    __shared__ float4 s_box[2][kRastThreads];  // (x lo, x hi, y lo, y hi), tile-local
    __shared__ float4 w_q[kRastThreads / 32][32];   // per-warp list of the entries that meet its block
    __shared__ float4 w_r[kRastThreads / 32][32];
    __shared__ float2 w_bj[kRastThreads / 32][32];  // (b, list position + 1 as bits)

    const int tile = a.order ? (int)a.order[blockIdx.x] : (int)blockIdx.x;
    GS_CHECK(tile >= 0 && tile < (int)gridDim.x);
    const int tx = tile % a.tiles_x, ty = tile / a.tiles_x;
    const float tile_x0 = (float)(tx * kTile), tile_y0 = (float)(ty * kTile);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int lbx0 = 8 * (warp & 1), lby0 = 8 * (warp >> 1);   // warp's 8x8 block, tile-local
    // the lane's two pixels: (lx, ly) and (lx, ly + 4)
    const int lx = lbx0 + (lane & 7), ly = lby0 + (lane >> 3);
    const int px = tx * kTile + lx, py = ty * kTile + ly;
    const float fbx0 = (float)lbx0, fbx1 = (float)(lbx0 + 7), fby0 = (float)lby0, fby1 = (float)(lby0 + 7);
    const uint2 range0 = a.ranges[tile];
    // a range with end < start can only come from a sort that was cut short
    // (its status is flagged): treat it as empty, never read past the list
    GS_CHECK(range0.y >= range0.x);
    const uint2 range = make_uint2(range0.x, max(range0.x, range0.y));
    const float2 nxy = make_float2(-(float)lx, -(float)ly);

    float T = 1.0f, C0 = 0.0f, C1 = 0.0f, C2 = 0.0f;
    float U = 1.0f, D0 = 0.0f, D1 = 0.0f, D2 = 0.0f;   // second pixel
    uint32_t last = 0, last2 = 0;
    bool done = !(px < a.width && py < a.height);
    bool done2 = !(px < a.width && py + 4 < a.height);

    auto fetch = [&](uint32_t idx, float4& r0, float4& r1, float4& r2) {
        uint32_t g = __ldg(a.sorted_vals + idx);
        // an index outside the scene can only come from a sort that was cut
        // short (its status is flagged); never read past the arrays
        GS_CHECK(g < a.n);
        if (g >= a.n) g = 0;
        r0 = __ldg(a.raster + 3 * g);
        r1 = __ldg(a.raster + 3 * g + 1);
        r2 = __ldg(a.raster + 3 * g + 2);
    };
    auto store = [&](int buf, const float4& r0, const float4& r1, const float4& r2) {
        const float mx = (r0.x - tile_x0) + r0.z, my = (r0.y - tile_y0) + r0.w;
        const uint32_t hb = __float_as_uint(r2.w);
        const __half2 h = *reinterpret_cast<const __half2*>(&hb);
        const float hx = __low2float(h), hy = __high2float(h);
        const float2 A = entry_origin_terms(mx, my, r1.x, r1.y, r1.z);
        s_q[buf][threadIdx.x] = make_float4(A.x, A.y, r1.x, r1.y);   // (A1, A2, k1, k2)
        s_r[buf][threadIdx.x] = make_float4(r1.z, r1.w, r2.x, r2.y);   // (k3, log2 o, r, g)
        s_b[buf][threadIdx.x] = r2.z;
        s_box[buf][threadIdx.x] = make_float4(mx - hx, mx + hx, my - hy, my + hy);
    };

    const uint32_t len = range.y - range.x;
    const uint32_t nbatch = (len + kRastThreads - 1) / kRastThreads;
    if (threadIdx.x < len) {
        float4 r0, r1, r2;
        fetch(range.x + threadIdx.x, r0, r1, r2);
        store(0, r0, r1, r2);
    }
    __syncthreads();

    for (uint32_t b = 0; b < nbatch; b++) {
        const int buf = b & 1;
        const uint32_t base = range.x + b * kRastThreads;
        // gather the next batch's record now; it is stored after the arithmetic
        const uint32_t nidx = base + kRastThreads + threadIdx.x;
        const bool have_next = b + 1 < nbatch && nidx < range.y;
        float4 n0, n1, n2;
        if (have_next) fetch(nidx, n0, n1, n2);

        const uint32_t cnt = min((uint32_t)kRastThreads, range.y - base);
        // groups of 32 batch entries: ballot the ones whose box meets this
        // warp's 8x8 pixel block, copy those records into the warp's list, then
        // evaluate the list in order for the warp's 64 pixels
#pragma unroll 1
        for (int i = 0; i < kRastThreads / 32; i++) {
            if (__all_sync(0xffffffffu, done && done2)) break;
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
                if constexpr (kAux)
                    w_bj[warp][pos] = make_float2(s_b[buf][j], __uint_as_float(base - range.x + j + 1));
                else
                    w_bj[warp][pos].x = s_b[buf][j];
            }
            __syncwarp();
            const int nh = __popc(m);
#pragma unroll 4
            for (int k = 0; k < nh; k++) {
                const float4 q = w_q[warp][k];
                const float4 r = w_r[warp][k];
                float ne, ne2;   // the exponents negated
                pixel_pair_neg_exponents(q, r.x, r.y, nxy, ne, ne2);
                // alpha = min(0.99, 2^e) < 1/255 is e < log2(1/255) (the same
                // decision in exact arithmetic; ex2 is only evaluated past it)
                const bool c = !done && ne <= -kLog2AlphaMin, c2 = !done2 && ne2 <= -kLog2AlphaMin;
                if (!(c || c2)) continue;
                float2 bj;
                if constexpr (kAux)
                    bj = w_bj[warp][k];
                else
                    bj.x = w_bj[warp][k].x;
                if (c) {
                    const float alpha = fminf(0.99f, fast_exp2(-ne));
                    const float w = alpha * T;
                    C0 += w * r.z;
                    C1 += w * r.w;
                    C2 += w * bj.x;
                    T -= w;
                    if constexpr (kAux) last = __float_as_uint(bj.y);
                    if (T < 1e-4f) done = true;
                }
                if (c2) {
                    const float alpha = fminf(0.99f, fast_exp2(-ne2));
                    const float w = alpha * U;
                    D0 += w * r.z;
                    D1 += w * r.w;
                    D2 += w * bj.x;
                    U -= w;
                    if constexpr (kAux) last2 = __float_as_uint(bj.y);
                    if (U < 1e-4f) done2 = true;
                }
            }
            __syncwarp();
        }
        if (have_next) store(buf ^ 1, n0, n1, n2);
        if (__syncthreads_count(done && done2) == kRastThreads) break;
    }
    if (px < a.width && py < a.height) {
        const int64_t p = (int64_t)py * a.width + px;
        a.image[3 * p] = C0 + T * a.bg0;
        a.image[3 * p + 1] = C1 + T * a.bg1;
        a.image[3 * p + 2] = C2 + T * a.bg2;
        if (a.final_T) a.final_T[p] = T;
        if (kAux && a.n_contrib) a.n_contrib[p] = last;
    }
    if (px < a.width && py + 4 < a.height) {
        const int64_t p = (int64_t)(py + 4) * a.width + px;
        a.image[3 * p] = D0 + U * a.bg0;
        a.image[3 * p + 1] = D1 + U * a.bg1;
        a.image[3 * p + 2] = D2 + U * a.bg2;
        if (a.final_T) a.final_T[p] = U;
        if (kAux && a.n_contrib) a.n_contrib[p] = last2;
    }
}

}  // namespace

cudaError_t launch_rasterize(const gs_projected& p, int64_t n, const uint32_t* sorted_vals, const uint32_t* ranges,
                             const uint32_t* tile_order, const CamConst& cam, float* image, float* final_T,
                             uint32_t* n_contrib, cudaStream_t s) {
    RastArgs a;
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
    a.image = image;
    a.final_T = final_T;
    a.n_contrib = n_contrib;
    const unsigned tiles = (unsigned)(cam.tiles_x * cam.tiles_y);
    if (n == 0) a.sorted_vals = nullptr;
    if (n_contrib)
        launch_k(rasterize_kernel<true>, tiles, kRastThreads, 0, s, a);
    else
        launch_k(rasterize_kernel<false>, tiles, kRastThreads, 0, s, a);
    return cudaGetLastError();
}

size_t tile_order_scratch_bytes(int tiles) {
    const size_t nb = (size_t)(tiles + kOrderMultiThreads - 1) / kOrderMultiThreads;
    return align_up(4 * (size_t)tiles) + align_up(4 * kOrderRows * nb) + align_up(4);
}

cudaError_t launch_tile_order_multi(const uint32_t* ranges, int tiles, void* scratch, uint32_t** tile_order,
                                    cudaStream_t s, uint32_t* done_zeroed) {
    char* w = static_cast<char*>(scratch);
    uint32_t* order = reinterpret_cast<uint32_t*>(w);
    const size_t nb = (size_t)(tiles + kOrderMultiThreads - 1) / kOrderMultiThreads;
    uint32_t* table = reinterpret_cast<uint32_t*>(w + align_up(4 * (size_t)tiles));
    uint32_t* done = reinterpret_cast<uint32_t*>(w + align_up(4 * (size_t)tiles) + align_up(4 * kOrderRows * nb));
    *tile_order = order;
    if (tiles <= 0) return cudaSuccess;
    if (nb > (size_t)kOrderMaxBlocks) return launch_tile_order(ranges, tiles, order, s);
    if (done_zeroed) {
        done = done_zeroed;
    } else {
        const cudaError_t e = cudaMemsetAsync(done, 0, sizeof(uint32_t), s);
        if (e != cudaSuccess) return e;
    }
    const uint2* r = reinterpret_cast<const uint2*>(ranges);
    launch_k(tile_order_count_kernel, (unsigned)nb, kOrderMultiThreads, 0, s, r, tiles, table, done);
    launch_k(tile_order_scatter_kernel, (unsigned)nb, kOrderMultiThreads, 0, s, r, tiles, table, order);
    return cudaGetLastError();
}

cudaError_t launch_tile_order(const uint32_t* ranges, int tiles, uint32_t* tile_order, cudaStream_t s) {
    launch_k(tile_order_kernel, 1, kOrderThreads, 0, s, reinterpret_cast<const uint2*>(ranges), tiles, tile_order);
    return cudaGetLastError();
}

GS_DEFINE_CHECK_SETTER(rasterize)

}  // namespace gs
