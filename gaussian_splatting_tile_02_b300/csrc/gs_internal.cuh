// Internal declarations shared by the CUDA translation units of the renderer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "gs.h"

namespace gs {

constexpr int kTile = 16;

// Programmatic dependent launch. Every kernel is launched through launch_k,
// with the programmatic-serialisation attribute (unless switched off by
// gs_set_programmatic_launch): the launch of a kernel then overlaps the end of
// the kernel before it on the stream instead of following it. So every
// kernel begins with grid_dependency_begin(), before any global memory
// access: it returns once the preceding kernel has completed and its writes
// are visible. A kernel launched without the attribute (or after a memset or
// an event) finds it a no-op. No kernel signals its dependents early: an
// early signal let the next kernel's blocks take SM slots during the last
// wave, and graph-replayed 5M frames got 9% slower.
__device__ __forceinline__ void grid_dependency_begin() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

extern std::atomic<int> g_programmatic_launch;

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = g_programmatic_launch.load(std::memory_order_relaxed) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Status header at the start of every workspace (256 bytes reserved).
struct StatusHeader {
    uint32_t flags;          // GS_FLAG_*
    uint32_t timeout_site;   // which wait ran out (debug aid)
    unsigned long long num_keys;
    uint32_t pad[60];
};
static_assert(sizeof(StatusHeader) == 256, "status header is 256 bytes");

constexpr size_t kAlign = 256;
__host__ __device__ constexpr size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// Radix digits of a key_bits-bit key: ceil(key_bits / 8) LSD passes of 8-bit
// digits from the least significant end, the last one narrower (13 bits ->
// 8 + 5). The sort and the producers that count its digits share this layout.
__host__ __device__ inline int digit_passes(int key_bits) { return (key_bits + 7) / 8; }
__host__ __device__ inline int digit_width(int key_bits, int p) {
    return key_bits - 8 * p < 8 ? key_bits - 8 * p : 8;
}
__host__ __device__ inline int digit_shift(int key_bits, int p) {
    (void)key_bits;
    return 8 * p;
}

// The compositing exponent of one list entry at a lane's two pixels (x, y)
// and (x, y + 4), in tile-local coordinates:
//   log2(alpha) = log2 o - t1^2 - t2^2,  t1 = k1 (mx - x),  t2 = k3 (mx - x) + k2 (my - y).
// The terms are expanded around the tile origin, A1 = k1 mx and
// A2 = k3 mx + k2 my once per entry, so that each pixel pair costs seven
// FMAs; nx = -x and ny = -y are the lane's constants. Compositing (through
// the negated form below) and its backward both compute exactly these values,
// so they take the same per-entry decisions bit for bit.
__device__ __forceinline__ float2 entry_origin_terms(float mx, float my, float k1, float k2, float k3) {
    return make_float2(__fmul_rn(k1, mx), __fmaf_rn(k3, mx, __fmul_rn(k2, my)));
}
__device__ __forceinline__ void pixel_pair_exponents(float A1, float A2, float k1, float k2, float k3, float log2o,
                                                     float nx, float ny, float& t1, float& t2, float& t22,
                                                     float& e, float& e2) {
    t1 = __fmaf_rn(k1, nx, A1);
    t2 = __fmaf_rn(k3, nx, __fmaf_rn(k2, ny, A2));
    t22 = __fmaf_rn(-4.0f, k2, t2);   // y + 4
    const float e1 = __fmaf_rn(-t1, t1, log2o);
    e = __fmaf_rn(-t2, t2, e1);
    e2 = __fmaf_rn(-t22, t22, e1);
}
// The same exponents negated, -e and -e2, with the independent FMAs paired
// into packed two-wide ones: (t1, k2 ny + A2) in one, the two squares in
// another. Round-to-nearest is symmetric, so fma(t, t, -x) is exactly
// -fma(-t, t, x): every value here is the negation of the one above, bit for
// bit, and the decisions taken on it are the same. q = (A1, A2, k1, k2),
// nxy = (nx, ny).
__device__ __forceinline__ void pixel_pair_neg_exponents(const float4& q, float k3, float log2o, float2 nxy,
                                                         float& ne, float& ne2) {
    const float2 tu = __ffma2_rn(make_float2(q.z, q.w), nxy, make_float2(q.x, q.y));
    const float t2 = __fmaf_rn(k3, nxy.x, tu.y);
    const float t22 = __fmaf_rn(-4.0f, q.w, t2);
    const float ne1 = __fmaf_rn(tu.x, tu.x, -log2o);
    const float2 n = __ffma2_rn(make_float2(t2, t22), make_float2(t2, t22), make_float2(ne1, ne1));
    ne = n.x;
    ne2 = n.y;
}

// The key a (tile, Gaussian) pair is sorted by, for a tile (tx, ty). Identity
// (cbx == 0): the tile id ty * tiles_x + tx. Block layout: the low cbits bits
// number the block of 8 x kKeyBlockH tiles, (ty / kKeyBlockH) * cbx + tx / 8,
// and the bits above them the tile inside it, so the first radix pass sorts by
// block (a Gaussian's few tiles mostly share one) and the next by the tile
// within. Either way each tile's pairs are contiguous after a stable sort, in
// the same order; only the order of the tiles' lists differs.
#ifndef GS_KEY_BLOCK_H
#define GS_KEY_BLOCK_H 4
#endif
constexpr int kKeyBlockH = GS_KEY_BLOCK_H;   // 4 or 8
constexpr int kKeyFineBits = kKeyBlockH == 8 ? 6 : 5;
struct TileKeyMap {
    int tiles_x;
    int cbx;     // blocks per row, or 0 for the identity
    int cbits;   // bits of the block number
};
__host__ __device__ inline uint32_t tile_key(const TileKeyMap& m, uint32_t tx, uint32_t ty) {
    if (m.cbx == 0) return ty * (uint32_t)m.tiles_x + tx;
    const uint32_t fine = ((ty % (uint32_t)kKeyBlockH) << 3) | (tx & 7u);
    return (fine << m.cbits) | ((ty / (uint32_t)kKeyBlockH) * (uint32_t)m.cbx + (tx >> 3));
}
__host__ __device__ inline uint32_t tile_of_key(const TileKeyMap& m, uint32_t key) {
    if (m.cbx == 0) return key;
    const uint32_t block = key & ((1u << m.cbits) - 1u), fine = key >> m.cbits;
    const uint32_t tx = (block % (uint32_t)m.cbx) * 8u + (fine & 7u);
    const uint32_t ty = (block / (uint32_t)m.cbx) * (uint32_t)kKeyBlockH + (fine >> 3);
    return ty * (uint32_t)m.tiles_x + tx;
}
inline TileKeyMap identity_keys(int tiles_x_) { return TileKeyMap{tiles_x_, 0, 0}; }
inline TileKeyMap block_keys(int tiles_x_, int tiles_y_) {
    TileKeyMap m{tiles_x_, (tiles_x_ + 7) / 8, 0};
    const int blocks = m.cbx * ((tiles_y_ + kKeyBlockH - 1) / kKeyBlockH);
    while ((1 << m.cbits) < blocks) m.cbits++;
    if (m.cbits == 0) m.cbits = 1;
    return m;
}
inline int tile_key_bits(const TileKeyMap& m, int tiles) {
    if (m.cbx == 0) {
        int b = 0;
        while ((1 << b) < tiles) b++;
        return b > 0 ? b : 1;
    }
    return m.cbits + kKeyFineBits;
}

inline int tiles_x(const gs_camera& c) { return (c.width + kTile - 1) / kTile; }
inline int tiles_y(const gs_camera& c) { return (c.height + kTile - 1) / kTile; }

// Camera constants as passed by value to kernels.
struct CamConst {
    float R[9];
    float t[3];
    float fx, fy, cx, cy, near_z;
    int32_t width, height;
    int32_t tiles_x, tiles_y;
    float bg[3];
    float campos[3];   // camera centre in world space, -R^T t
};
CamConst make_cam_const(const gs_camera& c);

// ---------------------------------------------------------------- debug checks
// Built with -DGS_DEBUG_CHECKS (libgs_b300_debug.so), the kernels check their
// index invariants and count each failure into a caller-given device counter
// (gs_debug_set_check_counter); they never trap. The counter pointer lives in
// one __device__ variable per translation unit, set by that unit's setter.
#ifdef GS_DEBUG_CHECKS
static __device__ unsigned long long* g_check_counter = nullptr;
#define GS_CHECK(cond)                                                         \
    do {                                                                       \
        if (!(cond) && g_check_counter) atomicAdd(g_check_counter, 1ull);      \
    } while (0)
#define GS_DEFINE_CHECK_SETTER(unit)                                           \
    cudaError_t set_check_counter_##unit(unsigned long long* p) {              \
        return cudaMemcpyToSymbol(g_check_counter, &p, sizeof(p));             \
    }
#else
#define GS_CHECK(cond) \
    do {               \
    } while (0)
#define GS_DEFINE_CHECK_SETTER(unit) \
    cudaError_t set_check_counter_##unit(unsigned long long*) { return cudaSuccess; }
#endif
cudaError_t set_check_counter_preprocess(unsigned long long* p);
cudaError_t set_check_counter_binning(unsigned long long* p);
cudaError_t set_check_counter_sort(unsigned long long* p);
cudaError_t set_check_counter_rasterize(unsigned long long* p);
cudaError_t set_check_counter_backward(unsigned long long* p);
cudaError_t set_check_counter_splat2d(unsigned long long* p);
cudaError_t set_check_counter_densify(unsigned long long* p);

// Default bound of every device-side spin, in polling iterations.
extern long long g_spin_limit;

// ---------------------------------------------------------------- device helpers

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void raise_flag(StatusHeader* h, uint32_t flag, uint32_t site) {
    atomicOr(&h->flags, flag);
    if (flag == GS_FLAG_TIMEOUT) atomicMax(&h->timeout_site, site);
}

// ---------------------------------------------------------------- bulk copies
// One-dimensional bulk copies from global to shared memory (cp.async.bulk,
// the TMA unit's untiled form), completed on a shared-memory mbarrier that
// counts the bytes still to land. Source and destination 16-byte aligned, size
// a multiple of 16 bytes. The copies read this GPU's own memory only.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// makes an initialised barrier visible to the copy engine (then a __syncthreads)
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// orders this thread's earlier shared-memory accesses before later bulk copies into them
__device__ __forceinline__ void fence_proxy_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Bound on the wait for a bulk copy to land, in polls. A copy from valid global
// memory always lands, so this bound is fixed and generous (it is not the
// adjustable bound on waits for other blocks' progress): a block never leaves
// while its copies are in flight unless the copy engine has failed.
constexpr long long kBulkWaitLimit = 1ll << 24;
// Waits for the phase of the given parity to complete; false once `limit` polls ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit) {
    for (long long it = 0; it < limit; it++)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---------------------------------------------------------------- launchers

// preprocess.cu
// Depth-order sort input written by the projection step (nullable): keys
// (depth bits, or 0xffffffff without tiles), values (indices), and the keys'
// 8-bit digit histograms [4][256], accumulated (zeroed by the caller).
struct DepthKeysOut {
    uint32_t* keys;
    uint32_t* vals;
    uint32_t* hist;
};
// status (nullable): with a status header the parameters are staged through
// shared memory by bulk copies when their arrays allow it (16-byte aligned);
// a bulk copy that did not land within kBulkWaitLimit polls sets GS_FLAG_TIMEOUT.
cudaError_t launch_preprocess(const gs_gaussians& g, const CamConst& cam, const gs_projected& out, cudaStream_t s,
                              const DepthKeysOut* dk = nullptr, StatusHeader* status = nullptr);

// binning.cu
size_t bin_scratch_bytes(int64_t n);
cudaError_t launch_bin(const gs_projected& p, int64_t n, const CamConst& cam, uint32_t* offsets,
                       uint64_t* keys, uint32_t* vals, int64_t key_capacity, uint64_t* num_keys,
                       StatusHeader* status, void* scratch, cudaStream_t s);

// hist (nullable): digit histograms of the written keys for the radix sort
// that follows, key_bits significant bits (32-bit keys). Scratch:
// bin_ordered_scratch_bytes(n, key_capacity).
size_t bin_ordered_scratch_bytes(int64_t n, int64_t key_capacity);
cudaError_t launch_bin_ordered(const gs_projected& p, const uint32_t* order, int64_t n, const CamConst& cam,
                               uint32_t* offsets, uint32_t* tile_keys, uint32_t* vals, int64_t key_capacity,
                               uint64_t* num_keys, StatusHeader* status, void* scratch, cudaStream_t s,
                               uint32_t* hist = nullptr, int key_bits = 0, const TileKeyMap* keymap = nullptr);
cudaError_t launch_depth_keys(const gs_projected& p, int64_t n, uint32_t* keys, uint32_t* vals, uint32_t* hist,
                              cudaStream_t s);

// sort.cu
size_t sort_scratch_bytes(int64_t key_capacity);
// The scratch of one sort in two parts: the head (digit histograms, which the
// producer of the keys fills when hist_ready, and the passes' tile counters,
// which the bases kernel clears) and the look-back rows.
size_t sort_head_bytes();
size_t sort_lookback_bytes(int64_t key_capacity);
cudaError_t launch_sort32_split(uint32_t* keys, uint32_t* vals, uint32_t* keys_alt, uint32_t* vals_alt,
                                const uint64_t* num_keys, int64_t key_capacity, int key_bits, StatusHeader* status,
                                void* head, void* lookback, long long spin_limit, cudaStream_t s, bool hist_ready);
cudaError_t launch_sort(uint64_t* keys, uint32_t* vals, uint64_t* keys_alt, uint32_t* vals_alt,
                        const uint64_t* num_keys, int64_t key_capacity, int key_bits,
                        StatusHeader* status, void* scratch, long long spin_limit, cudaStream_t s);
// hist_ready: the producer of the keys already filled the digit histograms
// (sort_histogram_of(scratch), zeroed by sort_prepare_histogram) with
// sort_count_digits for every key
cudaError_t launch_sort32(uint32_t* keys, uint32_t* vals, uint32_t* keys_alt, uint32_t* vals_alt,
                          const uint64_t* num_keys, int64_t key_capacity, int key_bits,
                          StatusHeader* status, void* scratch, long long spin_limit, cudaStream_t s,
                          bool hist_ready = false);
uint32_t* sort_histogram_of(void* scratch);
cudaError_t sort_prepare_histogram(void* scratch, cudaStream_t s);
cudaError_t launch_tile_ranges(const uint64_t* sorted_keys, const uint64_t* num_keys,
                               int64_t key_capacity, int n_tiles, uint32_t* ranges, cudaStream_t s);
// ranges_zeroed: the caller cleared the ranges already (otherwise a memset does)
cudaError_t launch_tile_ranges32(const uint32_t* sorted_tiles, const uint64_t* num_keys,
                                 int64_t key_capacity, int n_tiles, uint32_t* ranges, cudaStream_t s,
                                 bool ranges_zeroed = false, const TileKeyMap* keymap = nullptr);
cudaError_t launch_spin_timeout_test(StatusHeader* status, long long iterations, cudaStream_t s);

// tiledepth.cu: each tile's list (Gaussians in index order, [ranges.x, ranges.y) of vals)
// sorted by (depth bits, index) in place, tiles in the given launch order (nullable).
// keys_a, keys_b, vals_b: scratch of the key capacity (lists longer than a block's
// shared-memory sort go through them); scratch: tile_depth_scratch_bytes(tiles).
// One kernel per list-size class that the key capacity allows.
// counts: three uint32 the caller has zeroed.
size_t tile_depth_scratch_bytes(int tiles);
cudaError_t launch_tile_depth_sort(const uint32_t* ranges, const uint32_t* tile_order, int tiles, const float* depth,
                                   int64_t n, int64_t key_capacity, uint32_t* vals, uint32_t* keys_a,
                                   uint32_t* keys_b, uint32_t* vals_b, uint32_t* counts, void* scratch,
                                   cudaStream_t s);
cudaError_t set_check_counter_tiledepth(unsigned long long* p);

// tilelen.cu: the tile ranges from the Gaussians' tile rectangles alone (each
// tile's list length by a 2D difference array, then an exclusive scan in
// tile-key order), for grids whose difference array fits in shared memory
// (tile_len_fits). diff: tile_len_diff_bytes, zeroed by the caller; ranges
// zeroed by the caller; ranges are clamped to cap.
bool tile_len_fits(int tiles_x, int tiles_y);
size_t tile_len_diff_bytes(int tiles_x, int tiles_y);
cudaError_t launch_tile_len_ranges(const uint32_t* tiles_touched, const uint16_t* rect, int64_t n, int tiles_x,
                                   int tiles_y, const TileKeyMap& km, int key_bits, int64_t cap, int* diff,
                                   uint32_t* ranges, cudaStream_t s);
cudaError_t set_check_counter_tilelen(unsigned long long* p);

// rasterize.cu
// 2D splats: their per-Gaussian record into p (depth, tiles_touched, rect, raster)
cudaError_t launch_preprocess2d(const float* means, const float* covs, const float* colours, const float* opacities,
                                const float* depths, int64_t n, int width, int height, const gs_projected& p,
                                cudaStream_t s);
cudaError_t launch_conic_to_cov_grad(const float* covs, const uint32_t* tiles_touched, const float* g_conic,
                                     int64_t n, float* g_covs, cudaStream_t s);

size_t densify_scratch_bytes(int64_t n);
cudaError_t launch_densify_stats(const float* grad_mean2d, const uint32_t* tiles_touched, int64_t n, float* accum,
                                 uint32_t* count, cudaStream_t s);
cudaError_t launch_densify(const gs_gaussians& in, const gs_gaussians_out& out, int64_t capacity, const float* accum,
                           const uint32_t* count, const float* xi, float grad_threshold, float log_scale_threshold,
                           float logit_threshold, uint8_t* action, uint64_t* out_count, void* scratch,
                           cudaStream_t s);

// at most this many views per batched preprocess launch
constexpr int kMaxBatchViews = 8;
// cams[views], outs[views]: one projected record per view
cudaError_t launch_preprocess_batch(const gs_gaussians& g, const CamConst* cams, const gs_projected* outs,
                                    const DepthKeysOut* dks, int views, cudaStream_t s);
cudaError_t launch_rasterize_backward(const gs_projected& p, int64_t n, const uint32_t* sorted_vals,
                                      const uint32_t* ranges, const uint32_t* tile_order, const CamConst& cam,
                                      const float* final_T, const uint32_t* n_contrib, const float* grad_image,
                                      const gs_projected_grad& grad, cudaStream_t s);
cudaError_t launch_preprocess_backward(const gs_gaussians& g, const CamConst& cam, const uint32_t* tiles_touched,
                                       const gs_projected_grad& gin, const gs_gaussians_grad& gout,
                                       cudaStream_t s);

// Heavy-first launch order of the tiles from their ranges: tile_order[tiles]
// receives a permutation of the tile indices, longest lists first.
cudaError_t launch_tile_order(const uint32_t* ranges, int tiles, uint32_t* tile_order, cudaStream_t s);
// The same order from many blocks, into scratch of tile_order_scratch_bytes(tiles)
// bytes (the order itself first, *tile_order points at it). done: a uint32 the
// caller has zeroed, or null (the scratch's own, cleared by a memset).
size_t tile_order_scratch_bytes(int tiles);
cudaError_t launch_tile_order_multi(const uint32_t* ranges, int tiles, void* scratch, uint32_t** tile_order,
                                    cudaStream_t s, uint32_t* done = nullptr);
// tile_order (nullable): a launch order written by launch_tile_order; null
// launches the tiles in index order (same image)
cudaError_t launch_rasterize(const gs_projected& p, int64_t n, const uint32_t* sorted_vals, const uint32_t* ranges,
                             const uint32_t* tile_order, const CamConst& cam, float* image, float* final_T,
                             uint32_t* n_contrib, cudaStream_t s);

}  // namespace gs
