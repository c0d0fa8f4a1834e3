// Step 4 ("Depth-sort per tile" and the tiles' lists, lesson page "3D Gaussian
// Splatting à partir de zéro", section "Rastérisation, non rayée"): each
// tile's list length, and from the lengths the tile ranges, computed from the
// Gaussians' tile rectangles alone. A stable sort of the (tile key, Gaussian)
// pairs puts tile t's pairs at [the sum of the lengths of the tiles whose key
// is smaller than t's, that plus t's length), so the ranges follow from the
// lengths without the sorted list; the frame computes them on a second stream
// while the sorts run.
//
//   tile_len_diff_kernel   : per block, a 2D difference array of the tile
//                            counts in shared memory (four updates per
//                            Gaussian rectangle), added to a global one.
//   tile_len_ranges_kernel : one block: the 2D prefix sums (the per-tile
//                            lengths), an exclusive scan in tile-key order,
//                            and the ranges, clamped to the key capacity.
#include <mutex>
#include <set>

#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kLenThreads = 512;
constexpr int kRangesThreads = 1024;

__global__ void __launch_bounds__(kLenThreads) tile_len_diff_kernel(const uint32_t* __restrict__ tiles_touched,
                                                                    const ushort4* __restrict__ rect, int64_t n,
                                                                    int tiles_x, int tiles_y,
                                                                    int* __restrict__ diff) {
    grid_dependency_begin();
    extern __shared__ int s_diff[];
    const int W = tiles_x + 1, cells = W * (tiles_y + 1);
    for (int i = threadIdx.x; i < cells; i += kLenThreads) s_diff[i] = 0;
    __syncthreads();
    const int64_t stride = (int64_t)gridDim.x * kLenThreads;
    for (int64_t g = (int64_t)blockIdx.x * kLenThreads + threadIdx.x; g < n; g += stride) {
        if (__ldg(tiles_touched + g) == 0u) continue;
        const ushort4 r = __ldg(rect + g);   // inclusive tile rectangle (x0, y0, x1, y1)
        GS_CHECK(r.z < tiles_x && r.w < tiles_y && r.x <= r.z && r.y <= r.w);
        if (r.z >= tiles_x || r.w >= tiles_y || r.x > r.z || r.y > r.w) continue;
        atomicAdd(&s_diff[r.y * W + r.x], 1);
        atomicAdd(&s_diff[r.y * W + r.z + 1], -1);
        atomicAdd(&s_diff[(r.w + 1) * W + r.x], -1);
        atomicAdd(&s_diff[(r.w + 1) * W + r.z + 1], 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < cells; i += kLenThreads)
        if (s_diff[i]) atomicAdd(&diff[i], s_diff[i]);
}

__global__ void __launch_bounds__(kRangesThreads) tile_len_ranges_kernel(const int* __restrict__ diff, int tiles_x,
                                                                         int tiles_y, const TileKeyMap km,
                                                                         int key_bits, int64_t cap,
                                                                         uint2* __restrict__ ranges) {
    grid_dependency_begin();
    extern __shared__ int s_len[];   // [tiles_y][tiles_x + 1]: the difference array, then the lengths
    __shared__ uint32_t s_warp[kRangesThreads / 32];
    __shared__ uint32_t s_carry;
    const int W = tiles_x + 1;
    for (int i = threadIdx.x; i < tiles_y * W; i += kRangesThreads) s_len[i] = diff[i];
    __syncthreads();
    // prefix along x within each row, then along y within each column
    for (int y = threadIdx.x; y < tiles_y; y += kRangesThreads) {
        int run = 0;
        for (int x = 0; x < tiles_x; x++) {
            run += s_len[y * W + x];
            s_len[y * W + x] = run;
        }
    }
    __syncthreads();
    for (int x = threadIdx.x; x < tiles_x; x += kRangesThreads) {
        int run = 0;
        for (int y = 0; y < tiles_y; y++) {
            run += s_len[y * W + x];
            s_len[y * W + x] = run;
        }
    }
    __syncthreads();
    // exclusive scan of the lengths in key order, kRangesThreads keys per round
    const uint32_t keys = 1u << key_bits;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (uint32_t k0 = 0; k0 < keys; k0 += kRangesThreads) {
        const uint32_t k = k0 + threadIdx.x;
        uint32_t t = 0xffffffffu, len = 0;
        if (k < keys) {
            t = tile_of_key(km, k);
            const uint32_t tx = t % (uint32_t)tiles_x, ty = t / (uint32_t)tiles_x;
            // a key whose tile lies outside the grid (the block layout has some) has no pairs
            if (ty < (uint32_t)tiles_y && tile_key(km, tx, ty) == k) len = (uint32_t)s_len[ty * W + tx];
            else t = 0xffffffffu;
        }
        uint32_t v = len;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31) s_warp[warp] = v;
        __syncthreads();
        if (warp == 0) {
            uint32_t w = s_warp[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t u = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += u;
            }
            s_warp[lane] = w;   // inclusive over the warps
        }
        __syncthreads();
        const uint32_t start = s_carry + (warp > 0 ? s_warp[warp - 1] : 0u) + v - len;
        if (t != 0xffffffffu && len > 0) {
            const uint64_t lo = start < (uint64_t)cap ? start : (uint64_t)cap;
            const uint64_t hi = (uint64_t)start + len < (uint64_t)cap ? (uint64_t)start + len : (uint64_t)cap;
            ranges[t] = make_uint2((uint32_t)lo, (uint32_t)hi);
        }
        __syncthreads();
        if (threadIdx.x == 0) s_carry += s_warp[31];
        __syncthreads();
    }
}

}  // namespace

bool tile_len_fits(int tiles_x, int tiles_y) {
    return (size_t)(tiles_x + 1) * (size_t)(tiles_y + 1) * sizeof(int) <= 96 * 1024;
}

size_t tile_len_diff_bytes(int tiles_x, int tiles_y) {
    return (size_t)(tiles_x + 1) * (size_t)(tiles_y + 1) * sizeof(int);
}

cudaError_t launch_tile_len_ranges(const uint32_t* tiles_touched, const uint16_t* rect, int64_t n, int tiles_x,
                                   int tiles_y, const TileKeyMap& km, int key_bits, int64_t cap, int* diff,
                                   uint32_t* ranges, cudaStream_t s) {
    const size_t diff_bytes = tile_len_diff_bytes(tiles_x, tiles_y);
    const size_t len_bytes = (size_t)(tiles_x + 1) * (size_t)tiles_y * sizeof(int);
    {
        // the kernels' shared-memory limit, raised once per device
        static std::mutex mu;
        static std::set<int> done;
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        std::lock_guard<std::mutex> lock(mu);
        if (!done.count(dev)) {
            e = cudaFuncSetAttribute(tile_len_diff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(tile_len_ranges_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         96 * 1024);
            if (e != cudaSuccess) return e;
            done.insert(dev);
        }
    }
    if (n > 0) {
        const int64_t want = (n + 16 * kLenThreads - 1) / (16 * kLenThreads);
        const unsigned blocks = (unsigned)(want < 74 ? (want < 1 ? 1 : want) : 74);
        launch_k(tile_len_diff_kernel, blocks, kLenThreads, diff_bytes, s, tiles_touched,
                 reinterpret_cast<const ushort4*>(rect), n, tiles_x, tiles_y, diff);
    }
    launch_k(tile_len_ranges_kernel, 1, kRangesThreads, len_bytes, s, static_cast<const int*>(diff), tiles_x,
             tiles_y, km, key_bits, cap, reinterpret_cast<uint2*>(ranges));
    return cudaGetLastError();
}

GS_DEFINE_CHECK_SETTER(tilelen)

}  // namespace gs
