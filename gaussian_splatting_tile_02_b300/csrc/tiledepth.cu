// Step 3 ("Depth-sort per tile", flowchart of the lesson page "3D Gaussian
// Splatting à partir de zéro", section "Rastérisation, non rayée") done tile
// by tile, for frames whose tile lists are short.
//
// In this order of the steps the frame is binned in Gaussian-index order and
// the (tile, Gaussian) pairs are stably sorted by tile, so each tile's list
// holds its Gaussians in index order. A stable sort of each list by depth bits
// then gives exactly the per-tile (depth bits, index) order of the stable sort
// of the (tile << 32 | depth bits) keys over the index-ordered list. Depth >
// near > 0 for every Gaussian with tiles, so the depth bits order like the
// depths.
//
// Each list is sorted by one block, in registers and shared memory: a stable
// LSD radix sort of its (depth bits, index) pairs by depth bits, four 8-bit
// passes, each ranked with warp match/popc counters (position order = list
// order) and scattered through shared memory. Blocks come in three sizes:
//   128 threads x 4 keys  (lists of up to 512 entries; one block per tile,
//                          launched heavy-first; it hands a longer list on)
//   256 threads x 8 keys  (up to 2,048)
//   1024 threads x 8 keys (up to 8,192)
// and a list longer than that is sorted by long_tile_sort_kernel: the same
// passes over chunks of 4096 entries through scratch arrays.
#include <map>
#include <mutex>

#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kRadixTD = 256;

// an index outside the scene can only come from a sort that was cut short
// (its status is flagged): read the depth of Gaussian 0 instead
__device__ __forceinline__ uint32_t depth_bits(const float* __restrict__ depth, uint32_t g, uint32_t n) {
    return __float_as_uint(__ldg(depth + (g < n ? g : 0u)));
}

__device__ __forceinline__ uint32_t lane_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Shared memory of a block sort of T threads x I keys.
template <int T, int I>
struct BlockSortSmem {
    uint16_t wh[(T / 32) * kRadixTD];   // per-warp digit counters -> offsets
    uint32_t dstart[kRadixTD];          // first slot of each digit in the staging
    uint32_t part[T / 32];              // block scan of the digit totals
    uint32_t any_bits, all_bits;        // OR and AND of the keys
    uint32_t keys[T * I];
    uint32_t vals[T * I];
};

// Stable sort by key of the first n_valid items held in registers. ie =
// ceil(n_valid / T) items per thread are used (a block-uniform count, so a
// short list keeps every warp busy and ranks no empty item rounds): item i of
// thread (warp, lane) sits at position warp * 32 ie + 32 i + lane. Passes
// whose 8-bit digit is the same for every key are skipped (a stable sort on a
// constant digit leaves the order as it is). On return the registers hold the
// sorted items in the same layout.
template <int T, int I>
__device__ __forceinline__ void block_sort_by_depth(uint32_t (&key)[I], uint32_t (&val)[I], int n_valid, int ie,
                                                    BlockSortSmem<T, I>& sm) {
    constexpr int W = T / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int warp_base = warp * (ie * 32);
    const uint32_t lt = lane_lt();
    uint16_t* wh = sm.wh + warp * kRadixTD;
    // which key bits differ anywhere in the list
    if (tid == 0) {
        sm.any_bits = 0u;
        sm.all_bits = 0xffffffffu;
    }
    __syncthreads();
    {
        uint32_t o = 0u, a = 0xffffffffu;
#pragma unroll
        for (int i = 0; i < I; i++)
            if (i < ie && warp_base + i * 32 + lane < n_valid) {
                o |= key[i];
                a &= key[i];
            }
        o = __reduce_or_sync(0xffffffffu, o);
        a = __reduce_and_sync(0xffffffffu, a);
        if (lane == 0) {
            atomicOr(&sm.any_bits, o);
            atomicAnd(&sm.all_bits, a);
        }
    }
    __syncthreads();
    const uint32_t varying = sm.any_bits ^ sm.all_bits;
#pragma unroll 1
    for (int shift = 0; shift < 32; shift += 8) {
        if (((varying >> shift) & 255u) == 0u) continue;   // block-uniform
        for (int i = tid; i < W * kRadixTD; i += T) sm.wh[i] = 0;
        __syncthreads();
        uint32_t rank[I];
#pragma unroll
        for (int i = 0; i < I; i++) {
            rank[i] = 0;
            if (i >= ie) continue;   // block-uniform
            const bool ok = warp_base + i * 32 + lane < n_valid;
            const uint32_t d = (key[i] >> shift) & 255u;
            const uint32_t peers = __match_any_sync(0xffffffffu, ok ? d : 0xffffu) & __ballot_sync(0xffffffffu, ok);
            const uint32_t below = __popc(peers & lt);
            uint32_t r = 0;
            if (ok) r = wh[d] + below;
            __syncwarp();
            if (ok && below == 0) wh[d] = (uint16_t)(r + __popc(peers));
            __syncwarp();
            rank[i] = r;
        }
        __syncthreads();
        // per digit: each warp's offset within the digit's run, and the run's length;
        // then the runs' starts (a scan over the 256 digits, kRadixTD / T per thread)
        constexpr int D = kRadixTD / T > 0 ? kRadixTD / T : 1;
        uint32_t tot[D];
        uint32_t mine = 0;
#pragma unroll
        for (int k = 0; k < D; k++) {
            const int d = tid * D + k;
            uint32_t sum = 0;
            if (d < kRadixTD) {
#pragma unroll
                for (int w = 0; w < W; w++) {
                    const uint32_t c = sm.wh[w * kRadixTD + d];
                    sm.wh[w * kRadixTD + d] = (uint16_t)sum;
                    sum += c;
                }
            }
            tot[k] = sum;
            mine += sum;
        }
        uint32_t v = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31) sm.part[warp] = v;
        __syncthreads();
        uint32_t run = v - mine;
        for (int w = 0; w < warp; w++) run += sm.part[w];
#pragma unroll
        for (int k = 0; k < D; k++) {
            const int d = tid * D + k;
            if (d < kRadixTD) sm.dstart[d] = run;
            run += tot[k];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < I; i++) {
            if (i < ie && warp_base + i * 32 + lane < n_valid) {
                const uint32_t d = (key[i] >> shift) & 255u;
                const uint32_t loc = sm.dstart[d] + sm.wh[warp * kRadixTD + d] + rank[i];
                sm.keys[loc] = key[i];
                sm.vals[loc] = val[i];
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < I; i++) {
            const int li = warp_base + i * 32 + lane;
            if (i < ie && li < n_valid) {
                key[i] = sm.keys[li];
                val[i] = sm.vals[li];
            }
        }
        __syncthreads();
    }
}

// A list of at most 32 entries, sorted by one warp: lane l holds entry l and
// its rank is the number of entries before it in (depth bits, position) order.
__device__ __forceinline__ void warp_sort_short_list(const uint2 r, uint32_t len, const float* __restrict__ depth,
                                                     uint32_t n, uint32_t* __restrict__ vals) {
    const int lane = threadIdx.x & 31;
    const bool ok = lane < (int)len;
    const uint32_t v = ok ? vals[r.x + lane] : 0u;
    const uint32_t k = ok ? depth_bits(depth, v, n) : 0xffffffffu;
    uint32_t rank = 0;
#pragma unroll 8
    for (int j = 0; j < 32; j++) {
        const uint32_t kj = __shfl_sync(0xffffffffu, k, j);
        rank += (j < (int)len) && (kj < k || (kj == k && j < lane));
    }
    __syncwarp();
    if (ok) vals[r.x + rank] = v;
}

// Tile lists handed from one block size to the next: count[0..2] the lengths
// of mid, big and huge (tile ids).
struct TileLists {
    uint32_t* count;
    uint32_t* mid;    // 512 < length <= 2048
    uint32_t* big;    // 2048 < length <= 8192
    uint32_t* huge;   // 8192 < length
};

template <int T, int I>
__device__ __forceinline__ void sort_tile_list(const uint2 r, uint32_t len, const float* __restrict__ depth,
                                               uint32_t n, uint32_t* __restrict__ vals, BlockSortSmem<T, I>& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ie = (int)((len + T - 1) / T);   // items per thread, 1..I
    const int warp_base = warp * (ie * 32);
    uint32_t key[I], val[I];
#pragma unroll
    for (int i = 0; i < I; i++) {
        const int li = warp_base + i * 32 + lane;
        const bool ok = i < ie && li < (int)len;
        val[i] = ok ? vals[r.x + li] : 0u;
        key[i] = ok ? depth_bits(depth, val[i], n) : 0xffffffffu;
    }
    block_sort_by_depth<T, I>(key, val, (int)len, ie, sm);
#pragma unroll
    for (int i = 0; i < I; i++) {
        const int li = warp_base + i * 32 + lane;
        if (i < ie && li < (int)len) vals[r.x + li] = val[i];
    }
}

// One block per tile (in the launch order): lists of up to 512 entries here,
// longer ones appended to the next size's list.
constexpr int kSmallT = 128, kSmallI = 4, kSmallCap = kSmallT * kSmallI;
constexpr int kMidT = 256, kMidI = 8, kMidCap = kMidT * kMidI;
constexpr int kBigT = 1024, kBigI = 8, kBigCap = kBigT * kBigI;

__global__ void __launch_bounds__(kSmallT) tile_sort_small_kernel(const uint2* __restrict__ ranges,
                                                                  const uint32_t* __restrict__ order,
                                                                  const float* __restrict__ depth, uint32_t n,
                                                                  uint32_t* __restrict__ vals, TileLists lists) {
    grid_dependency_begin();
    __shared__ BlockSortSmem<kSmallT, kSmallI> sm;
    const uint32_t tile = order ? order[blockIdx.x] : blockIdx.x;
    const uint2 r = ranges[tile];
    const uint32_t len = r.y > r.x ? r.y - r.x : 0u;
    if (len <= 1) return;
    if (len <= 32) {
        if (threadIdx.x < 32) warp_sort_short_list(r, len, depth, n, vals);
        return;
    }
    if (len > (uint32_t)kSmallCap) {
        if (threadIdx.x == 0) {
            const int c = len <= (uint32_t)kMidCap ? 0 : len <= (uint32_t)kBigCap ? 1 : 2;
            uint32_t* l = c == 0 ? lists.mid : c == 1 ? lists.big : lists.huge;
            l[atomicAdd(lists.count + c, 1u)] = tile;
        }
        return;
    }
    sort_tile_list<kSmallT, kSmallI>(r, len, depth, n, vals, sm);
}

template <int T, int I>
__global__ void __launch_bounds__(T, (T <= 256 ? 4 : 1)) tile_sort_list_kernel(const uint2* __restrict__ ranges,
                                                           const uint32_t* __restrict__ count_p,
                                                           const uint32_t* __restrict__ list,
                                                           const float* __restrict__ depth, uint32_t n,
                                                           uint32_t* __restrict__ vals) {
    grid_dependency_begin();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    auto& sm = *reinterpret_cast<BlockSortSmem<T, I>*>(smem_raw);
    const uint32_t count = *count_p;
    for (uint32_t q = blockIdx.x; q < count; q += gridDim.x) {
        const uint2 r = ranges[list[q]];
        sort_tile_list<T, I>(r, r.y - r.x, depth, n, vals, sm);
        __syncthreads();
    }
}

// Lists longer than kBigCap: the same four stable passes, chunk by chunk
// (4096 entries, in list order) through scratch arrays: (keys_a, vals) and
// (keys_b, vals_b), each used over the list's own range of [0, K).
constexpr int kLTThreads = 512, kLTItems = 8, kLTWarps = kLTThreads / 32, kLTChunk = kLTThreads * kLTItems;

__global__ void __launch_bounds__(kLTThreads) long_tile_sort_kernel(const uint2* __restrict__ ranges,
                                                                    const uint32_t* __restrict__ count_p,
                                                                    const uint32_t* __restrict__ list,
                                                                    const float* __restrict__ depth, uint32_t n,
                                                                    uint32_t* __restrict__ vals,
                                                                    uint32_t* __restrict__ keys_a,
                                                                    uint32_t* __restrict__ keys_b,
                                                                    uint32_t* __restrict__ vals_b) {
    grid_dependency_begin();
    __shared__ uint16_t s_wh[kLTWarps * kRadixTD];   // per-warp digit counters of a chunk
    __shared__ uint32_t s_off[kRadixTD];             // next output slot of each digit (list-relative)
    __shared__ uint32_t s_dstart[kRadixTD];          // a digit's first slot in the chunk's staging
    __shared__ uint32_t s_wt[kRadixTD / 32];
    __shared__ uint32_t s_ck[kLTChunk];
    __shared__ uint32_t s_cv[kLTChunk];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t lt = lane_lt();
    const uint32_t count = *count_p;
    for (uint32_t q = blockIdx.x; q < count; q += gridDim.x) {
        const uint2 r = ranges[list[q]];
        const uint32_t len = r.y - r.x;
        for (int p = 0; p < 4; p++) {
            const int shift = 8 * p;
            // p = 0: keys from the depths of vals; even p read (keys_a, vals), odd p (keys_b, vals_b)
            const uint32_t* kin = (p & 1) ? keys_b : keys_a;
            const uint32_t* vin = (p & 1) ? vals_b : vals;
            uint32_t* kout = (p & 1) ? keys_a : keys_b;
            uint32_t* vout = (p & 1) ? vals : vals_b;
            // the list's digit histogram (one atomic per group of equal digits in a warp),
            // scanned into the first slot of each digit
            if (tid < kRadixTD) s_off[tid] = 0;
            __syncthreads();
            for (uint32_t i0 = 0; i0 < len; i0 += kLTThreads) {
                const uint32_t i = i0 + tid;
                const bool ok = i < len;
                const uint32_t k = ok ? (p == 0 ? depth_bits(depth, vin[r.x + i], n) : kin[r.x + i]) : 0u;
                const uint32_t d = (k >> shift) & 255u;
                const uint32_t peers = __match_any_sync(0xffffffffu, ok ? d : 0xffffu) & __ballot_sync(0xffffffffu, ok);
                if (ok && (peers & lt) == 0) atomicAdd(&s_off[d], (uint32_t)__popc(peers));
            }
            __syncthreads();
            uint32_t c = 0, v = 0;
            if (tid < kRadixTD) {
                c = s_off[tid];
                v = c;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += u;
                }
                if (lane == 31) s_wt[warp] = v;
            }
            __syncthreads();
            if (tid < kRadixTD) {
                uint32_t before = v - c;
                for (int w = 0; w < warp; w++) before += s_wt[w];
                s_off[tid] = before;
            }
            __syncthreads();
            // chunks in list order, each ranked stably and scattered after the earlier chunks'
            for (uint32_t c0 = 0; c0 < len; c0 += kLTChunk) {
                const int n_valid = (int)(len - c0 < (uint32_t)kLTChunk ? len - c0 : (uint32_t)kLTChunk);
                for (int i = tid; i < kLTWarps * kRadixTD; i += kLTThreads) s_wh[i] = 0;
                const int warp_base = warp * (kLTItems * 32);
                uint32_t key[kLTItems], val[kLTItems], rank[kLTItems];
#pragma unroll
                for (int i = 0; i < kLTItems; i++) {
                    const int li = warp_base + i * 32 + lane;
                    val[i] = li < n_valid ? vin[r.x + c0 + li] : 0u;
                    key[i] = li < n_valid ? (p == 0 ? depth_bits(depth, val[i], n) : kin[r.x + c0 + li]) : 0u;
                }
                __syncthreads();
                uint16_t* wh = s_wh + warp * kRadixTD;
#pragma unroll
                for (int i = 0; i < kLTItems; i++) {
                    const int li = warp_base + i * 32 + lane;
                    const bool ok = li < n_valid;
                    const uint32_t d = (key[i] >> shift) & 255u;
                    const uint32_t peers =
                        __match_any_sync(0xffffffffu, ok ? d : 0xffffu) & __ballot_sync(0xffffffffu, ok);
                    uint32_t rk = 0;
                    if (ok) rk = wh[d] + __popc(peers & lt);
                    __syncwarp();
                    if (ok && (peers & lt) == 0) wh[d] = (uint16_t)(wh[d] + __popc(peers));
                    __syncwarp();
                    rank[i] = rk;
                }
                __syncthreads();
                uint32_t total = 0, sum = 0;
                if (tid < kRadixTD) {
#pragma unroll
                    for (int w = 0; w < kLTWarps; w++) {
                        const uint32_t x = s_wh[w * kRadixTD + tid];
                        s_wh[w * kRadixTD + tid] = (uint16_t)total;
                        total += x;
                    }
                    uint32_t y = total;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t u = __shfl_up_sync(0xffffffffu, y, o);
                        if (lane >= o) y += u;
                    }
                    if (lane == 31) s_wt[warp] = y;
                    sum = y - total;
                }
                __syncthreads();
                if (tid < kRadixTD) {
                    uint32_t add = 0;
                    for (int w = 0; w < warp; w++) add += s_wt[w];
                    s_dstart[tid] = sum + add;
                }
                __syncthreads();
#pragma unroll
                for (int i = 0; i < kLTItems; i++) {
                    const int li = warp_base + i * 32 + lane;
                    if (li < n_valid) {
                        const uint32_t d = (key[i] >> shift) & 255u;
                        const uint32_t loc = s_dstart[d] + s_wh[warp * kRadixTD + d] + rank[i];
                        s_ck[loc] = key[i];
                        s_cv[loc] = val[i];
                    }
                }
                __syncthreads();
                for (int j = tid; j < n_valid; j += kLTThreads) {
                    const uint32_t kk = s_ck[j];
                    const uint32_t d = (kk >> shift) & 255u;
                    const uint32_t o = s_off[d] + (uint32_t)j - s_dstart[d];
                    GS_CHECK(o < len);
                    if (o < len) {
                        kout[r.x + o] = kk;
                        vout[r.x + o] = s_cv[j];
                    }
                }
                __syncthreads();
                if (tid < kRadixTD) s_off[tid] += total;
                __syncthreads();
            }
        }
    }
}

// Grids of the list kernels: their resident blocks (dynamic shared memory allowed
// once per device).
struct ListGrids {
    unsigned mid, big;
};
cudaError_t list_grids(ListGrids* out) {
    static std::mutex mu;
    static std::map<int, ListGrids> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it == cache.end()) {
        int sms = 0, pm = 0, pb = 0;
        constexpr int mid_bytes = (int)sizeof(BlockSortSmem<kMidT, kMidI>);
        constexpr int big_bytes = (int)sizeof(BlockSortSmem<kBigT, kBigI>);
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tile_sort_list_kernel<kMidT, kMidI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     mid_bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tile_sort_list_kernel<kBigT, kBigI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     big_bytes);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&pm, tile_sort_list_kernel<kMidT, kMidI>, kMidT,
                                                              mid_bytes);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&pb, tile_sort_list_kernel<kBigT, kBigI>, kBigT,
                                                              big_bytes);
        if (e != cudaSuccess) return e;
        ListGrids g;
        g.mid = (unsigned)(sms * (pm > 0 ? pm : 1));
        g.big = (unsigned)(sms * (pb > 0 ? pb : 1));
        it = cache.emplace(dev, g).first;
    }
    *out = it->second;
    return cudaSuccess;
}

}  // namespace

size_t tile_depth_scratch_bytes(int tiles) { return 3 * align_up(4 * (size_t)(tiles > 0 ? tiles : 1)); }

cudaError_t launch_tile_depth_sort(const uint32_t* ranges, const uint32_t* tile_order, int tiles, const float* depth,
                                   int64_t n, int64_t key_capacity, uint32_t* vals, uint32_t* keys_a,
                                   uint32_t* keys_b, uint32_t* vals_b, uint32_t* counts, void* scratch,
                                   cudaStream_t s) {
    if (tiles <= 0 || n <= 0 || key_capacity <= 1) return cudaSuccess;
    char* w = static_cast<char*>(scratch);
    const size_t stride = align_up(4 * (size_t)tiles);
    TileLists lists;
    lists.count = counts;
    lists.mid = reinterpret_cast<uint32_t*>(w);
    lists.big = reinterpret_cast<uint32_t*>(w + stride);
    lists.huge = reinterpret_cast<uint32_t*>(w + 2 * stride);
    ListGrids grids;
    cudaError_t e = list_grids(&grids);
    if (e != cudaSuccess) return e;
    // no list is longer than the key capacity: the classes above it are not launched
    const uint2* r = reinterpret_cast<const uint2*>(ranges);
    const uint32_t un = (uint32_t)n;
    launch_k(tile_sort_small_kernel, (unsigned)tiles, kSmallT, 0, s, r, tile_order, depth, un, vals, lists);
    if (key_capacity > kSmallCap)
        launch_k(tile_sort_list_kernel<kMidT, kMidI>, grids.mid, kMidT, sizeof(BlockSortSmem<kMidT, kMidI>), s,
                 r, lists.count, lists.mid, depth, un, vals);
    if (key_capacity > kMidCap)
        launch_k(tile_sort_list_kernel<kBigT, kBigI>, grids.big, kBigT, sizeof(BlockSortSmem<kBigT, kBigI>), s,
                 r, lists.count + 1, lists.big, depth, un, vals);
    if (key_capacity > kBigCap)
        launch_k(long_tile_sort_kernel, 148, kLTThreads, 0, s, r, lists.count + 2, lists.huge, depth, un, vals, keys_a,
                 keys_b, vals_b);
    return cudaGetLastError();
}

GS_DEFINE_CHECK_SETTER(tiledepth)

}  // namespace gs
