// Step 3 (flowchart box "Depth-sort per tile" on the lesson page "3D Gaussian
// Splatting à partir de zéro") and step 4 (per-tile ranges).
//
// Stable least-significant-digit radix sort of (uint64 key, uint32 value)
// pairs with 8-bit digits. Sorting the binning keys (tile id in the high
// word, depth bits in the low word) orders each tile's entries by depth, with
// equal keys kept in Gaussian-index order.
//
//   sort_histogram : one read of all keys; 256-bin histograms of every digit
//                    position at once (shared-memory counters, then global
//                    atomics). Also clears the look-back status rows.
//   sort_bases     : exclusive scan of each histogram -> digit base offsets.
//   onesweep pass  : one kernel per digit. Each block takes the next 4096-key
//                    tile (tile ids from an atomic counter, so a block only
//                    ever waits on blocks that are already running), ranks its
//                    keys stably with warp match/popc counters, publishes its
//                    per-digit counts, and finds its global offsets by
//                    decoupled look-back over earlier tiles. Keys are then
//                    reordered in shared memory and written out in
//                    digit-contiguous runs (coalesced), values likewise.
//   copy back      : only when the pass count is odd.
//
// Every wait in the look-back is bounded (polling iterations, with backoff);
// a wait that runs out sets GS_FLAG_TIMEOUT in the workspace header and the
// block still publishes a status so that no other block waits on it. All
// stores are bounds-checked against the key count.
#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortItems = 16;
constexpr int kSortTile = kSortThreads * kSortItems;  // 4096 keys per tile
constexpr int kRadix = 256;
constexpr int kMaxPasses = 8;
constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagIncl = 2u << 30;
constexpr uint32_t kValueMask = (1u << 30) - 1u;

struct SortScratch {
    uint32_t* hist;      // [kMaxPasses][256], becomes the digit bases
    uint32_t* counters;  // [kMaxPasses] tile-id counters
    uint32_t* lookback;  // [2][max_tiles][256]
    int64_t max_tiles;
};

__host__ __device__ inline int64_t sort_max_tiles(int64_t cap) { return (cap + kSortTile - 1) / kSortTile; }

SortScratch carve(void* scratch, int64_t cap) {
    SortScratch s;
    char* p = static_cast<char*>(scratch);
    s.hist = reinterpret_cast<uint32_t*>(p);
    p += align_up(sizeof(uint32_t) * kMaxPasses * kRadix);
    s.counters = reinterpret_cast<uint32_t*>(p);
    p += align_up(sizeof(uint32_t) * kMaxPasses);
    s.lookback = reinterpret_cast<uint32_t*>(p);
    s.max_tiles = sort_max_tiles(cap > 0 ? cap : 1);
    return s;
}

__device__ __forceinline__ int64_t key_count(const uint64_t* num_keys, int64_t cap) {
    const unsigned long long k = *num_keys;
    return k < (unsigned long long)cap ? (int64_t)k : cap;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Polls *p until a status flag is present. Returns false if the bound ran out
// or another block already reported a timeout.
__device__ bool bounded_wait(const uint32_t* p, uint32_t& v, long long limit, const StatusHeader* h) {
    long long it = 0;
    while (true) {
        v = ld_acquire_u32(p);
        if (v & (kFlagAgg | kFlagIncl)) return true;
        if (++it > limit) return false;
        if ((it & 31) == 0 && (ld_volatile_u32(&h->flags) & GS_FLAG_TIMEOUT)) return false;
        __nanosleep(it < 32 ? 32 : 256);
    }
}

__global__ void __launch_bounds__(kSortThreads) sort_histogram_kernel(const uint64_t* __restrict__ keys,
                                                                      const uint64_t* __restrict__ num_keys,
                                                                      int64_t cap, int passes, int key_bits,
                                                                      uint32_t* __restrict__ hist,
                                                                      uint32_t* __restrict__ lookback,
                                                                      int64_t max_tiles) {
    __shared__ uint32_t s_hist[kMaxPasses * kRadix];
    for (int i = threadIdx.x; i < passes * kRadix; i += kSortThreads) s_hist[i] = 0;
    __syncthreads();
    const int64_t K = key_count(num_keys, cap);
    const int64_t stride = (int64_t)gridDim.x * kSortThreads;
    for (int64_t i = (int64_t)blockIdx.x * kSortThreads + threadIdx.x; i < K; i += stride) {
        const uint64_t k = keys[i];
        for (int p = 0; p < passes; p++) {
            const int w = key_bits - 8 * p < 8 ? key_bits - 8 * p : 8;
            const uint32_t d = (uint32_t)(k >> (8 * p)) & ((1u << w) - 1u);
            atomicAdd(&s_hist[p * kRadix + d], 1u);
        }
    }
    // clear the look-back rows this sort will use (both ping-pong arrays)
    const int64_t tiles = (K + kSortTile - 1) / kSortTile;
    for (int64_t i = (int64_t)blockIdx.x * kSortThreads + threadIdx.x; i < tiles * kRadix; i += stride) {
        lookback[i] = 0;
        lookback[max_tiles * kRadix + i] = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < passes * kRadix; i += kSortThreads)
        if (s_hist[i]) atomicAdd(&hist[i], s_hist[i]);
}

__global__ void __launch_bounds__(kRadix) sort_bases_kernel(uint32_t* __restrict__ hist) {
    __shared__ uint32_t warp_tot[kRadix / 32];
    uint32_t* h = hist + blockIdx.x * kRadix;
    const uint32_t x = h[threadIdx.x];
    uint32_t v = x;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[wid] = v;
    __syncthreads();
    uint32_t add = 0;
    for (int w = 0; w < wid; w++) add += warp_tot[w];
    h[threadIdx.x] = v + add - x;
}

struct PassArgs {
    const uint64_t* keys_in;
    const uint32_t* vals_in;
    uint64_t* keys_out;
    uint32_t* vals_out;
    const uint64_t* num_keys;
    int64_t cap;
    int pass;
    int digit_bits;
    const uint32_t* bases;    // [256] for this pass
    uint32_t* counter;        // tile-id counter for this pass
    uint32_t* status;         // look-back rows of this pass
    uint32_t* status_clear;   // rows of the other array, cleared for the pass after next
    StatusHeader* header;
    long long spin_limit;
};

__global__ void __launch_bounds__(kSortThreads) onesweep_kernel(const PassArgs a) {
    __shared__ uint32_t s_hist[kSortWarps * kRadix];  // per-warp digit counters -> offsets
    __shared__ uint32_t s_dstart[kRadix];
    __shared__ uint32_t s_goff[kRadix];
    __shared__ uint32_t s_warp_tot[kSortWarps];
    __shared__ __align__(16) uint64_t s_keys[kSortTile];
    __shared__ uint32_t s_tile;
    __shared__ int s_timed_out;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_tile = atomicAdd(a.counter, 1u);
        s_timed_out = 0;
    }
    for (int i = tid; i < kSortWarps * kRadix; i += kSortThreads) s_hist[i] = 0;
    __syncthreads();
    const int64_t K = key_count(a.num_keys, a.cap);
    const uint32_t tile = s_tile;
    const int64_t start = (int64_t)tile * kSortTile;
    if (start >= K) return;
    const int n_valid = (int)(K - start < kSortTile ? K - start : kSortTile);
    if (a.status_clear) {
        // rows used by the previous pass are not read again until two passes on
        a.status_clear[(int64_t)tile * kRadix + tid] = 0;
    }

    const int shift = 8 * a.pass;
    const uint32_t dmask = (1u << a.digit_bits) - 1u;
    const int warp_base = warp * (kSortItems * 32);
    uint64_t key[kSortItems];
#pragma unroll
    for (int i = 0; i < kSortItems; i++) {
        const int li = warp_base + i * 32 + lane;
        key[i] = li < n_valid ? a.keys_in[start + li] : 0ull;
    }

    // stable rank within the warp: position order is (i, lane)
    uint32_t* wh = s_hist + warp * kRadix;
    const uint32_t lt = lanemask_lt();
    uint16_t rank[kSortItems];
#pragma unroll
    for (int i = 0; i < kSortItems; i++) {
        const int li = warp_base + i * 32 + lane;
        const bool v = li < n_valid;
        const uint32_t d = v ? ((uint32_t)(key[i] >> shift) & dmask) : 0xffffu;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        uint32_t r = 0;
        if (v) r = wh[d] + __popc(peers & lt);
        __syncwarp();
        if (v && (peers & lt) == 0) wh[d] += __popc(peers);
        __syncwarp();
        rank[i] = (uint16_t)r;
    }
    __syncthreads();

    // per digit (thread = digit): offsets of each warp inside the block
    {
        const int d = tid;
        uint32_t sum = 0;
#pragma unroll
        for (int w = 0; w < kSortWarps; w++) {
            const uint32_t c = s_hist[w * kRadix + d];
            s_hist[w * kRadix + d] = sum;
            sum += c;
        }
        // publish this tile's count, then look back over earlier tiles
        uint32_t* row = a.status + (int64_t)tile * kRadix;
        if (tile == 0) {
            st_release_u32(row + d, kFlagIncl | sum);
            s_goff[d] = a.bases[d];
        } else {
            st_release_u32(row + d, kFlagAgg | sum);
            uint32_t excl = 0;
            bool ok = true;
            for (int64_t j = (int64_t)tile - 1; j >= 0; j--) {
                uint32_t v;
                if (!bounded_wait(a.status + j * kRadix + d, v, a.spin_limit, a.header)) {
                    ok = false;
                    break;
                }
                excl += v & kValueMask;
                if (v & kFlagIncl) break;
            }
            if (!ok) {
                raise_flag(a.header, GS_FLAG_TIMEOUT, 1u);
                s_timed_out = 1;
            }
            st_release_u32(row + d, kFlagIncl | ((excl + sum) & kValueMask));
            s_goff[d] = a.bases[d] + excl;
        }
        // block-wide exclusive scan of the counts -> digit run starts in the tile
        uint32_t v = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        if (lane == 31) s_warp_tot[warp] = v;
        __syncthreads();
        uint32_t add = 0;
        for (int w = 0; w < warp; w++) add += s_warp_tot[w];
        s_dstart[d] = v + add - sum;
    }
    __syncthreads();
    const bool skip = s_timed_out != 0;

    // reorder keys in shared memory by (digit, rank)
    uint16_t loc[kSortItems];
#pragma unroll
    for (int i = 0; i < kSortItems; i++) {
        const int li = warp_base + i * 32 + lane;
        if (li < n_valid) {
            const uint32_t d = (uint32_t)(key[i] >> shift) & dmask;
            loc[i] = (uint16_t)(s_dstart[d] + s_hist[warp * kRadix + d] + rank[i]);
            s_keys[loc[i]] = key[i];
        }
    }
    __syncthreads();
    uint32_t dest[kSortItems];
#pragma unroll
    for (int k = 0; k < kSortItems; k++) {
        const int j = k * kSortThreads + tid;
        dest[k] = 0xffffffffu;
        if (j < n_valid) {
            const uint64_t kk = s_keys[j];
            const uint32_t d = (uint32_t)(kk >> shift) & dmask;
            const uint32_t o = s_goff[d] + (uint32_t)j - s_dstart[d];
            if (!skip && (int64_t)o < K) {
                a.keys_out[o] = kk;
                dest[k] = o;
            }
        }
    }
    __syncthreads();
    uint32_t* s_vals = reinterpret_cast<uint32_t*>(s_keys);
#pragma unroll
    for (int i = 0; i < kSortItems; i++) {
        const int li = warp_base + i * 32 + lane;
        if (li < n_valid) s_vals[loc[i]] = a.vals_in[start + li];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kSortItems; k++) {
        const int j = k * kSortThreads + tid;
        if (j < n_valid && dest[k] != 0xffffffffu) a.vals_out[dest[k]] = s_vals[j];
    }
}

__global__ void copy_back_kernel(const uint64_t* __restrict__ ks, const uint32_t* __restrict__ vs,
                                 uint64_t* __restrict__ kd, uint32_t* __restrict__ vd,
                                 const uint64_t* __restrict__ num_keys, int64_t cap) {
    const int64_t K = key_count(num_keys, cap);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < K; i += stride) {
        kd[i] = ks[i];
        vd[i] = vs[i];
    }
}

__global__ void tile_ranges_kernel(const uint64_t* __restrict__ keys, const uint64_t* __restrict__ num_keys,
                                   int64_t cap, int n_tiles, uint2* __restrict__ ranges) {
    const int64_t K = key_count(num_keys, cap);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < K; i += stride) {
        const uint32_t t = (uint32_t)(keys[i] >> 32);
        if (t >= (uint32_t)n_tiles) continue;
        const uint32_t prev = i > 0 ? (uint32_t)(keys[i - 1] >> 32) : 0xffffffffu;
        const uint32_t next = i + 1 < K ? (uint32_t)(keys[i + 1] >> 32) : 0xffffffffu;
        if (t != prev) ranges[t].x = (uint32_t)i;
        if (t != next) ranges[t].y = (uint32_t)(i + 1);
    }
}

__global__ void spin_timeout_test_kernel(StatusHeader* h, long long iterations) {
    uint32_t v;
    // pad[0] of the header is never written by anyone: the wait must run out
    if (!bounded_wait(&h->pad[0], v, iterations, h)) raise_flag(h, GS_FLAG_TIMEOUT, 2u);
}

int grid_for(int64_t work, int threads, int max_blocks) {
    int64_t b = (work + threads - 1) / threads;
    if (b < 1) b = 1;
    return (int)(b < max_blocks ? b : max_blocks);
}

}  // namespace

size_t sort_scratch_bytes(int64_t cap) {
    return align_up(sizeof(uint32_t) * kMaxPasses * kRadix) + align_up(sizeof(uint32_t) * kMaxPasses) +
           align_up(sizeof(uint32_t) * 2 * (size_t)sort_max_tiles(cap > 0 ? cap : 1) * kRadix);
}

cudaError_t launch_sort(uint64_t* keys, uint32_t* vals, uint64_t* keys_alt, uint32_t* vals_alt,
                        const uint64_t* num_keys, int64_t cap, int key_bits, StatusHeader* status,
                        void* scratch, long long spin_limit, cudaStream_t s) {
    if (cap == 0) return cudaSuccess;
    const SortScratch sc = carve(scratch, cap);
    const int passes = (key_bits + 7) / 8;
    cudaError_t e = cudaMemsetAsync(sc.hist, 0, sizeof(uint32_t) * kMaxPasses * kRadix, s);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(sc.counters, 0, sizeof(uint32_t) * kMaxPasses, s);
    if (e != cudaSuccess) return e;
    sort_histogram_kernel<<<grid_for(cap, kSortThreads * 16, 148 * 8), kSortThreads, 0, s>>>(
        keys, num_keys, cap, passes, key_bits, sc.hist, sc.lookback, sc.max_tiles);
    sort_bases_kernel<<<passes, kRadix, 0, s>>>(sc.hist);
    const unsigned tiles = (unsigned)sc.max_tiles;
    for (int p = 0; p < passes; p++) {
        PassArgs a;
        const bool even = (p % 2) == 0;
        a.keys_in = even ? keys : keys_alt;
        a.vals_in = even ? vals : vals_alt;
        a.keys_out = even ? keys_alt : keys;
        a.vals_out = even ? vals_alt : vals;
        a.num_keys = num_keys;
        a.cap = cap;
        a.pass = p;
        a.digit_bits = key_bits - 8 * p < 8 ? key_bits - 8 * p : 8;
        a.bases = sc.hist + p * kRadix;
        a.counter = sc.counters + p;
        a.status = sc.lookback + (int64_t)(p % 2) * sc.max_tiles * kRadix;
        a.status_clear = p >= 1 ? sc.lookback + (int64_t)((p + 1) % 2) * sc.max_tiles * kRadix : nullptr;
        a.header = status;
        a.spin_limit = spin_limit;
        onesweep_kernel<<<tiles, kSortThreads, 0, s>>>(a);
    }
    if (passes % 2 == 1)
        copy_back_kernel<<<grid_for(cap, 256 * 8, 148 * 8), 256, 0, s>>>(keys_alt, vals_alt, keys, vals, num_keys, cap);
    return cudaGetLastError();
}

cudaError_t launch_tile_ranges(const uint64_t* sorted_keys, const uint64_t* num_keys, int64_t cap, int n_tiles,
                               uint32_t* ranges, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(ranges, 0, sizeof(uint32_t) * 2 * (size_t)n_tiles, s);
    if (e != cudaSuccess || cap == 0) return e;
    tile_ranges_kernel<<<grid_for(cap, 256 * 8, 148 * 8), 256, 0, s>>>(sorted_keys, num_keys, cap, n_tiles,
                                                                      reinterpret_cast<uint2*>(ranges));
    return cudaGetLastError();
}

cudaError_t launch_spin_timeout_test(StatusHeader* status, long long iterations, cudaStream_t s) {
    spin_timeout_test_kernel<<<1, 1, 0, s>>>(status, iterations);
    return cudaGetLastError();
}

}  // namespace gs
