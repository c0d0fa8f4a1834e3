// Step 3 (flowchart box "Depth-sort per tile" on the lesson page "3D Gaussian
// Splatting à partir de zéro") and step 4 (per-tile ranges).
//
// Stable least-significant-digit radix sort of (key, uint32 value) pairs with
// 8-bit digits, for 64-bit keys (the binning keys: tile id in the high word,
// depth bits in the low word) and 32-bit keys (depth bits; tile ids). Equal
// keys keep their input order.
//
//   sort_histogram : one read of all keys; 256-bin histograms of every digit
//                    position at once (shared-memory counters, then global
//                    atomics). Also clears the look-back rows the passes use.
//   sort_bases     : exclusive scan of each histogram -> digit base offsets.
//   onesweep pass  : one kernel per digit. Each block takes the next tile of
//                    keys (tile ids from an atomic counter, so a block only
//                    ever waits on blocks that are already running), ranks
//                    its keys stably with warp match/popc counters, publishes
//                    its per-digit counts (before the ranking when the whole
//                    pass is one wave of resident blocks), and finds its global
//                    offsets by decoupled look-back over earlier tiles. Keys and values
//                    are then reordered in shared memory (together for 32-bit
//                    keys, one after the other for 64-bit keys) and written
//                    out in digit-contiguous runs (coalesced).
//   copy back      : only when the pass count is odd.
//
// A look-back status word is (flag << 30 | count), written and read as one
// relaxed 32-bit access: the count travels with its flag, so no fence is
// needed. Every wait is bounded (polling iterations, with backoff); a wait
// that runs out sets GS_FLAG_TIMEOUT in the workspace header and the block
// still publishes a status so that no other block waits on it. All stores are
// bounds-checked against the key count.
#include <map>
#include <mutex>

#include "gs_internal.cuh"

#ifndef GS_SORT_THREADS
#define GS_SORT_THREADS 512
#endif
#ifndef GS_SORT_ITEMS
#define GS_SORT_ITEMS 8
#endif
#ifndef GS_SORT_MIN_BLOCKS
#define GS_SORT_MIN_BLOCKS 2
#endif
#ifndef GS_SORT_LOOKBACK
#define GS_SORT_LOOKBACK 8
#endif

namespace gs {
namespace {

constexpr int kSortThreads = GS_SORT_THREADS;
constexpr int kSortItems = GS_SORT_ITEMS;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortTile = kSortThreads * kSortItems;
constexpr int kRadix = 256;
constexpr int kMaxPasses = 8;
constexpr int kLookback = GS_SORT_LOOKBACK;
constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagIncl = 2u << 30;
constexpr uint32_t kValueMask = (1u << 30) - 1u;
static_assert(kSortThreads >= kRadix, "one thread per digit");
static_assert(kSortTile <= 65535, "tile offsets are 16-bit");

struct SortScratch {
    uint32_t* hist;      // [kMaxPasses][256], becomes the digit bases
    uint32_t* counters;  // [kMaxPasses] tile-id counters
    uint32_t* lookback;  // [2][max_tiles][256]
    int64_t max_tiles;
};

__host__ __device__ inline int64_t sort_max_tiles(int64_t cap) { return (cap + kSortTile - 1) / kSortTile; }

constexpr size_t kHeadBytes = align_up(sizeof(uint32_t) * kMaxPasses * kRadix) + align_up(sizeof(uint32_t) * kMaxPasses);

// head: the histograms, then the counters; lookback: the look-back rows
SortScratch carve(void* head, void* lookback, int64_t cap) {
    SortScratch s;
    char* p = static_cast<char*>(head);
    s.hist = reinterpret_cast<uint32_t*>(p);
    s.counters = reinterpret_cast<uint32_t*>(p + align_up(sizeof(uint32_t) * kMaxPasses * kRadix));
    s.lookback = static_cast<uint32_t*>(lookback);
    s.max_tiles = sort_max_tiles(cap > 0 ? cap : 1);
    return s;
}

// number of keys: min(*num_keys, cap), or cap when the count is known on the host
__device__ __forceinline__ int64_t key_count(const uint64_t* num_keys, int64_t cap) {
    if (!num_keys) return cap;
    const unsigned long long k = *num_keys;
    return k < (unsigned long long)cap ? (int64_t)k : cap;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Polls *p until a status flag is present. Returns false if the bound ran out
// or another block already reported a timeout.
__device__ bool bounded_wait(const uint32_t* p, uint32_t& v, long long limit, const StatusHeader* h) {
    long long it = 0;
    while (true) {
        v = ld_relaxed_u32(p);
        if (v & (kFlagAgg | kFlagIncl)) return true;
        if (++it > limit) return false;
        if ((it & 31) == 0 && (ld_volatile_u32(&h->flags) & GS_FLAG_TIMEOUT)) return false;
        __nanosleep(it < 32 ? 32 : 256);
    }
}

template <typename KeyT>
__device__ __forceinline__ uint32_t digit_of(KeyT k, int shift, uint32_t mask) {
    return (uint32_t)(k >> shift) & mask;
}

template <typename KeyT>
__global__ void __launch_bounds__(256) sort_histogram_kernel(const KeyT* __restrict__ keys,
                                                             const uint64_t* __restrict__ num_keys, int64_t cap,
                                                             int passes, int key_bits, uint32_t* __restrict__ hist) {
    grid_dependency_begin();
    __shared__ uint32_t s_hist[kMaxPasses * kRadix];
    for (int i = threadIdx.x; i < passes * kRadix; i += blockDim.x) s_hist[i] = 0;
    __syncthreads();
    const int64_t K = key_count(num_keys, cap);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < K; i += stride) {
        const KeyT k = keys[i];
        for (int p = 0; p < passes; p++) {
            const int w = digit_width(key_bits, p);
            atomicAdd(&s_hist[p * kRadix + digit_of(k, digit_shift(key_bits, p), (1u << w) - 1u)], 1u);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < passes * kRadix; i += blockDim.x)
        if (s_hist[i]) atomicAdd(&hist[i], s_hist[i]);
}

// Blocks [0, passes): exclusive scan of one digit histogram -> digit bases;
// block 0 also clears the passes' tile-id counters. The other blocks clear the
// look-back rows the passes will use (both ping-pong arrays), for the tiles of
// this sort only.
__global__ void __launch_bounds__(kRadix) sort_bases_kernel(uint32_t* __restrict__ hist, int passes,
                                                            const uint64_t* __restrict__ num_keys, int64_t cap,
                                                            uint32_t* __restrict__ lookback, int64_t max_tiles,
                                                            uint32_t* __restrict__ counters) {
    grid_dependency_begin();
    __shared__ uint32_t warp_tot[kRadix / 32];
    if (blockIdx.x == 0 && threadIdx.x < kMaxPasses) counters[threadIdx.x] = 0;
    if ((int)blockIdx.x >= passes) {
        const int64_t K = key_count(num_keys, cap);
        const int64_t words = (K + kSortTile - 1) / kSortTile * kRadix;
        const int64_t stride = (int64_t)(gridDim.x - passes) * kRadix;
        for (int64_t i = (int64_t)(blockIdx.x - passes) * kRadix + threadIdx.x; i < words; i += stride) {
            lookback[i] = 0;
            lookback[max_tiles * kRadix + i] = 0;
        }
        return;
    }
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

template <typename KeyT>
struct PassArgs {
    const KeyT* keys_in;
    const uint32_t* vals_in;
    KeyT* keys_out;
    uint32_t* vals_out;
    const uint64_t* num_keys;
    int64_t cap;
    int pass;
    int shift;
    int digit_bits;
    const uint32_t* bases;    // [256] for this pass
    uint32_t* counter;        // tile-id counter for this pass
    uint32_t* status;         // look-back rows of this pass
    uint32_t* status_clear;   // rows of the other array, cleared for the pass after next
    StatusHeader* header;
    long long spin_limit;
};

// Stable rank of a warp's keys within the warp: position order is (i, lane).
// wh: the warp's 256 16-bit digit counters. The leader of each group of equal
// digits (its lowest lane) advances the counter from the value it read.
// kFull: all kSortItems x 32 positions hold keys (no validity masks).
// The lanes holding the same digit come from match.any, whose cost grows with
// the number of distinct digits in the warp; for digits of at most five bits
// (a pass over the top bits of the tile keys, where most of a warp's 32
// lanes hold different digits) five ballots give the same lane set at a
// fixed cost.
template <bool kFull, typename KeyT>
__device__ __forceinline__ void rank_in_warp(const KeyT (&key)[kSortItems], uint32_t (&rank)[kSortItems], int shift,
                                             uint32_t dmask, int warp_base, int n_valid, uint16_t* wh,
                                             uint32_t lt, int lane) {
    if (dmask <= 31u) {
#pragma unroll
        for (int i = 0; i < kSortItems; i++) {
            const uint32_t d = digit_of(key[i], shift, dmask);
            const bool v = kFull || warp_base + i * 32 + lane < n_valid;
            uint32_t peers = __ballot_sync(0xffffffffu, v);
#pragma unroll
            for (int b = 0; b < 5; b++) {
                const uint32_t bal = __ballot_sync(0xffffffffu, (d >> b) & 1u);
                peers &= ((d >> b) & 1u) ? bal : ~bal;
            }
            const uint32_t below = __popc(peers & lt);
            uint32_t r = 0;
            if (v) r = wh[d] + below;
            __syncwarp();
            if (v && below == 0) wh[d] = (uint16_t)(r + __popc(peers));
            __syncwarp();
            rank[i] = r;
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < kSortItems; i++) {
        const uint32_t d = digit_of(key[i], shift, dmask);
        if constexpr (kFull) {
            const uint32_t peers = __match_any_sync(0xffffffffu, d);
            const uint32_t below = __popc(peers & lt);
            const uint32_t r = wh[d] + below;
            __syncwarp();
            if (below == 0) wh[d] = (uint16_t)(r + __popc(peers));
            __syncwarp();
            rank[i] = r;
        } else {
            const bool v = warp_base + i * 32 + lane < n_valid;
            const uint32_t peers = __match_any_sync(0xffffffffu, v ? d : 0xffffu) & __ballot_sync(0xffffffffu, v);
            const uint32_t below = __popc(peers & lt);
            uint32_t r = 0;
            if (v) r = wh[d] + below;
            __syncwarp();
            if (v && below == 0) wh[d] = (uint16_t)(r + __popc(peers));
            __syncwarp();
            rank[i] = r;
        }
    }
}

// kEarly: the tile's digit counts are taken (shared atomics) and published as
// its aggregate before the ranking, so that later tiles' look-back finds them
// sooner. That pays when every tile of the pass is resident at once (a single
// wave, where each tile's look-back walks back over tiles started at the same
// moment); with several waves the extra counting costs more than it saves.
template <typename KeyT, bool kEarly>
__global__ void __launch_bounds__(kSortThreads, GS_SORT_MIN_BLOCKS) onesweep_kernel(const PassArgs<KeyT> a) {
    grid_dependency_begin();
    __shared__ uint16_t s_hist[kSortWarps * kRadix];  // per-warp digit counters -> offsets
    __shared__ uint32_t s_dstart[kRadix];
    __shared__ uint32_t s_goff[kRadix];
    __shared__ uint32_t s_warp_tot[kRadix / 32];
    __shared__ __align__(16) KeyT s_keys[kSortTile];
    // 32-bit keys: the values get their own staging, so keys and values move
    // in one round (64-bit keys and their values would not fit the 48 KB of
    // static shared memory; the values then reuse the key staging afterwards)
    constexpr bool kJoint = sizeof(KeyT) == 4;
    __shared__ uint32_t s_vals_joint[kJoint ? kSortTile : 1];
    __shared__ uint32_t s_tile;
    __shared__ int s_timed_out;
    __shared__ uint32_t s_early[kEarly ? kRadix : 1];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_tile = atomicAdd(a.counter, 1u);
        s_timed_out = 0;
    }
    for (int i = tid; i < kSortWarps * kRadix; i += kSortThreads) s_hist[i] = 0;
    if (kEarly && tid < kRadix) s_early[tid] = 0;
    __syncthreads();
    const int64_t K = key_count(a.num_keys, a.cap);
    const uint32_t tile = s_tile;
    const int64_t start = (int64_t)tile * kSortTile;
    if (start >= K) return;
    const int n_valid = (int)(K - start < kSortTile ? K - start : kSortTile);
    if (a.status_clear && tid < kRadix) {
        // rows used by the previous pass are not read again until two passes on
        a.status_clear[(int64_t)tile * kRadix + tid] = 0;
    }

    const int shift = a.shift;
    const uint32_t dmask = (1u << a.digit_bits) - 1u;
    const int warp_base = warp * (kSortItems * 32);
    KeyT key[kSortItems];
    uint32_t val[kSortItems];
#pragma unroll
    for (int i = 0; i < kSortItems; i++) {
        const int li = warp_base + i * 32 + lane;
        key[i] = li < n_valid ? a.keys_in[start + li] : (KeyT)0;
    }
#pragma unroll
    for (int i = 0; i < kSortItems; i++) {
        const int li = warp_base + i * 32 + lane;
        val[i] = li < n_valid ? a.vals_in[start + li] : 0u;
    }

    if constexpr (kEarly) {
#pragma unroll
        for (int i = 0; i < kSortItems; i++) {
            const int li = warp_base + i * 32 + lane;
            if (li < n_valid) atomicAdd(&s_early[digit_of(key[i], shift, dmask)], 1u);
        }
        __syncthreads();
        if (tid < kRadix && tile != 0) st_relaxed_u32(a.status + (int64_t)tile * kRadix + tid, kFlagAgg | s_early[tid]);
    }

    // stable rank within the warp: position order is (i, lane)
    uint16_t* wh = s_hist + warp * kRadix;
    const uint32_t lt = lanemask_lt();
    uint32_t rank[kSortItems];
    if (n_valid == kSortTile)
        rank_in_warp<true>(key, rank, shift, dmask, warp_base, n_valid, wh, lt, lane);
    else
        rank_in_warp<false>(key, rank, shift, dmask, warp_base, n_valid, wh, lt, lane);
    __syncthreads();

    // per digit (thread = digit): offsets of each warp inside the block, the
    // tile's count published for later tiles, and the look-back over earlier ones
    uint32_t sum = 0;
    if (tid < kRadix) {
        const int d = tid;
#pragma unroll
        for (int w = 0; w < kSortWarps; w++) {
            const uint32_t c = s_hist[w * kRadix + d];
            s_hist[w * kRadix + d] = (uint16_t)sum;
            sum += c;
        }
        uint32_t* row = a.status + (int64_t)tile * kRadix;
        if (tile == 0) {
            st_relaxed_u32(row + d, kFlagIncl | sum);
            s_goff[d] = a.bases[d];
        } else {
            if (!kEarly) st_relaxed_u32(row + d, kFlagAgg | sum);
            // look back in windows of kLookback earlier tiles: the window's
            // loads are issued together, then consumed nearest first until an
            // inclusive prefix is met (a not-yet-published one is waited for)
            uint32_t excl = 0;
            bool ok = true, found = false;
            for (int64_t j = (int64_t)tile - 1; j >= 0 && ok && !found; j -= kLookback) {
                uint32_t v[kLookback];
#pragma unroll
                for (int k = 0; k < kLookback; k++)
                    v[k] = j - k >= 0 ? ld_relaxed_u32(a.status + (j - k) * kRadix + d) : 0u;
#pragma unroll
                for (int k = 0; k < kLookback; k++) {
                    if (found || !ok || j - k < 0) break;
                    uint32_t x = v[k];
                    if (!(x & (kFlagAgg | kFlagIncl)) &&
                        !bounded_wait(a.status + (j - k) * kRadix + d, x, a.spin_limit, a.header)) {
                        ok = false;
                        break;
                    }
                    excl += x & kValueMask;
                    if (x & kFlagIncl) found = true;
                }
            }
            if (!ok) {
                raise_flag(a.header, GS_FLAG_TIMEOUT, 1u);
                s_timed_out = 1;
            }
            st_relaxed_u32(row + d, kFlagIncl | ((excl + sum) & kValueMask));
            s_goff[d] = a.bases[d] + excl;
        }
        // warp-level inclusive scan of the counts (block scan finished below)
        uint32_t v = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        if (lane == 31) s_warp_tot[warp] = v;
        sum = v - sum;  // exclusive within the warp
    }
    __syncthreads();
    if (tid < kRadix) {
        uint32_t add = 0;
        for (int w = 0; w < warp; w++) add += s_warp_tot[w];
        s_dstart[tid] = sum + add;
    }
    __syncthreads();
    const bool skip = s_timed_out != 0;

    // reorder keys in shared memory by (digit, rank)
    if constexpr (kJoint) {
#pragma unroll
        for (int i = 0; i < kSortItems; i++) {
            const int li = warp_base + i * 32 + lane;
            if (li < n_valid) {
                const uint32_t d = digit_of(key[i], shift, dmask);
                const uint32_t loc = s_dstart[d] + s_hist[warp * kRadix + d] + rank[i];
                s_keys[loc] = key[i];
                s_vals_joint[loc] = val[i];
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kSortItems; k++) {
            const int j = k * kSortThreads + tid;
            if (j < n_valid) {
                const KeyT kk = s_keys[j];
                const uint32_t d = digit_of(kk, shift, dmask);
                const uint32_t o = s_goff[d] + (uint32_t)j - s_dstart[d];
                GS_CHECK(skip || (int64_t)o < K);
                if (!skip && (int64_t)o < K) {
                    a.keys_out[o] = kk;
                    a.vals_out[o] = s_vals_joint[j];
                }
            }
        }
    } else {
        // 64-bit keys: keys first, then the values through the same staging
        uint32_t loc[kSortItems];
#pragma unroll
        for (int i = 0; i < kSortItems; i++) {
            const int li = warp_base + i * 32 + lane;
            loc[i] = 0xffffffffu;
            if (li < n_valid) {
                const uint32_t d = digit_of(key[i], shift, dmask);
                loc[i] = s_dstart[d] + s_hist[warp * kRadix + d] + rank[i];
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
                const KeyT kk = s_keys[j];
                const uint32_t d = digit_of(kk, shift, dmask);
                const uint32_t o = s_goff[d] + (uint32_t)j - s_dstart[d];
                GS_CHECK(skip || (int64_t)o < K);
                if (!skip && (int64_t)o < K) {
                    a.keys_out[o] = kk;
                    dest[k] = o;
                }
            }
        }
        __syncthreads();
        uint32_t* s_vals = reinterpret_cast<uint32_t*>(s_keys);
#pragma unroll
        for (int i = 0; i < kSortItems; i++)
            if (loc[i] != 0xffffffffu) s_vals[loc[i]] = val[i];
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kSortItems; k++) {
            const int j = k * kSortThreads + tid;
            if (j < n_valid && dest[k] != 0xffffffffu) a.vals_out[dest[k]] = s_vals[j];
        }
    }
}

// Persistent pass for 32-bit keys, used when a pass spans several waves of
// blocks (large key counts): each block claims tiles from the pass's counter
// and, while it ranks and scatters one tile, the bulk-copy engine already
// brings the next tile's keys and values into the other half of a
// double-buffered shared-memory stage (cp.async.bulk on an mbarrier), so the
// loads of one tile overlap the latency-bound phases of the previous one. The
// tile's digit counts are published before the ranking, as in the single-wave
// case. The ranking, look-back and scatter are those of onesweep_kernel. Tiles
// are claimed in increasing order and a block only claims its next tile while
// it holds a lower one, so every tile a look-back waits on is being processed.
// A bulk copy that did not land within kBulkWaitLimit polls sets
// GS_FLAG_TIMEOUT; the block then waits (bounded) for both of its copies and
// leaves.
constexpr int kPipeBytes = (6 * kSortTile) * 4 + kSortWarps * kRadix * 2;
__global__ void __launch_bounds__(kSortThreads, 2) onesweep_pipe_kernel(const PassArgs<uint32_t> a) {
    grid_dependency_begin();
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* s_kin = reinterpret_cast<uint32_t*>(smem);          // [2][kSortTile]
    uint32_t* s_vin = s_kin + 2 * kSortTile;                       // [2][kSortTile]
    uint32_t* s_keys = s_vin + 2 * kSortTile;                      // [kSortTile] sorted staging
    uint32_t* s_vals = s_keys + kSortTile;                         // [kSortTile]
    uint16_t* s_hist = reinterpret_cast<uint16_t*>(s_vals + kSortTile);   // [kSortWarps][kRadix]
    __shared__ uint32_t s_dstart[kRadix];
    __shared__ uint32_t s_goff[kRadix];
    __shared__ uint32_t s_warp_tot[kRadix / 32];
    __shared__ uint32_t s_early[kRadix];
    __shared__ uint32_t s_tile[2];
    __shared__ int s_timed_out;
    __shared__ __align__(8) uint64_t s_bar[2];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t K = key_count(a.num_keys, a.cap);
    const int64_t ntiles = (K + kSortTile - 1) / kSortTile;
    const int shift = a.shift;
    const uint32_t dmask = (1u << a.digit_bits) - 1u;
    auto whole = [&](int64_t t) { return (t + 1) * kSortTile <= K; };
    auto issue = [&](int64_t t, int b) {
        mbar_arrive_expect_tx(&s_bar[b], 2u * kSortTile * 4u);
        bulk_copy_g2s(s_kin + b * kSortTile, a.keys_in + t * kSortTile, kSortTile * 4, &s_bar[b]);
        bulk_copy_g2s(s_vin + b * kSortTile, a.vals_in + t * kSortTile, kSortTile * 4, &s_bar[b]);
    };
    if (tid == 0) {
        mbar_init(&s_bar[0], 1);
        mbar_init(&s_bar[1], 1);
        mbar_init_fence();
        s_tile[0] = atomicAdd(a.counter, 1u);
    }
    __syncthreads();
    if (tid == 0 && (int64_t)s_tile[0] < ntiles && whole(s_tile[0])) issue(s_tile[0], 0);
    uint32_t parity = 0;   // bit b: parity of the next phase of s_bar[b]
    int buf = 0;
    while (true) {
        const int64_t tile = s_tile[buf];
        if (tile >= ntiles) break;
        if (tid == 0) {
            const uint32_t nt = atomicAdd(a.counter, 1u);
            s_tile[buf ^ 1] = nt;
            if ((int64_t)nt < ntiles && whole(nt)) {
                fence_proxy_async_shared();
                issue(nt, buf ^ 1);
            }
            s_timed_out = 0;
        }
        for (int i = tid; i < kSortWarps * kRadix / 2; i += kSortThreads) reinterpret_cast<uint32_t*>(s_hist)[i] = 0;
        if (tid < kRadix) s_early[tid] = 0;
        const int64_t start = tile * kSortTile;
        const int n_valid = (int)(K - start < kSortTile ? K - start : kSortTile);
        uint32_t* kin = s_kin + buf * kSortTile;
        uint32_t* vin = s_vin + buf * kSortTile;
        bool landed = true;
        if (whole(tile)) {
            landed = mbar_wait_bounded(&s_bar[buf], (parity >> buf) & 1u, kBulkWaitLimit);
            parity ^= 1u << buf;
        } else {
            for (int i = tid; i < n_valid; i += kSortThreads) {
                kin[i] = a.keys_in[start + i];
                vin[i] = a.vals_in[start + i];
            }
        }
        if (__syncthreads_or(!landed)) {
            if (tid == 0) raise_flag(a.header, GS_FLAG_TIMEOUT, 4u);
            mbar_wait_bounded(&s_bar[buf], ((parity >> buf) & 1u) ^ 1u, kBulkWaitLimit);
            mbar_wait_bounded(&s_bar[buf ^ 1], (parity >> (buf ^ 1)) & 1u, kBulkWaitLimit);
            return;
        }
        if (a.status_clear && tid < kRadix) a.status_clear[tile * kRadix + tid] = 0;

        const int warp_base = warp * (kSortItems * 32);
        uint32_t key[kSortItems];
#pragma unroll
        for (int i = 0; i < kSortItems; i++) {
            const int li = warp_base + i * 32 + lane;
            key[i] = li < n_valid ? kin[li] : 0u;
            if (li < n_valid) atomicAdd(&s_early[digit_of(key[i], shift, dmask)], 1u);
        }
        __syncthreads();
        if (tid < kRadix && tile != 0) st_relaxed_u32(a.status + tile * kRadix + tid, kFlagAgg | s_early[tid]);

        uint16_t* wh = s_hist + warp * kRadix;
        const uint32_t lt = lanemask_lt();
        uint32_t rank[kSortItems];
        // (the full-tile ranking of onesweep_kernel measured slower here: 5M and
        // stress tile sorts +4% and +8%)
#pragma unroll
        for (int i = 0; i < kSortItems; i++) {
            const int li = warp_base + i * 32 + lane;
            const bool v = li < n_valid;
            const uint32_t d = digit_of(key[i], shift, dmask);
            const uint32_t peers = __match_any_sync(0xffffffffu, v ? d : 0xffffu) & __ballot_sync(0xffffffffu, v);
            uint32_t r = 0;
            if (v) r = wh[d] + __popc(peers & lt);
            __syncwarp();
            if (v && (peers & lt) == 0) wh[d] = (uint16_t)(wh[d] + __popc(peers));
            __syncwarp();
            rank[i] = r;
        }
        __syncthreads();
        uint32_t sum = 0;
        if (tid < kRadix) {
            const int d = tid;
#pragma unroll
            for (int w = 0; w < kSortWarps; w++) {
                const uint32_t c = s_hist[w * kRadix + d];
                s_hist[w * kRadix + d] = (uint16_t)sum;
                sum += c;
            }
            uint32_t* row = a.status + tile * kRadix;
            if (tile == 0) {
                st_relaxed_u32(row + d, kFlagIncl | sum);
                s_goff[d] = a.bases[d];
            } else {
                uint32_t excl = 0;
                bool ok = true, found = false;
                for (int64_t j = tile - 1; j >= 0 && ok && !found; j -= kLookback) {
                    uint32_t v[kLookback];
#pragma unroll
                    for (int k = 0; k < kLookback; k++)
                        v[k] = j - k >= 0 ? ld_relaxed_u32(a.status + (j - k) * kRadix + d) : 0u;
#pragma unroll
                    for (int k = 0; k < kLookback; k++) {
                        if (found || !ok || j - k < 0) break;
                        uint32_t x = v[k];
                        if (!(x & (kFlagAgg | kFlagIncl)) &&
                            !bounded_wait(a.status + (j - k) * kRadix + d, x, a.spin_limit, a.header)) {
                            ok = false;
                            break;
                        }
                        excl += x & kValueMask;
                        if (x & kFlagIncl) found = true;
                    }
                }
                if (!ok) {
                    raise_flag(a.header, GS_FLAG_TIMEOUT, 1u);
                    s_timed_out = 1;
                }
                st_relaxed_u32(row + d, kFlagIncl | ((excl + sum) & kValueMask));
                s_goff[d] = a.bases[d] + excl;
            }
            uint32_t v = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            if (lane == 31) s_warp_tot[warp] = v;
            sum = v - sum;
        }
        __syncthreads();
        if (tid < kRadix) {
            uint32_t add = 0;
            for (int w = 0; w < warp; w++) add += s_warp_tot[w];
            s_dstart[tid] = sum + add;
        }
        __syncthreads();
        const bool skip = s_timed_out != 0;
#pragma unroll
        for (int i = 0; i < kSortItems; i++) {
            const int li = warp_base + i * 32 + lane;
            if (li < n_valid) {
                const uint32_t d = digit_of(key[i], shift, dmask);
                const uint32_t loc = s_dstart[d] + s_hist[warp * kRadix + d] + rank[i];
                s_keys[loc] = key[i];
                s_vals[loc] = vin[li];
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kSortItems; k++) {
            const int j = k * kSortThreads + tid;
            if (j < n_valid) {
                const uint32_t kk = s_keys[j];
                const uint32_t d = digit_of(kk, shift, dmask);
                const uint32_t o = s_goff[d] + (uint32_t)j - s_dstart[d];
                GS_CHECK(skip || (int64_t)o < K);
                if (!skip && (int64_t)o < K) {
                    a.keys_out[o] = kk;
                    a.vals_out[o] = s_vals[j];
                }
            }
        }
        __syncthreads();
        buf ^= 1;
    }
}

template <typename KeyT>
__global__ void copy_back_kernel(const KeyT* __restrict__ ks, const uint32_t* __restrict__ vs,
                                 KeyT* __restrict__ kd, uint32_t* __restrict__ vd,
                                 const uint64_t* __restrict__ num_keys, int64_t cap) {
    grid_dependency_begin();
    const int64_t K = key_count(num_keys, cap);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < K; i += stride) {
        kd[i] = ks[i];
        vd[i] = vs[i];
    }
}

// ranges from sorted keys whose tile id is (key >> shift). Each thread takes
// a run of kRangeItems consecutive keys (16-byte vector loads when the key
// array is 16-byte aligned) and the key on either side of it, so every key
// is read about once; a tile's start and end are written where its id
// differs from the previous and the next key's.
constexpr int kRangeItems = 8;

template <typename KeyT>
__global__ void __launch_bounds__(256) tile_ranges_kernel(const KeyT* __restrict__ keys,
                                                          const uint64_t* __restrict__ num_keys, int64_t cap,
                                                          int shift, int n_tiles, bool vec,
                                                          uint2* __restrict__ ranges, const TileKeyMap km) {
    grid_dependency_begin();
    static_assert(kRangeItems * sizeof(KeyT) % 16 == 0, "a run is whole 16-byte vectors");
    const int64_t K = key_count(num_keys, cap);
    const int64_t runs = (K + kRangeItems - 1) / kRangeItems;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < runs; c += stride) {
        const int64_t i0 = c * kRangeItems;
        const int n = K - i0 < kRangeItems ? (int)(K - i0) : kRangeItems;
        KeyT k[kRangeItems];
        if (vec && n == kRangeItems) {
            constexpr int kVec = kRangeItems * (int)sizeof(KeyT) / 16;
            const uint4* p = reinterpret_cast<const uint4*>(keys + i0);
            uint4 v[kVec];
#pragma unroll
            for (int j = 0; j < kVec; j++) v[j] = __ldg(p + j);
            memcpy(k, v, sizeof(k));
        } else {
#pragma unroll
            for (int j = 0; j < kRangeItems; j++) k[j] = j < n ? keys[i0 + j] : (KeyT)0;
        }
        uint32_t prev = i0 > 0 ? (uint32_t)(keys[i0 - 1] >> shift) : 0xffffffffu;
        const uint32_t after = i0 + n < K ? (uint32_t)(keys[i0 + n] >> shift) : 0xffffffffu;
#pragma unroll
        for (int j = 0; j < kRangeItems; j++) {
            if (j < n) {
                const uint32_t t = (uint32_t)(k[j] >> shift);
                const uint32_t next = j + 1 < n ? (uint32_t)(k[j + 1] >> shift) : after;
                if (t != prev || t != next) {   // a list's first or last entry
                    const uint32_t tile = tile_of_key(km, t);
                    GS_CHECK(tile < (uint32_t)n_tiles);
                    if (tile < (uint32_t)n_tiles) {
                        if (t != prev) ranges[tile].x = (uint32_t)(i0 + j);
                        if (t != next) ranges[tile].y = (uint32_t)(i0 + j + 1);
                    }
                }
                prev = t;
            }
        }
    }
}

__global__ void spin_timeout_test_kernel(StatusHeader* h, long long iterations) {
    grid_dependency_begin();
    uint32_t v;
    // pad[0] of the header is never written by anyone: the wait must run out
    if (!bounded_wait(&h->pad[0], v, iterations, h)) raise_flag(h, GS_FLAG_TIMEOUT, 2u);
}

int grid_for(int64_t work, int threads, int max_blocks) {
    int64_t b = (work + threads - 1) / threads;
    if (b < 1) b = 1;
    return (int)(b < max_blocks ? b : max_blocks);
}

// Blocks of the pass kernel resident on the current GPU at once, and the grid
// of the persistent pass (its resident blocks; 0 where it cannot run), with
// its dynamic shared memory allowed. Computed once per device and key width.
struct PassShapes {
    unsigned resident;      // blocks of onesweep_kernel resident at once
    unsigned pipe_blocks;   // grid of onesweep_pipe_kernel (0: not available)
};

template <typename KeyT>
cudaError_t resident_tiles(PassShapes* out) {
    static std::mutex mu;
    static std::map<int, PassShapes> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it == cache.end()) {
        int sms = 0, per_sm = 0, pipe_per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, onesweep_kernel<KeyT, false>, kSortThreads, 0);
        if (e != cudaSuccess) return e;
        if (sizeof(KeyT) == 4) {
            e = cudaFuncSetAttribute(onesweep_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPipeBytes);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&pipe_per_sm, onesweep_pipe_kernel, kSortThreads,
                                                                  kPipeBytes);
            if (e != cudaSuccess) return e;
        }
        PassShapes ps;
        ps.resident = (unsigned)(sms * per_sm);
        ps.pipe_blocks = (unsigned)(sms * pipe_per_sm);
        it = cache.emplace(dev, ps).first;
    }
    *out = it->second;
    return cudaSuccess;
}

// hist_ready: the digit histograms were already accumulated into the
// scratch's histogram array (zeroed by sort_prepare_histogram) by the kernel
// that produced the keys.
template <typename KeyT>
cudaError_t launch_sort_t(KeyT* keys, uint32_t* vals, KeyT* keys_alt, uint32_t* vals_alt, const uint64_t* num_keys,
                          int64_t cap, int key_bits, StatusHeader* status, void* head, void* lookback,
                          long long spin_limit, cudaStream_t s, bool hist_ready) {
    if (cap == 0) return cudaSuccess;
    const SortScratch sc = carve(head, lookback, cap);
    const int passes = (key_bits + 7) / 8;
    cudaError_t e;
    if (!hist_ready) {
        e = cudaMemsetAsync(sc.hist, 0, sizeof(uint32_t) * kMaxPasses * kRadix, s);
        if (e != cudaSuccess) return e;
        launch_k(sort_histogram_kernel<KeyT>, grid_for(cap, 256 * 16, 148 * 8), 256, 0, s, keys, num_keys, cap, passes,
                 key_bits, sc.hist);
    }
    const unsigned tiles = (unsigned)sc.max_tiles;
    PassShapes shapes;
    e = resident_tiles<KeyT>(&shapes);
    if (e != cudaSuccess) return e;
    const unsigned resident = shapes.resident, pipe_blocks = shapes.pipe_blocks;
    const int clear_blocks = grid_for(2 * sc.max_tiles * kRadix, kRadix * 8, 148 * 2);
    launch_k(sort_bases_kernel, passes + clear_blocks, kRadix, 0, s, sc.hist, passes, num_keys, cap, sc.lookback,
             sc.max_tiles, sc.counters);
    for (int p = 0; p < passes; p++) {
        PassArgs<KeyT> a;
        const bool even = (p % 2) == 0;
        a.keys_in = even ? keys : keys_alt;
        a.vals_in = even ? vals : vals_alt;
        a.keys_out = even ? keys_alt : keys;
        a.vals_out = even ? vals_alt : vals;
        a.num_keys = num_keys;
        a.cap = cap;
        a.pass = p;
        a.digit_bits = digit_width(key_bits, p);
        a.shift = digit_shift(key_bits, p);
        a.bases = sc.hist + p * kRadix;
        a.counter = sc.counters + p;
        a.status = sc.lookback + (int64_t)(p % 2) * sc.max_tiles * kRadix;
        a.status_clear = p >= 1 ? sc.lookback + (int64_t)((p + 1) % 2) * sc.max_tiles * kRadix : nullptr;
        a.header = status;
        a.spin_limit = spin_limit;
        bool piped = false;
        if constexpr (sizeof(KeyT) == 4) {
            // three waves or more, and arrays the bulk copies can read
            piped = pipe_blocks > 0 && tiles >= 3u * resident && ((uintptr_t)a.keys_in & 15) == 0 &&
                    ((uintptr_t)a.vals_in & 15) == 0;
            if (piped) launch_k(onesweep_pipe_kernel, pipe_blocks, kSortThreads, kPipeBytes, s, a);
        }
        if (!piped) {
            if (tiles <= resident)
                launch_k(onesweep_kernel<KeyT, true>, tiles, kSortThreads, 0, s, a);
            else
                launch_k(onesweep_kernel<KeyT, false>, tiles, kSortThreads, 0, s, a);
        }
    }
    if (passes % 2 == 1)
        launch_k(copy_back_kernel<KeyT>, grid_for(cap, 256 * 8, 148 * 8), 256, 0, s, keys_alt, vals_alt, keys, vals,
                 num_keys, cap);
    return cudaGetLastError();
}

}  // namespace

size_t sort_head_bytes() { return kHeadBytes; }
size_t sort_lookback_bytes(int64_t cap) {
    return align_up(sizeof(uint32_t) * 2 * (size_t)sort_max_tiles(cap > 0 ? cap : 1) * kRadix);
}
size_t sort_scratch_bytes(int64_t cap) { return sort_head_bytes() + sort_lookback_bytes(cap); }

cudaError_t launch_sort(uint64_t* keys, uint32_t* vals, uint64_t* keys_alt, uint32_t* vals_alt,
                        const uint64_t* num_keys, int64_t cap, int key_bits, StatusHeader* status, void* scratch,
                        long long spin_limit, cudaStream_t s) {
    return launch_sort_t<uint64_t>(keys, vals, keys_alt, vals_alt, num_keys, cap, key_bits, status, scratch,
                                   static_cast<char*>(scratch) + kHeadBytes, spin_limit, s, false);
}

cudaError_t launch_sort32(uint32_t* keys, uint32_t* vals, uint32_t* keys_alt, uint32_t* vals_alt,
                          const uint64_t* num_keys, int64_t cap, int key_bits, StatusHeader* status, void* scratch,
                          long long spin_limit, cudaStream_t s, bool hist_ready) {
    return launch_sort_t<uint32_t>(keys, vals, keys_alt, vals_alt, num_keys, cap, key_bits, status, scratch,
                                   static_cast<char*>(scratch) + kHeadBytes, spin_limit, s, hist_ready);
}

cudaError_t launch_sort32_split(uint32_t* keys, uint32_t* vals, uint32_t* keys_alt, uint32_t* vals_alt,
                                const uint64_t* num_keys, int64_t cap, int key_bits, StatusHeader* status, void* head,
                                void* lookback, long long spin_limit, cudaStream_t s, bool hist_ready) {
    return launch_sort_t<uint32_t>(keys, vals, keys_alt, vals_alt, num_keys, cap, key_bits, status, head, lookback,
                                   spin_limit, s, hist_ready);
}

uint32_t* sort_histogram_of(void* scratch) { return static_cast<uint32_t*>(scratch); }

cudaError_t sort_prepare_histogram(void* scratch, cudaStream_t s) {
    return cudaMemsetAsync(scratch, 0, sizeof(uint32_t) * kMaxPasses * kRadix, s);
}

cudaError_t launch_tile_ranges(const uint64_t* sorted_keys, const uint64_t* num_keys, int64_t cap, int n_tiles,
                               uint32_t* ranges, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(ranges, 0, sizeof(uint32_t) * 2 * (size_t)n_tiles, s);
    if (e != cudaSuccess || cap == 0) return e;
    const bool vec = (reinterpret_cast<uintptr_t>(sorted_keys) & 15) == 0;
    launch_k(tile_ranges_kernel<uint64_t>, grid_for(cap, 256 * kRangeItems, 148 * 8), 256, 0, s,
             sorted_keys, num_keys, cap, 32, n_tiles, vec, reinterpret_cast<uint2*>(ranges), identity_keys(0));
    return cudaGetLastError();
}

cudaError_t launch_tile_ranges32(const uint32_t* sorted_tiles, const uint64_t* num_keys, int64_t cap, int n_tiles,
                                 uint32_t* ranges, cudaStream_t s, bool ranges_zeroed, const TileKeyMap* keymap) {
    cudaError_t e = ranges_zeroed ? cudaSuccess : cudaMemsetAsync(ranges, 0, sizeof(uint32_t) * 2 * (size_t)n_tiles, s);
    if (e != cudaSuccess || cap == 0) return e;
    const bool vec = (reinterpret_cast<uintptr_t>(sorted_tiles) & 15) == 0;
    launch_k(tile_ranges_kernel<uint32_t>, grid_for(cap, 256 * kRangeItems, 148 * 8), 256, 0, s,
             sorted_tiles, num_keys, cap, 0, n_tiles, vec, reinterpret_cast<uint2*>(ranges),
             keymap ? *keymap : identity_keys(0));
    return cudaGetLastError();
}

cudaError_t launch_spin_timeout_test(StatusHeader* status, long long iterations, cudaStream_t s) {
    launch_k(spin_timeout_test_kernel, 1, 1, 0, s, status, iterations);
    return cudaGetLastError();
}

GS_DEFINE_CHECK_SETTER(sort)

}  // namespace gs
