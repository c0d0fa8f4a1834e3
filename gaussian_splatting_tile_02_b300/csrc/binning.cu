// Step 2 of the forward renderer: tile binning (flowchart box "Assign to
// tiles (16x16 screen-space)" on the lesson page "3D Gaussian Splatting à
// partir de zéro", section "Rastérisation, non rayée").
//
// A device prefix scan over tiles_touched gives each Gaussian the slot of its
// first key and the frame's key count K; the Gaussian's keys are then written
// in row-major order over its tile rectangle:
//     key = (uint64)(ty * tiles_x + tx) << 32 | float_bits(depth),  value = index.
// The same kernels also run over the Gaussians in a given order (the depth
// order) and then write 32-bit keys holding the tile id alone: a stable sort
// of those by tile gives the same per-tile (depth, index) order as the sort of
// the 64-bit keys, with a 13-bit key at 1080p instead of a 45-bit one.
//
// Three kernels: a per-chunk reduction (2048 Gaussians per block), a
// single-block scan of the chunk sums (which also publishes K), and the
// duplication, which re-scans its chunk and writes the keys warp by warp:
// the 32 lanes of a warp share the keys of 32 consecutive Gaussians
// (coalesced stores), so a Gaussian with many tiles does not serialise one
// thread.
#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kBinThreads = 512;
constexpr int kBinItems = 4;
constexpr int kBinChunk = kBinThreads * kBinItems;  // Gaussians per block

// Block-wide inclusive scan of one 64-bit value per thread (kBinThreads threads).
__device__ __forceinline__ unsigned long long block_scan_incl(unsigned long long v, unsigned long long* warp_tot,
                                                              unsigned long long* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[wid] = v;
    __syncthreads();
    if (wid == 0) {
        constexpr int NW = kBinThreads / 32;
        unsigned long long w = lane < NW ? warp_tot[lane] : 0ull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            unsigned long long t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        if (lane < NW) warp_tot[lane] = w;
        if (lane == NW - 1) *total = w;
    }
    __syncthreads();
    if (wid > 0) v += warp_tot[wid - 1];
    return v;
}

// Digit histograms of 32-bit keys in the radix sort's digit layout
// (digit_shift / digit_width, [pass][256]); accumulated in shared memory,
// flushed with one global atomic per non-zero bin.
constexpr int kHistPasses = 4;
__device__ __forceinline__ uint32_t digit(uint32_t key, int key_bits, int p) {
    return (key >> digit_shift(key_bits, p)) & ((1u << digit_width(key_bits, p)) - 1u);
}
__device__ __forceinline__ void count_digits(uint32_t* s_hist, uint32_t key, int key_bits) {
    const int passes = digit_passes(key_bits);
#pragma unroll
    for (int p = 0; p < kHistPasses; p++)
        if (p < passes) atomicAdd(&s_hist[p * 256 + digit(key, key_bits, p)], 1u);
}
__device__ __forceinline__ void flush_digits(const uint32_t* s_hist, uint32_t* hist, int key_bits) {
    const int n = digit_passes(key_bits) * 256;
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        if (s_hist[i]) atomicAdd(&hist[i], s_hist[i]);
}

// Gaussian at list position i: the identity, or order[i]
__device__ __forceinline__ uint32_t at(const uint32_t* __restrict__ order, int64_t i) {
    return order ? __ldg(order + i) : (uint32_t)i;
}

__global__ void __launch_bounds__(kBinThreads) bin_reduce_kernel(const uint32_t* __restrict__ tiles_touched,
                                                                 const uint32_t* __restrict__ order, int64_t n,
                                                                 unsigned long long* __restrict__ block_sums) {
    grid_dependency_begin();
    __shared__ unsigned long long warp_tot[kBinThreads / 32];
    __shared__ unsigned long long total;
    const int64_t base = (int64_t)blockIdx.x * kBinChunk + (int64_t)threadIdx.x * kBinItems;
    unsigned long long s = 0;
#pragma unroll
    for (int i = 0; i < kBinItems; i++)
        if (base + i < n) s += __ldg(tiles_touched + at(order, base + i));
    block_scan_incl(s, warp_tot, &total);
    if (threadIdx.x == 0) block_sums[blockIdx.x] = total;
}

// Exclusive scan of the chunk sums in place; K = total.
__global__ void __launch_bounds__(1024) bin_scan_sums_kernel(unsigned long long* __restrict__ sums, int nb,
                                                             int64_t key_capacity, uint64_t* __restrict__ num_keys,
                                                             StatusHeader* __restrict__ status) {
    grid_dependency_begin();
    __shared__ unsigned long long warp_tot[32];
    __shared__ unsigned long long carry;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int start = 0; start < nb; start += 1024) {
        const int i = start + threadIdx.x;
        const unsigned long long x = i < nb ? sums[i] : 0ull;
        unsigned long long v = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        if (lane == 31) warp_tot[wid] = v;
        __syncthreads();
        if (wid == 0) {
            unsigned long long w = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                unsigned long long t = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += t;
            }
            warp_tot[lane] = w;
        }
        __syncthreads();
        const unsigned long long incl = v + (wid > 0 ? warp_tot[wid - 1] : 0ull) + carry;
        if (i < nb) sums[i] = incl - x;
        __syncthreads();
        if (threadIdx.x == 1023) carry = incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *num_keys = carry;
        status->num_keys = carry;
        if (carry > (unsigned long long)key_capacity) atomicOr(&status->flags, GS_FLAG_CAPACITY);
    }
}

// KeyT = uint64_t: key = tile << 32 | depth bits; KeyT = uint32_t: key = tile.
// q = floor(r / w) for r < 2^24, 1 <= w < 2^16: a float quotient, then one
// exact correction step either way.
__device__ __forceinline__ uint32_t div_small(uint32_t r, uint32_t w) {
    uint32_t q = (uint32_t)__fdiv_rz((float)r, (float)w);
    if (q * w > r) q--;
    else if ((q + 1u) * w <= r) q++;
    return q;
}

// Keys of a chunk of 2048 list positions, in four rounds of 512 (one
// position per thread). Per round a block scan gives every position its key
// slot; then each warp writes the keys of its 32 consecutive positions
// together: lane j takes the warp's keys j, j + 32, ... (coalesced stores),
// finds the position that owns key j by a 5-step search over the lanes'
// offsets (shuffles), and the tile from the key's rank in that position's
// row-major tile rectangle.
// hist (32-bit keys only, nullable): digit histograms of the written keys for
// the radix sort that follows (key_bits significant bits).
template <typename KeyT>
__global__ void __launch_bounds__(kBinThreads) bin_duplicate_kernel(
    const uint32_t* __restrict__ tiles_touched, const ushort4* __restrict__ rect, const float* __restrict__ depth,
    const uint32_t* __restrict__ order, int64_t n, int tiles_x, const unsigned long long* __restrict__ block_prefix,
    int64_t key_capacity, uint32_t* __restrict__ offsets, KeyT* __restrict__ keys, uint32_t* __restrict__ vals,
    uint32_t* __restrict__ hist, int key_bits) {
    grid_dependency_begin();
    __shared__ uint32_t s_dhist[kHistPasses * 256];
    __shared__ unsigned long long warp_tot[kBinThreads / 32];
    __shared__ unsigned long long total;

    const int lane = threadIdx.x & 31;
    if (hist)
        for (int i = threadIdx.x; i < kHistPasses * 256; i += kBinThreads) s_dhist[i] = 0;
    const int64_t chunk0 = (int64_t)blockIdx.x * kBinChunk;
    unsigned long long carry = block_prefix[blockIdx.x];   // key slot of the chunk's first key

    for (int round = 0; round < kBinItems; round++) {
        const int64_t pos = chunk0 + (int64_t)round * kBinThreads + threadIdx.x;
        const bool in = pos < n;
        const uint32_t g = in ? at(order, pos) : 0u;
        const uint32_t t = in ? __ldg(tiles_touched + g) : 0u;
        ushort4 r = make_ushort4(0, 0, 0, 0);
        uint32_t db = 0;
        if (t) {
            r = __ldg(rect + g);
            if (sizeof(KeyT) == 8) db = __float_as_uint(__ldg(depth + g));
        }
        const unsigned long long incl = block_scan_incl((unsigned long long)t, warp_tot, &total);
        const unsigned long long first = carry + incl - t;   // global slot of this position's first key
        if (in && offsets) offsets[pos] = (uint32_t)(carry + incl);

        // keys of this warp's 32 positions, relative to the warp's first key
        const unsigned long long wbase = __shfl_sync(0xffffffffu, first, 0);
        const uint32_t rel_excl = (uint32_t)(first - wbase);            // < 2^32 for any sane input
        const uint32_t wcount = __shfl_sync(0xffffffffu, (uint32_t)(first - wbase) + t, 31);
        const uint32_t w_rect = (uint32_t)r.z - r.x + 1u;
        const uint32_t packed_xy = (uint32_t)r.x | ((uint32_t)r.y << 16);
        for (uint32_t j0 = 0; j0 < wcount; j0 += 32) {
            const uint32_t j = j0 + lane;
            // owner: the last lane whose first key is <= j
            int owner = 0;
#pragma unroll
            for (int step = 16; step >= 1; step >>= 1) {
                const uint32_t cand_first = __shfl_sync(0xffffffffu, rel_excl, owner + step);
                if (cand_first <= j) owner += step;
            }
            const uint32_t o_first = __shfl_sync(0xffffffffu, rel_excl, owner);
            const uint32_t o_w = __shfl_sync(0xffffffffu, w_rect, owner);
            const uint32_t o_xy = __shfl_sync(0xffffffffu, packed_xy, owner);
            const uint32_t o_g = __shfl_sync(0xffffffffu, g, owner);
            const uint32_t o_db = __shfl_sync(0xffffffffu, db, owner);
            const unsigned long long slot = wbase + j;
            if (j < wcount && (long long)slot < key_capacity) {
                const uint32_t rank = j - o_first;
                const uint32_t dy = div_small(rank, o_w);
                const uint32_t tx = (o_xy & 0xffffu) + (rank - dy * o_w), ty = (o_xy >> 16) + dy;
                const uint64_t tile = (uint64_t)ty * (uint64_t)tiles_x + tx;
                if (sizeof(KeyT) == 8) {
                    keys[slot] = (KeyT)((tile << 32) | o_db);
                } else {
                    keys[slot] = (KeyT)tile;
                    if (hist) count_digits(s_dhist, (uint32_t)tile, key_bits);
                }
                vals[slot] = o_g;
            }
        }
        carry += total;
        __syncthreads();   // warp_tot and total are reused by the next round's scan
    }
    if (hist) {
        __syncthreads();
        flush_digits(s_dhist, hist, key_bits);
    }
}

// ---------------------------------------------------------------- key-balanced expansion
// Used for a given order (the depth order). A chunk of Gaussians can hold
// wildly different numbers of keys (in depth order the many-tile Gaussians of
// one dense region sit together), so the expansion is balanced by keys: one
// block per kKeysPerBlock key slots.
//   bin_offsets_kernel : each position's first key slot (exclusive prefix), and
//                        for every block boundary k * kKeysPerBlock the position
//                        that owns that slot.
//   bin_expand_kernel  : block k writes slots [k, k + 1) * kKeysPerBlock; it
//                        loads the positions from the owner of its first slot
//                        on, and finds each slot's position by binary search.
constexpr int kKeysPerBlock = 2048;
constexpr int kExpandThreads = 256;
constexpr int kWindow = 1024;   // positions staged per step

// Rectangles in list order (coalesced reads for the three kernels below); a
// Gaussian without tiles gets the marker x0 = 0xffff. The list is the given
// order, or the index order when order is null.
__global__ void gather_rect_kernel(const uint32_t* __restrict__ tiles_touched, const ushort4* __restrict__ rect,
                                   const uint32_t* __restrict__ order, int64_t n, ushort4* __restrict__ rs) {
    grid_dependency_begin();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t g = at(order, i);
        // an index outside the scene can only come from a depth sort that was
        // cut short (flagged): no tiles, never a read past the arrays
        GS_CHECK(g < n);
        rs[i] = (g < n && __ldg(tiles_touched + g)) ? __ldg(rect + g) : make_ushort4(0xffff, 0, 0, 0);
    }
}

__device__ __forceinline__ uint32_t rect_tiles(const ushort4 r) {
    return r.x == 0xffff ? 0u : ((uint32_t)r.z - r.x + 1u) * ((uint32_t)r.w - r.y + 1u);
}

__global__ void __launch_bounds__(kBinThreads) bin_reduce_rect_kernel(const ushort4* __restrict__ rs, int64_t n,
                                                                      unsigned long long* __restrict__ block_sums) {
    grid_dependency_begin();
    __shared__ unsigned long long warp_tot[kBinThreads / 32];
    __shared__ unsigned long long total;
    const int64_t base = (int64_t)blockIdx.x * kBinChunk + (int64_t)threadIdx.x * kBinItems;
    unsigned long long s = 0;
#pragma unroll
    for (int i = 0; i < kBinItems; i++)
        if (base + i < n) s += rect_tiles(__ldg(rs + base + i));
    block_scan_incl(s, warp_tot, &total);
    if (threadIdx.x == 0) block_sums[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kBinThreads) bin_offsets_kernel(
    const ushort4* __restrict__ rs, int64_t n,
    const unsigned long long* __restrict__ block_prefix, int64_t key_capacity, uint32_t* __restrict__ first_slot,
    uint32_t* __restrict__ owner, uint32_t* __restrict__ offsets) {
    grid_dependency_begin();
    __shared__ unsigned long long warp_tot[kBinThreads / 32];
    __shared__ unsigned long long total;
    const int64_t chunk0 = (int64_t)blockIdx.x * kBinChunk;
    unsigned long long carry = block_prefix[blockIdx.x];
    for (int round = 0; round < kBinItems; round++) {
        const int64_t pos = chunk0 + (int64_t)round * kBinThreads + threadIdx.x;
        const bool in = pos < n;
        const uint32_t t = in ? rect_tiles(__ldg(rs + pos)) : 0u;
        const unsigned long long incl = block_scan_incl((unsigned long long)t, warp_tot, &total);
        const unsigned long long first = carry + incl - t;
        if (in) {
            first_slot[pos] = first < 0xffffffffull ? (uint32_t)first : 0xffffffffu;
            if (offsets) offsets[pos] = (uint32_t)(carry + incl);
            if (t) {
                const unsigned long long last = first + t - 1;
                const unsigned long long lim = (unsigned long long)key_capacity;
                for (unsigned long long k = (first + kKeysPerBlock - 1) / kKeysPerBlock;
                     k * kKeysPerBlock <= last && k * kKeysPerBlock < lim; k++)
                    owner[k] = (uint32_t)pos;
            }
        }
        carry += total;
        __syncthreads();
    }
}

// hist (nullable): digit histograms of the written tile keys (key_bits bits).
// Each thread owns kRun consecutive slots of the block's range: one binary
// search for the position owning its first slot, then a walk along that
// position's tile rectangle (and on to the next positions). Keys go through
// shared memory so that the global stores are coalesced.
constexpr int kRun = kKeysPerBlock / kExpandThreads;   // 8 slots per thread
__global__ void __launch_bounds__(kExpandThreads) bin_expand_kernel(
    const ushort4* __restrict__ rs, const uint32_t* __restrict__ order, int64_t n, const TileKeyMap km,
    const uint32_t* __restrict__ first_slot, const uint32_t* __restrict__ owner,
    const uint64_t* __restrict__ num_keys, int64_t key_capacity, uint32_t* __restrict__ keys,
    uint32_t* __restrict__ vals, uint32_t* __restrict__ hist, int key_bits) {
    grid_dependency_begin();
    __shared__ uint32_t s_first[kWindow];
    __shared__ ushort4 s_rect[kWindow];
    __shared__ uint32_t s_g[kWindow];
    // staged keys, one padding word per 32 so that the per-thread runs of 8
    // (stride-8 writes across a warp) fall in distinct banks
    __shared__ uint32_t s_key[kKeysPerBlock + kKeysPerBlock / 32];
    __shared__ uint32_t s_val[kKeysPerBlock + kKeysPerBlock / 32];
    __shared__ uint32_t s_dhist[kHistPasses * 256];
    __shared__ uint32_t s_end;

    const unsigned long long K = *num_keys;
    const unsigned long long Keff = K < (unsigned long long)key_capacity ? K : (unsigned long long)key_capacity;
    const unsigned long long S0 = (unsigned long long)blockIdx.x * kKeysPerBlock;
    if (S0 >= Keff) return;
    const unsigned long long S1 = S0 + kKeysPerBlock < Keff ? S0 + kKeysPerBlock : Keff;
    if (hist)
        for (int i = threadIdx.x; i < kHistPasses * 256; i += kExpandThreads) s_dhist[i] = 0;
    // each digit is counted per run of consecutive keys with the same value of
    // that digit (one shared atomic per run): along a rectangle's row the
    // identity layout's high digits and the block layout's low digit repeat
    const int passes = digit_passes(key_bits);
    const unsigned long long r0 = S0 + (unsigned long long)threadIdx.x * kRun;   // this thread's slots
    const unsigned long long r1 = r0 + kRun < S1 ? r0 + kRun : S1;

    int64_t p = owner[blockIdx.x];
    const int64_t p_last = S1 < Keff ? (int64_t)owner[blockIdx.x + 1] : n - 1;
    while (true) {
        __syncthreads();
        int64_t wn = p_last - p + 1;
        wn = wn < kWindow ? wn : kWindow;
        wn = wn < n - p ? wn : n - p;
        for (int i = threadIdx.x; i < wn; i += kExpandThreads) {
            s_first[i] = __ldg(first_slot + p + i);
            s_g[i] = at(order, p + i);
            s_rect[i] = __ldg(rs + p + i);
        }
        if (threadIdx.x == 0)
            s_end = p + wn < n ? __ldg(first_slot + p + wn) : (uint32_t)(K < 0xffffffffull ? K : 0xffffffffull);
        __syncthreads();
        // this thread's slots that this window owns
        const unsigned long long a0 = r0 > (unsigned long long)s_first[0] ? r0 : (unsigned long long)s_first[0];
        const unsigned long long a1 = r1 < (unsigned long long)s_end ? r1 : (unsigned long long)s_end;
        if (a0 < a1) {
            int lo = 0, hi = (int)wn - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_first[mid] <= a0) lo = mid; else hi = mid - 1;
            }
            ushort4 r = s_rect[lo];
            uint32_t w = (uint32_t)r.z - r.x + 1u;
            uint32_t rank = (uint32_t)(a0 - s_first[lo]);
            uint32_t dy = div_small(rank, w);
            uint32_t ty = r.y + dy, tx = r.x + (rank - dy * w);
            uint32_t run_d[kHistPasses], run_n[kHistPasses];
#pragma unroll
            for (int q = 0; q < kHistPasses; q++) {
                run_d[q] = 0xffffffffu;
                run_n[q] = 0;
            }
            for (unsigned long long j = a0; j < a1; j++) {
                // step to the next position once this one's tiles are used up
                while (lo + 1 < wn && s_first[lo + 1] <= j) {
                    lo++;
                    r = s_rect[lo];
                    w = (uint32_t)r.z - r.x + 1u;
                    tx = r.x;
                    ty = r.y;
                }
                const uint32_t tile = tile_key(km, tx, ty);
                const uint32_t si = (uint32_t)(j - S0);
                GS_CHECK(si < (uint32_t)kKeysPerBlock && j < (unsigned long long)key_capacity && tx <= r.z);
                s_key[si + (si >> 5)] = tile;
                s_val[si + (si >> 5)] = s_g[lo];
                if (hist) {
#pragma unroll
                    for (int q = 0; q < kHistPasses; q++) {
                        if (q < passes) {
                            const uint32_t d = digit(tile, key_bits, q);
                            if (d != run_d[q]) {
                                if (run_n[q]) atomicAdd(&s_dhist[q * 256 + run_d[q]], run_n[q]);
                                run_d[q] = d;
                                run_n[q] = 0;
                            }
                            run_n[q]++;
                        }
                    }
                }
                if (++tx > r.z) {
                    tx = r.x;
                    ty++;
                }
            }
            if (hist) {
#pragma unroll
                for (int q = 0; q < kHistPasses; q++)
                    if (q < passes && run_n[q]) atomicAdd(&s_dhist[q * 256 + run_d[q]], run_n[q]);
            }
        }
        if (s_end >= S1 || p + wn >= n) break;
        p += wn;
    }
    __syncthreads();
    const int cnt = (int)(S1 - S0);
    for (int i = threadIdx.x; i < cnt; i += kExpandThreads) {
        keys[S0 + i] = s_key[i + (i >> 5)];
        vals[S0 + i] = s_val[i + (i >> 5)];
    }
    if (hist) flush_digits(s_dhist, hist, key_bits);
}

// Depth-order sort input: key = depth bits for Gaussians with tiles (depth >
// near > 0, so the bits order like the depths), 0xffffffff for the others
// (sorted last); value = index.
__global__ void __launch_bounds__(256) depth_keys_kernel(const float* __restrict__ depth,
                                                         const uint32_t* __restrict__ tiles_touched, int64_t n,
                                                         uint32_t* __restrict__ keys, uint32_t* __restrict__ vals,
                                                         uint32_t* __restrict__ hist) {
    grid_dependency_begin();
    __shared__ uint32_t s_dhist[kHistPasses * 256];
    if (hist)
        for (int i = threadIdx.x; i < kHistPasses * 256; i += blockDim.x) s_dhist[i] = 0;
    __syncthreads();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t k = __ldg(tiles_touched + i) ? __float_as_uint(__ldg(depth + i)) : 0xffffffffu;
        keys[i] = k;
        vals[i] = (uint32_t)i;
        if (hist) count_digits(s_dhist, k, 32);
    }
    if (hist) {
        __syncthreads();
        flush_digits(s_dhist, hist, 32);
    }
}

}  // namespace

size_t bin_scratch_bytes(int64_t n) {
    const int64_t nb = (n + kBinChunk - 1) / kBinChunk;
    return align_up((size_t)(nb > 0 ? nb : 1) * sizeof(unsigned long long));
}

template <typename KeyT>
cudaError_t launch_bin_t(const gs_projected& p, const uint32_t* order, int64_t n, const CamConst& cam,
                         uint32_t* offsets, KeyT* keys, uint32_t* vals, int64_t key_capacity, uint64_t* num_keys,
                         StatusHeader* status, void* scratch, cudaStream_t s, uint32_t* hist = nullptr,
                         int key_bits = 0) {
    if (n == 0) {
        cudaError_t e = cudaMemsetAsync(num_keys, 0, sizeof(uint64_t), s);
        if (e != cudaSuccess) return e;
        return cudaMemsetAsync(&status->num_keys, 0, sizeof(unsigned long long), s);
    }
    const int nb = (int)((n + kBinChunk - 1) / kBinChunk);
    auto* sums = static_cast<unsigned long long*>(scratch);
    launch_k(bin_reduce_kernel, nb, kBinThreads, 0, s, p.tiles_touched, order, n, sums);
    launch_k(bin_scan_sums_kernel, 1, 1024, 0, s, sums, nb, key_capacity, num_keys, status);
    launch_k(bin_duplicate_kernel<KeyT>, nb, kBinThreads, 0, s, p.tiles_touched,
             reinterpret_cast<const ushort4*>(p.rect), p.depth, order, n, cam.tiles_x, sums, key_capacity, offsets,
             keys, vals, hist, key_bits);
    return cudaGetLastError();
}

cudaError_t launch_bin(const gs_projected& p, int64_t n, const CamConst& cam, uint32_t* offsets, uint64_t* keys,
                       uint32_t* vals, int64_t key_capacity, uint64_t* num_keys, StatusHeader* status,
                       void* scratch, cudaStream_t s) {
    return launch_bin_t<uint64_t>(p, nullptr, n, cam, offsets, keys, vals, key_capacity, num_keys, status, scratch,
                                  s);
}

size_t bin_ordered_scratch_bytes(int64_t n, int64_t key_capacity) {
    const size_t un = (size_t)(n > 0 ? n : 0);
    const size_t blocks = (size_t)((key_capacity > 0 ? key_capacity : 0) + kKeysPerBlock - 1) / kKeysPerBlock + 1;
    return bin_scratch_bytes(n) + align_up(4 * un) + align_up(4 * blocks) + align_up(8 * un);
}

cudaError_t launch_bin_ordered(const gs_projected& p, const uint32_t* order, int64_t n, const CamConst& cam,
                               uint32_t* offsets, uint32_t* tile_keys, uint32_t* vals, int64_t key_capacity,
                               uint64_t* num_keys, StatusHeader* status, void* scratch, cudaStream_t s,
                               uint32_t* hist, int key_bits, const TileKeyMap* keymap) {
    const TileKeyMap km = keymap ? *keymap : identity_keys(cam.tiles_x);
    if (n == 0) {
        cudaError_t e = cudaMemsetAsync(num_keys, 0, sizeof(uint64_t), s);
        if (e != cudaSuccess) return e;
        return cudaMemsetAsync(&status->num_keys, 0, sizeof(unsigned long long), s);
    }
    const int nb = (int)((n + kBinChunk - 1) / kBinChunk);
    char* w = static_cast<char*>(scratch);
    auto* sums = reinterpret_cast<unsigned long long*>(w);
    auto* first_slot = reinterpret_cast<uint32_t*>(w + bin_scratch_bytes(n));
    const size_t blocks_b = (size_t)((key_capacity > 0 ? key_capacity : 0) + kKeysPerBlock - 1) / kKeysPerBlock + 1;
    auto* owner = reinterpret_cast<uint32_t*>(w + bin_scratch_bytes(n) + align_up(4 * (size_t)n));
    auto* rs = reinterpret_cast<ushort4*>(w + bin_scratch_bytes(n) + align_up(4 * (size_t)n) + align_up(4 * blocks_b));
    const int64_t gb = (n + 255) / 256;
    launch_k(gather_rect_kernel, (unsigned)(gb < 148 * 16 ? gb : 148 * 16), 256, 0, s,
             p.tiles_touched, reinterpret_cast<const ushort4*>(p.rect), order, n, rs);
    launch_k(bin_reduce_rect_kernel, nb, kBinThreads, 0, s, rs, n, sums);
    launch_k(bin_scan_sums_kernel, 1, 1024, 0, s, sums, nb, key_capacity, num_keys, status);
    launch_k(bin_offsets_kernel, nb, kBinThreads, 0, s, rs, n, sums, key_capacity, first_slot, owner, offsets);
    if (key_capacity > 0) {
        const unsigned blocks = (unsigned)((key_capacity + kKeysPerBlock - 1) / kKeysPerBlock);
        launch_k(bin_expand_kernel, blocks, kExpandThreads, 0, s, rs, order, n, km, first_slot, owner,
                 num_keys, key_capacity, tile_keys, vals, hist, key_bits);
    }
    return cudaGetLastError();
}

cudaError_t launch_depth_keys(const gs_projected& p, int64_t n, uint32_t* keys, uint32_t* vals, uint32_t* hist,
                              cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    int64_t b = (n + 1023) / 1024;
    launch_k(depth_keys_kernel, (unsigned)(b < 148 * 4 ? b : 148 * 4), 256, 0, s, p.depth, p.tiles_touched, n, keys,
             vals, hist);
    return cudaGetLastError();
}

GS_DEFINE_CHECK_SETTER(binning)

}  // namespace gs
