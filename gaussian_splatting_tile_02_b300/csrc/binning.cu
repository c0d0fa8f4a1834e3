// Step 2 of the forward renderer: tile binning (flowchart box "Assign to
// tiles (16x16 screen-space)" on the lesson page "3D Gaussian Splatting à
// partir de zéro", section "Rastérisation, non rayée").
//
// A device prefix scan over tiles_touched gives each Gaussian the slot of its
// first key and the frame's key count K; the Gaussian's keys are then written
// in row-major order over its tile rectangle:
//     key = (uint64)(ty * tiles_x + tx) << 32 | float_bits(depth),  value = index.
//
// Three kernels: a per-chunk reduction (2048 Gaussians per block), a
// single-block scan of the chunk sums (which also publishes K), and the
// duplication, which re-scans its chunk in shared memory and then writes the
// chunk's keys load-balanced: consecutive threads write consecutive key slots
// (coalesced 8- and 4-byte stores) and find their Gaussian by binary search
// over the chunk's inclusive offsets, so a Gaussian with many tiles does not
// serialise one thread.
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

__global__ void __launch_bounds__(kBinThreads) bin_reduce_kernel(const uint32_t* __restrict__ tiles_touched, int64_t n,
                                                                 unsigned long long* __restrict__ block_sums) {
    __shared__ unsigned long long warp_tot[kBinThreads / 32];
    __shared__ unsigned long long total;
    const int64_t base = (int64_t)blockIdx.x * kBinChunk + (int64_t)threadIdx.x * kBinItems;
    unsigned long long s = 0;
#pragma unroll
    for (int i = 0; i < kBinItems; i++)
        if (base + i < n) s += __ldg(tiles_touched + base + i);
    block_scan_incl(s, warp_tot, &total);
    if (threadIdx.x == 0) block_sums[blockIdx.x] = total;
}

// Exclusive scan of the chunk sums in place; K = total.
__global__ void __launch_bounds__(1024) bin_scan_sums_kernel(unsigned long long* __restrict__ sums, int nb,
                                                             int64_t key_capacity, uint64_t* __restrict__ num_keys,
                                                             StatusHeader* __restrict__ status) {
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

__global__ void __launch_bounds__(kBinThreads) bin_duplicate_kernel(
    const uint32_t* __restrict__ tiles_touched, const ushort4* __restrict__ rect, const float* __restrict__ depth,
    int64_t n, int tiles_x, const unsigned long long* __restrict__ block_prefix, int64_t key_capacity,
    uint32_t* __restrict__ offsets, uint64_t* __restrict__ keys, uint32_t* __restrict__ vals) {
    __shared__ unsigned long long s_incl[kBinChunk];
    __shared__ ushort4 s_rect[kBinChunk];
    __shared__ uint32_t s_depth[kBinChunk];
    __shared__ unsigned long long warp_tot[kBinThreads / 32];
    __shared__ unsigned long long total;

    const int64_t chunk0 = (int64_t)blockIdx.x * kBinChunk;
    const int64_t base = chunk0 + (int64_t)threadIdx.x * kBinItems;
    uint32_t t[kBinItems];
    unsigned long long s = 0;
#pragma unroll
    for (int i = 0; i < kBinItems; i++) {
        t[i] = base + i < n ? __ldg(tiles_touched + base + i) : 0u;
        s += t[i];
    }
    const unsigned long long incl = block_scan_incl(s, warp_tot, &total);
    const unsigned long long prefix = block_prefix[blockIdx.x];
    unsigned long long run = incl - s;
#pragma unroll
    for (int i = 0; i < kBinItems; i++) {
        run += t[i];
        const int li = threadIdx.x * kBinItems + i;
        s_incl[li] = run;
        if (base + i < n) {
            offsets[base + i] = (uint32_t)(prefix + run);
            if (t[i]) {
                s_rect[li] = __ldg(rect + base + i);
                s_depth[li] = __float_as_uint(__ldg(depth + base + i));
            }
        }
    }
    __syncthreads();
    if ((long long)prefix >= key_capacity) return;
    const unsigned long long room = (unsigned long long)key_capacity - prefix;
    const unsigned long long limit = total < room ? total : room;
    for (unsigned long long j = threadIdx.x; j < limit; j += kBinThreads) {
        // first chunk slot whose inclusive offset exceeds j
        int lo = 0, hi = kBinChunk - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (s_incl[mid] > j) hi = mid; else lo = mid + 1;
        }
        const unsigned long long first = lo > 0 ? s_incl[lo - 1] : 0ull;
        const uint32_t rank = (uint32_t)(j - first);
        const ushort4 r = s_rect[lo];
        const uint32_t w = (uint32_t)r.z - r.x + 1u;
        const uint32_t ty = r.y + rank / w, tx = r.x + rank % w;
        const uint64_t tile = (uint64_t)ty * (uint64_t)tiles_x + tx;
        keys[prefix + j] = (tile << 32) | s_depth[lo];
        vals[prefix + j] = (uint32_t)(chunk0 + lo);
    }
}

}  // namespace

size_t bin_scratch_bytes(int64_t n) {
    const int64_t nb = (n + kBinChunk - 1) / kBinChunk;
    return align_up((size_t)(nb > 0 ? nb : 1) * sizeof(unsigned long long));
}

cudaError_t launch_bin(const gs_projected& p, int64_t n, const CamConst& cam, uint32_t* offsets,
                       uint64_t* keys, uint32_t* vals, int64_t key_capacity, uint64_t* num_keys,
                       StatusHeader* status, void* scratch, cudaStream_t s) {
    if (n == 0) {
        cudaError_t e = cudaMemsetAsync(num_keys, 0, sizeof(uint64_t), s);
        if (e != cudaSuccess) return e;
        return cudaMemsetAsync(&status->num_keys, 0, sizeof(unsigned long long), s);
    }
    const int nb = (int)((n + kBinChunk - 1) / kBinChunk);
    auto* sums = static_cast<unsigned long long*>(scratch);
    bin_reduce_kernel<<<nb, kBinThreads, 0, s>>>(p.tiles_touched, n, sums);
    bin_scan_sums_kernel<<<1, 1024, 0, s>>>(sums, nb, key_capacity, num_keys, status);
    bin_duplicate_kernel<<<nb, kBinThreads, 0, s>>>(p.tiles_touched, reinterpret_cast<const ushort4*>(p.rect),
                                                    p.depth, n, cam.tiles_x, sums, key_capacity, offsets, keys,
                                                    vals);
    return cudaGetLastError();
}

}  // namespace gs
