// Densification and pruning of the Gaussian set, as device compaction.
//
// Method: lesson page "3D Gaussian Splatting à partir de zéro", section
// "Densation et taille": every N iterations,
//   clone  a Gaussian whose gradient magnitude is high but whose scale is
//          small (a copy at its current position),
//   split  a large Gaussian whose gradient is high into two smaller ones,
//   prune  Gaussians whose opacity fell below a threshold.
// The gradient magnitude is the norm of the image-space mean gradient
// dL/d(u, v), averaged over the iterations in which the Gaussian touched a
// tile (densify_stats_kernel accumulates it). "Small" and "large" compare the
// largest scale with a threshold. A split child sits at mu + R S xi for a
// caller-given standard normal xi (one per child) and has its scales divided
// by 1.6; a clone is an exact copy placed right after its original.
//
// The decisions are integer results, taken in binary32 on values both sides
// compute identically: the opacity test is logit < logit_threshold and the
// scale test is max(log_scale) > log_scale_threshold, with both thresholds
// mapped by the caller (o < t iff logit < log(t / (1 - t)); max s > t iff
// max log s > log t); the gradient test is (accum / count) >= threshold with
// a correctly rounded division. Output order is stable: survivors keep the
// input order, children replace their parent, clones follow their original.
#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kDensThreads = 256;

__global__ void __launch_bounds__(256) densify_stats_kernel(const float2* __restrict__ grad_mean2d,
                                                            const uint32_t* __restrict__ tiles_touched, int64_t n,
                                                            float* __restrict__ accum, uint32_t* __restrict__ count) {
    grid_dependency_begin();
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n || tiles_touched[g] == 0) return;
    const float2 d = grad_mean2d[g];
    accum[g] += sqrtf(d.x * d.x + d.y * d.y);
    count[g] += 1u;
}

struct DensArgs {
    gs_gaussians in;
    gs_gaussians_out out;
    int64_t capacity;
    const float* accum;
    const uint32_t* count;
    const float* xi;           // [n][2][3]
    float grad_threshold;
    float log_scale_threshold;
    float logit_threshold;
    uint8_t* action;           // [n] nullable
    uint32_t* slots;           // [n] output slots per Gaussian (0, 1 or 2)
    unsigned long long* block_sums;
    unsigned long long* total;
    StatusHeader* header;
};

// 0 keep, 1 clone, 2 split, 3 prune
__device__ __forceinline__ int decide(const DensArgs& a, int64_t g) {
    if (a.in.opacity_logits[g] < a.logit_threshold) return 3;
    const uint32_t c = a.count[g];
    if (c == 0) return 0;
    const float avg = __fdiv_rn(a.accum[g], (float)c);
    if (!(avg >= a.grad_threshold)) return 0;
    const float* ls = a.in.log_scales + 3 * g;
    const float m = fmaxf(fmaxf(ls[0], ls[1]), ls[2]);
    return m > a.log_scale_threshold ? 2 : 1;
}

// per block: slot counts and their block total
__global__ void __launch_bounds__(kDensThreads) densify_count_kernel(const DensArgs a) {
    grid_dependency_begin();
    __shared__ unsigned long long s_sum;
    if (threadIdx.x == 0) s_sum = 0;
    __syncthreads();
    const int64_t g = (int64_t)blockIdx.x * kDensThreads + threadIdx.x;
    uint32_t slots = 0;
    if (g < a.in.n) {
        const int act = decide(a, g);
        if (a.action) a.action[g] = (uint8_t)act;
        slots = act == 3 ? 0u : (act == 0 ? 1u : 2u);
        a.slots[g] = slots;
    }
    const uint32_t ws = __reduce_add_sync(0xffffffffu, slots);
    if ((threadIdx.x & 31) == 0 && ws) atomicAdd(&s_sum, (unsigned long long)ws);
    __syncthreads();
    if (threadIdx.x == 0) a.block_sums[blockIdx.x] = s_sum;
}

// exclusive scan of the block totals (one block), the new count and the
// capacity flag
__global__ void __launch_bounds__(1024) densify_scan_kernel(const DensArgs a, int nb) {
    grid_dependency_begin();
    __shared__ unsigned long long s_carry;
    __shared__ unsigned long long s_warp[32];
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int base = 0; base < nb; base += 1024) {
        const int i = base + threadIdx.x;
        const unsigned long long v = i < nb ? a.block_sums[i] : 0ull;
        unsigned long long x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp[w] = x;
        __syncthreads();
        if (w == 0) {
            unsigned long long t = s_warp[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            s_warp[lane] = t;
        }
        __syncthreads();
        const unsigned long long incl = x + (w > 0 ? s_warp[w - 1] : 0ull);
        if (i < nb) a.block_sums[i] = s_carry + incl - v;
        __syncthreads();
        if (threadIdx.x == 1023) s_carry += incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *a.total = s_carry;
        if (s_carry > (unsigned long long)a.capacity) atomicOr(&a.header->flags, (unsigned)GS_FLAG_CAPACITY);
        a.header->num_keys = s_carry;
    }
}

// scatter: block offset + rank inside the block; then each warp copies its
// 32 Gaussians one after another with all lanes (coalesced rows), and the
// owner of a split Gaussian writes its children's centres and scales
__global__ void __launch_bounds__(kDensThreads) densify_scatter_kernel(const DensArgs a) {
    grid_dependency_begin();
    __shared__ uint32_t s_warp[kDensThreads / 32];
    const int64_t g = (int64_t)blockIdx.x * kDensThreads + threadIdx.x;
    const uint32_t slots = g < a.in.n ? a.slots[g] : 0u;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t x = slots;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    uint32_t before = 0;
    for (int i = 0; i < w; i++) before += s_warp[i];
    const unsigned long long o = a.block_sums[blockIdx.x] + before + x - slots;
    const bool fits = slots > 0 && o + slots <= (unsigned long long)a.capacity;   // overflow is flagged by the scan
    const int nk3 = (a.in.sh_degree + 1) * (a.in.sh_degree + 1) * 3;
    const int64_t gw = g - lane;   // the warp's first Gaussian
    uint32_t todo = __ballot_sync(0xffffffffu, fits);
    while (todo) {
        const int j = __ffs(todo) - 1;
        todo &= todo - 1;
        const int64_t gj = gw + j;
        const int64_t oj = (int64_t)__shfl_sync(0xffffffffu, (unsigned long long)o, j);
        const uint32_t sj = __shfl_sync(0xffffffffu, slots, j);
        for (uint32_t c = 0; c < sj; c++) {
            const int64_t oc = oj + c;
            for (int k = lane; k < nk3; k += 32) a.out.sh[(int64_t)nk3 * oc + k] = a.in.sh[(int64_t)nk3 * gj + k];
            if (lane < 3) a.out.means[3 * oc + lane] = a.in.means[3 * gj + lane];
            else if (lane < 7) a.out.quats[4 * oc + lane - 3] = a.in.quats[4 * gj + lane - 3];
            else if (lane < 10) a.out.log_scales[3 * oc + lane - 7] = a.in.log_scales[3 * gj + lane - 7];
            else if (lane == 10) a.out.opacity_logits[oc] = a.in.opacity_logits[gj];
        }
    }
    __syncwarp();
    if (!fits || slots == 1) return;
    const float* ls = a.in.log_scales + 3 * g;
    const float m = fmaxf(fmaxf(ls[0], ls[1]), ls[2]);
    if (!(m > a.log_scale_threshold)) return;   // clone: two identical copies
    // split: children at mu + R S xi_c, scales / 1.6
    const float* q = a.in.quats + 4 * g;
    const float qn = rsqrtf(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
    const float w0 = q[0] * qn, x0 = q[1] * qn, y0 = q[2] * qn, z0 = q[3] * qn;
    const float R[9] = {1.f - 2.f * (y0 * y0 + z0 * z0), 2.f * (x0 * y0 - w0 * z0), 2.f * (x0 * z0 + w0 * y0),
                        2.f * (x0 * y0 + w0 * z0), 1.f - 2.f * (x0 * x0 + z0 * z0), 2.f * (y0 * z0 - w0 * x0),
                        2.f * (x0 * z0 - w0 * y0), 2.f * (y0 * z0 + w0 * x0), 1.f - 2.f * (x0 * x0 + y0 * y0)};
    const float sc[3] = {expf(ls[0]), expf(ls[1]), expf(ls[2])};
    constexpr float kLog16 = 0.47000362924573558f;   // log(1.6)
    for (int c = 0; c < 2; c++) {
        const float* e = a.xi + 6 * g + 3 * c;
        const int64_t oc = (int64_t)o + c;
        for (int i = 0; i < 3; i++)
            a.out.means[3 * oc + i] = a.in.means[3 * g + i] + R[3 * i] * sc[0] * e[0] + R[3 * i + 1] * sc[1] * e[1] +
                                      R[3 * i + 2] * sc[2] * e[2];
        for (int i = 0; i < 3; i++) a.out.log_scales[3 * oc + i] = ls[i] - kLog16;
    }
}

}  // namespace

size_t densify_scratch_bytes(int64_t n) {
    const size_t nb = (size_t)((n + kDensThreads - 1) / kDensThreads) + 1;
    return align_up(sizeof(StatusHeader)) + align_up(4 * (size_t)(n > 0 ? n : 1)) + align_up(8 * nb) + align_up(8);
}

cudaError_t launch_densify_stats(const float* grad_mean2d, const uint32_t* tiles_touched, int64_t n, float* accum,
                                 uint32_t* count, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    launch_k(densify_stats_kernel, (unsigned)((n + 255) / 256), 256, 0, s, reinterpret_cast<const float2*>(grad_mean2d),
             tiles_touched, n, accum, count);
    return cudaGetLastError();
}

cudaError_t launch_densify(const gs_gaussians& in, const gs_gaussians_out& out, int64_t capacity, const float* accum,
                           const uint32_t* count, const float* xi, float grad_threshold, float log_scale_threshold,
                           float logit_threshold, uint8_t* action, uint64_t* out_count, void* scratch,
                           cudaStream_t s) {
    char* w = static_cast<char*>(scratch);
    DensArgs a;
    a.in = in;
    a.out = out;
    a.capacity = capacity;
    a.accum = accum;
    a.count = count;
    a.xi = xi;
    a.grad_threshold = grad_threshold;
    a.log_scale_threshold = log_scale_threshold;
    a.logit_threshold = logit_threshold;
    a.action = action;
    a.header = reinterpret_cast<StatusHeader*>(w);
    a.slots = reinterpret_cast<uint32_t*>(w + align_up(sizeof(StatusHeader)));
    const int nb = (int)((in.n + kDensThreads - 1) / kDensThreads);
    a.block_sums = reinterpret_cast<unsigned long long*>(w + align_up(sizeof(StatusHeader)) +
                                                          align_up(4 * (size_t)(in.n > 0 ? in.n : 1)));
    a.total = reinterpret_cast<unsigned long long*>(out_count);
    cudaError_t e = cudaMemsetAsync(a.header, 0, sizeof(StatusHeader), s);
    if (e != cudaSuccess) return e;
    if (in.n == 0) return cudaMemsetAsync(out_count, 0, sizeof(uint64_t), s);
    launch_k(densify_count_kernel, nb, kDensThreads, 0, s, a);
    launch_k(densify_scan_kernel, 1, 1024, 0, s, a, nb);
    launch_k(densify_scatter_kernel, nb, kDensThreads, 0, s, a);
    return cudaGetLastError();
}

GS_DEFINE_CHECK_SETTER(densify)

}  // namespace gs
