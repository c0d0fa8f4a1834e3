// gs_bin_static: tile binning that allocates nothing.
//
// Some callers cannot allocate device memory: plugins whose host application
// hands out GPU memory only through its own pools and forbids allocations
// by third-party libraries, and real-time render loops that ban cudaMalloc
// after start-up because it can synchronise the device and stall a frame.
// For them this entry point runs the same binning kernels as gs_bin, with
// the scratch those kernels need (a 256-byte status header and one 64-bit
// partial sum per 2048 Gaussians) kept in a file-scope device array instead
// of a caller-provided workspace. Inputs and outputs are still the caller's.
//
// The array is 256 + 8 * (16,777,216 / 2048) = 65,792 bytes and lives on
// every device that loads this library until the process exits. Its device
// address is looked up with cudaGetSymbolAddress, with the device current:
// on every call whose stream is not being captured (so that an address made
// stale by cudaDeviceReset is replaced), and taken from the per-device cache
// while the stream is being captured (so a first call must precede capture).
#include <mutex>

#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int64_t kStaticMaxGaussians = GS_BIN_STATIC_MAX_GAUSSIANS;
constexpr int kBinChunkStatic = 2048;  // Gaussians per partial sum, as in binning.cu
constexpr size_t kStaticBytes =
    sizeof(StatusHeader) + (size_t)(kStaticMaxGaussians / kBinChunkStatic) * sizeof(unsigned long long);

static __device__ __align__(256) unsigned char g_bin_scratch[kStaticBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_dev_ptr[kMaxDevices] = {};

// Device address of g_bin_scratch on the current device: looked up again on
// every call outside stream capture, from the cache during capture.
cudaError_t static_scratch(cudaStream_t s, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    if (cap == cudaStreamCaptureStatusNone || !g_dev_ptr[dev]) {
        if (cap != cudaStreamCaptureStatusNone) return cudaErrorStreamCaptureUnsupported;
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_bin_scratch);
        if (e != cudaSuccess) return e;
        g_dev_ptr[dev] = p;
    }
    *out = g_dev_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace gs

using namespace gs;

extern "C" gs_status gs_bin_static(const gs_projected* p, int64_t n, const gs_camera* cam, uint32_t* offsets,
                                   uint64_t* keys, uint32_t* vals, int64_t key_capacity, uint64_t* num_keys,
                                   void* stream) {
    if (n < 0 || n > kStaticMaxGaussians || !cam || !p || !num_keys) return GS_ERR_INVALID_ARG;
    if (sizeof(StatusHeader) + bin_scratch_bytes(n) > kStaticBytes) return GS_ERR_INVALID_ARG;
    if (key_capacity < 0 || key_capacity > (1ll << 30) - 1) return GS_ERR_INVALID_ARG;
    if (cam->width < 1 || cam->height < 1 || cam->width > 32768 || cam->height > 32768) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!offsets || !p->tiles_touched || !p->rect || !p->depth)) return GS_ERR_INVALID_ARG;
    if (n > 0 && ((uintptr_t)p->rect % 8 != 0 || (uintptr_t)p->tiles_touched % 4 != 0)) return GS_ERR_INVALID_ARG;
    if (key_capacity > 0 && (!keys || !vals || (uintptr_t)keys % 8 != 0 || (uintptr_t)vals % 4 != 0))
        return GS_ERR_INVALID_ARG;
    if ((uintptr_t)num_keys % 8 != 0) return GS_ERR_INVALID_ARG;

    cudaStream_t s = (cudaStream_t)stream;
    void* base = nullptr;
    if (static_scratch(s, &base) != cudaSuccess) return GS_ERR_CUDA;
    auto* header = static_cast<StatusHeader*>(base);
    // the array keeps the previous call's contents: the header's flags must start at zero
    // (the partial sums are fully rewritten by every call)
    if (cudaMemsetAsync(header, 0, sizeof(StatusHeader), s) != cudaSuccess) return GS_ERR_CUDA;
    const cudaError_t e = launch_bin(*p, n, make_cam_const(*cam), offsets, keys, vals, key_capacity, num_keys,
                                     header, static_cast<char*>(base) + sizeof(StatusHeader), s);
    return e == cudaSuccess ? GS_OK : GS_ERR_CUDA;
}
