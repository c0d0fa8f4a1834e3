// Host side of the C ABI declared in include/gs.h: argument validation,
// workspace layout and the chaining of the five steps on one stream.
#include <math.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>

#include "gs_internal.cuh"

namespace gs {

long long g_spin_limit = 1ll << 22;   // ~1 s of polling with backoff
std::atomic<int> g_programmatic_launch{1};
constexpr long long kDefaultSpin = 1ll << 22;
constexpr int64_t kMaxKeyCapacity = (1ll << 30) - 1;   // look-back status words keep 30 bits
constexpr int64_t kMaxGaussians = (1ll << 32) - 1;     // values are uint32 indices
constexpr int kCoarseKeyTiles = 4096;                   // block-layout tile keys from this many tiles
constexpr int64_t kSideRangesMaxN = 1ll << 21;          // ranges on a second stream up to this many Gaussians

CamConst make_cam_const(const gs_camera& c) {
    CamConst k;
    for (int i = 0; i < 9; i++) k.R[i] = c.R[i];
    for (int i = 0; i < 3; i++) {
        k.t[i] = c.t[i];
        k.bg[i] = c.bg[i];
    }
    k.fx = c.fx; k.fy = c.fy; k.cx = c.cx; k.cy = c.cy; k.near_z = c.near_z;
    k.width = c.width; k.height = c.height;
    k.tiles_x = tiles_x(c);
    k.tiles_y = tiles_y(c);
    // camera centre -R^T t, in double then rounded
    for (int i = 0; i < 3; i++) {
        double s = 0.0;
        for (int j = 0; j < 3; j++) s += (double)c.R[3 * j + i] * (double)c.t[j];
        k.campos[i] = (float)(-s);
    }
    return k;
}

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool camera_ok(const gs_camera* c) {
    if (!c) return false;
    if (c->width < 1 || c->height < 1 || c->width > 32768 || c->height > 32768) return false;
    if (!(c->near_z > 0.0f) || !isfinite(c->near_z)) return false;
    const float v[] = {c->fx, c->fy, c->cx, c->cy, c->bg[0], c->bg[1], c->bg[2]};
    for (float x : v)
        if (!isfinite(x)) return false;
    for (int i = 0; i < 9; i++)
        if (!isfinite(c->R[i])) return false;
    for (int i = 0; i < 3; i++)
        if (!isfinite(c->t[i])) return false;
    return true;
}

bool gaussians_ok(const gs_gaussians* g) {
    if (!g || g->n < 0 || g->n > kMaxGaussians || g->sh_degree < 0 || g->sh_degree > 3) return false;
    if (g->n == 0) return true;
    if (!g->means || !g->quats || !g->log_scales || !g->opacity_logits || !g->sh) return false;
    if (!aligned(g->quats, 16) || !aligned(g->means, 4) || !aligned(g->log_scales, 4) ||
        !aligned(g->opacity_logits, 4) || !aligned(g->sh, 16))
        return false;
    return true;
}

// fields the binning reads (the projection writes those and any non-null rest)
bool projected_ok(const gs_projected* p, int64_t n) {
    if (!p) return false;
    if (n == 0) return true;
    return p->depth && p->tiles_touched && p->rect && aligned(p->mean2d, 8) && aligned(p->conic_opacity, 16) &&
           aligned(p->rgb, 4) && aligned(p->depth, 4) && aligned(p->radius, 4) && aligned(p->tiles_touched, 4) &&
           aligned(p->rect, 8) && aligned(p->raster, 16);
}

gs_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GS_OK : GS_ERR_CUDA; }

// gs_render workspace layout. The buffers a frame must find zeroed sit at
// the start, [header, zero_end), so one memset at the frame's start clears
// them all and no memset separates two kernels of the frame (each kernel is
// then launched as a programmatic dependent of the one before it).
struct RenderLayout {
    size_t header, num_keys, depth_head, ranges, order_done, td_counts, tile_head, len_diff, zero_end, raster, depth,
        touched, rect, dkeys, dkeys_alt, order, order_alt, bin, keys, vals, keys_alt, vals_alt, depth_lb, tile_lb,
        tile_order, tdepth, pgrad, total;
};

RenderLayout render_layout(int64_t n, int32_t w, int32_t h, int64_t cap) {
    RenderLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o += align_up(bytes);
        return at;
    };
    const size_t un = (size_t)(n > 0 ? n : 0), uc = (size_t)(cap > 0 ? cap : 0);
    const size_t tiles = (size_t)((w + kTile - 1) / kTile) * (size_t)((h + kTile - 1) / kTile);
    L.header = take(sizeof(StatusHeader));
    L.num_keys = take(sizeof(uint64_t));
    L.depth_head = take(sort_head_bytes());      // the depth sort's digit histograms and counters
    L.ranges = take(8 * tiles);
    L.order_done = take(sizeof(uint32_t));       // the tile order's finished-block counter
    L.td_counts = take(3 * sizeof(uint32_t));    // the per-tile depth sort's list lengths
    L.tile_head = take(sort_head_bytes());       // the tile sort's digit histograms and counters
    L.len_diff = take(tile_len_diff_bytes((w + kTile - 1) / kTile, (h + kTile - 1) / kTile));
    L.zero_end = o;
    L.raster = take(48 * un);
    L.depth = take(4 * un);
    L.touched = take(4 * un);
    L.rect = take(8 * un);
    L.dkeys = take(4 * un);
    L.dkeys_alt = take(4 * un);
    L.order = take(4 * un);
    L.order_alt = take(4 * un);
    L.bin = take(bin_ordered_scratch_bytes(n, cap));
    L.keys = take(4 * uc);
    L.vals = take(4 * uc);
    L.keys_alt = take(4 * uc);
    L.vals_alt = take(4 * uc);
    L.depth_lb = take(sort_lookback_bytes(n));
    L.tile_lb = take(sort_lookback_bytes(cap));
    L.tile_order = take(tile_order_scratch_bytes((int)tiles));
    L.tdepth = take(tile_depth_scratch_bytes((int)tiles));
    L.pgrad = take(36 * un);   // backward: dL/d(u, v), dL/d(conic), dL/do, dL/dc
    L.total = o;
    return L;
}

// The projected record of a view inside its gs_render workspace (only what
// binning and compositing read).
gs_projected view_projected(char* w, const RenderLayout& L) {
    gs_projected p;
    p.mean2d = nullptr;
    p.conic_opacity = nullptr;
    p.rgb = nullptr;
    p.radius = nullptr;
    p.raster = reinterpret_cast<float*>(w + L.raster);
    p.depth = reinterpret_cast<float*>(w + L.depth);
    p.tiles_touched = reinterpret_cast<uint32_t*>(w + L.touched);
    p.rect = reinterpret_cast<uint16_t*>(w + L.rect);
    return p;
}

}  // namespace
}  // namespace gs

namespace gs {
namespace {

// How the depth-order input of a view comes about.
enum class Step1 {
    kProject,      // run the projection here; it also writes the depth keys and their histograms
    kKeysReady,    // the caller projected into this workspace and wrote the keys and histograms
    kRecordOnly,   // the caller wrote the record only (2D splats): derive the keys here
};

// The depth-order keys of a view's workspace.
DepthKeysOut view_depth_keys(char* w, const RenderLayout& L) {
    DepthKeysOut dk;
    dk.keys = reinterpret_cast<uint32_t*>(w + L.dkeys);
    dk.vals = reinterpret_cast<uint32_t*>(w + L.order);
    dk.hist = sort_histogram_of(w + L.depth_head);
    return dk;
}

// The order of steps 2-4 for a frame. Tile-first (bin in index order, stable
// sort by tile, then each tile's list by depth) when the key capacity is at
// most kTileFirstMaxKeys: below about a million pairs the four global passes
// of the depth sort are short, latency-bound launches, and the per-tile sorts
// (shared memory, one block per list) cost less. Above it the per-tile sorts
// cost more than the depth sort of the Gaussians they replace, and the frame
// is depth-first (depth order of the Gaussians, bin in that order, stable sort
// by tile). Both give the same lists bit for bit. gs_set_steps_order can pin
// either order.
#ifndef GS_TILE_FIRST_MAX_KEYS
#define GS_TILE_FIRST_MAX_KEYS (1 << 20)
#endif
constexpr int64_t kTileFirstMaxKeys = GS_TILE_FIRST_MAX_KEYS;
std::atomic<int32_t> g_steps_order{0};   // 0 automatic, 1 depth-first, 2 tile-first
bool tile_first(int64_t key_capacity, Step1 step1) {
    if (step1 == Step1::kRecordOnly) return false;
    const int32_t o = g_steps_order.load(std::memory_order_relaxed);
    if (o != 0) return o == 2;
    return key_capacity <= kTileFirstMaxKeys;
}

// The tile-sort key layout of a frame with this tile grid.
TileKeyMap frame_tile_keys(int tiles_x_, int tiles_y_) {
    return tiles_x_ * tiles_y_ >= kCoarseKeyTiles ? block_keys(tiles_x_, tiles_y_) : identity_keys(tiles_x_);
}

// The second stream a frame computes its tile ranges and launch order on, and
// the events that fork it from the frame's stream and join it back: one set per
// host thread and device, created on first use outside a stream capture and
// kept (a cudaDeviceReset invalidates them, as it does gs_render_batch's
// events). *found = false: none exists yet and `main` is capturing, so none is
// created now (the frame then runs on one stream).
struct SideStream {
    cudaStream_t s;
    cudaEvent_t fork, join;
};
cudaError_t side_stream(cudaStream_t main, SideStream* out, bool* found) {
    thread_local std::map<int, SideStream> mine;
    *found = false;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto it = mine.find(dev);
    if (it == mine.end()) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(main, &cs);
        if (e != cudaSuccess) return e;
        if (cs != cudaStreamCaptureStatusNone) return cudaSuccess;
        SideStream ss{};
        e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        it = mine.emplace(dev, ss).first;
    }
    *out = it->second;
    *found = true;
    return cudaSuccess;
}

#ifndef GS_SIDE_RANGES
#define GS_SIDE_RANGES 1
#endif

// Steps 2-5 of one view (step 1 as `step1` says), on stream s. events: null,
// or 7 handles recorded at the stage boundaries (see gs_render_profiled for
// their order in each order of the steps).
cudaError_t view_pipeline(const gs_gaussians* g, const gs_camera* cam, int64_t key_capacity, char* w,
                          const RenderLayout& L, float* image, float* final_T, uint32_t* n_contrib, cudaStream_t s,
                          void* const* events, Step1 step1) {
    auto* header = reinterpret_cast<StatusHeader*>(w + L.header);
    auto* num_keys = reinterpret_cast<uint64_t*>(w + L.num_keys);
    gs_projected p = view_projected(w, L);
    auto* dkeys = reinterpret_cast<uint32_t*>(w + L.dkeys);
    auto* dkeys_alt = reinterpret_cast<uint32_t*>(w + L.dkeys_alt);
    auto* order = reinterpret_cast<uint32_t*>(w + L.order);
    auto* order_alt = reinterpret_cast<uint32_t*>(w + L.order_alt);
    auto* keys = reinterpret_cast<uint32_t*>(w + L.keys);
    auto* vals = reinterpret_cast<uint32_t*>(w + L.vals);
    auto* keys_alt = reinterpret_cast<uint32_t*>(w + L.keys_alt);
    auto* vals_alt = reinterpret_cast<uint32_t*>(w + L.vals_alt);
    auto* ranges = reinterpret_cast<uint32_t*>(w + L.ranges);
    const CamConst cc = make_cam_const(*cam);

    // the tile sort's keys: the tile block in the low digit from 4096 tiles up
    // (a warp's first-pass ranking then sees far fewer distinct digits)
    const TileKeyMap km = frame_tile_keys(cc.tiles_x, cc.tiles_y);
    const int tbits = tile_key_bits(km, cc.tiles_x * cc.tiles_y);
    auto mark = [&](int i) {
        return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) : cudaSuccess;
    };
    uint32_t* tile_hist = sort_histogram_of(w + L.tile_head);
    const int n_tiles = cc.tiles_x * cc.tiles_y;
    // the frame's setup, before the first stage mark (so that stage 1 brackets
    // the projection alone): one memset of the buffers the frame finds zeroed;
    // a batch view keeps the depth histograms its projection filled
    cudaError_t e;
    if (step1 == Step1::kKeysReady) {
        e = cudaMemsetAsync(w + L.header, 0, L.depth_head - L.header, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(w + L.ranges, 0, L.zero_end - L.ranges, s);
    } else {
        e = cudaMemsetAsync(w + L.header, 0, L.zero_end - L.header, s);
    }
    if (e == cudaSuccess) e = mark(0);
    uint32_t* tile_order = nullptr;
    auto* order_done = reinterpret_cast<uint32_t*>(w + L.order_done);
    // the tile ranges and the launch order: from the sorted keys, after the tile
    // sort; or, when the projection runs here, the tile grid's difference array
    // fits in shared memory and the depth sort's passes leave SMs free (up to
    // kSideRangesMaxN Gaussians; beyond, its persistent passes fill every SM
    // and the side work slowed them), from the tile rectangles on a second
    // stream forked after the projection, while the sorts run
    bool overlap = GS_SIDE_RANGES && step1 == Step1::kProject && g->n <= kSideRangesMaxN &&
                   tile_len_fits(cc.tiles_x, cc.tiles_y);
    SideStream side{};
    if (overlap && e == cudaSuccess) e = side_stream(s, &side, &overlap);
    auto fork_ranges = [&]() {
        cudaError_t r = cudaEventRecord(side.fork, s);
        if (r == cudaSuccess) r = cudaStreamWaitEvent(side.s, side.fork, 0);
        if (r == cudaSuccess)
            r = launch_tile_len_ranges(p.tiles_touched, p.rect, g->n, cc.tiles_x, cc.tiles_y, km, tbits,
                                       key_capacity, reinterpret_cast<int*>(w + L.len_diff), ranges, side.s);
        if (r == cudaSuccess)
            r = launch_tile_order_multi(ranges, n_tiles, w + L.tile_order, &tile_order, side.s, order_done);
        if (r == cudaSuccess) r = cudaEventRecord(side.join, side.s);
        return r;
    };
    auto ranges_and_order = [&]() {
        if (overlap) return cudaStreamWaitEvent(s, side.join, 0);
        cudaError_t r = launch_tile_ranges32(keys, num_keys, key_capacity, n_tiles, ranges, s, true, &km);
        if (r == cudaSuccess) r = launch_tile_order_multi(ranges, n_tiles, w + L.tile_order, &tile_order, s, order_done);
        return r;
    };
    if (tile_first(key_capacity, step1)) {
        // bin in index order, stable sort by tile, then each tile's list by (depth bits, index)
        if (e == cudaSuccess && step1 == Step1::kProject) e = launch_preprocess(*g, cc, p, s, nullptr, header);
        if (e == cudaSuccess) e = mark(1);
        if (e == cudaSuccess && overlap) e = fork_ranges();
        if (e == cudaSuccess)
            e = launch_bin_ordered(p, nullptr, g->n, cc, nullptr, keys, vals, key_capacity, num_keys, header,
                                   w + L.bin, s, tile_hist, tbits, &km);
        if (e == cudaSuccess) e = mark(2);
        if (e == cudaSuccess)
            e = launch_sort32_split(keys, vals, keys_alt, vals_alt, num_keys, key_capacity, tbits, header,
                                    w + L.tile_head, w + L.tile_lb, g_spin_limit, s, true);
        if (e == cudaSuccess) e = mark(3);
        if (e == cudaSuccess) e = ranges_and_order();
        if (e == cudaSuccess) e = mark(4);
        // the tile ids are not read again: their array is the long lists' key scratch
        if (e == cudaSuccess)
            e = launch_tile_depth_sort(ranges, tile_order, n_tiles, p.depth, g->n, key_capacity, vals, keys,
                                       keys_alt, vals_alt, reinterpret_cast<uint32_t*>(w + L.td_counts),
                                       w + L.tdepth, s);
        if (e == cudaSuccess) e = mark(5);
        if (e == cudaSuccess)
            e = launch_rasterize(p, g->n, vals, ranges, tile_order, cc, image, final_T, n_contrib, s);
        if (e == cudaSuccess) e = mark(6);
        return e;
    }
    // depth order first, then (tile, index) pairs in that order, then a stable
    // sort by tile: the same per-tile (depth, index) order as sorting the
    // 64-bit tile|depth keys, with far fewer key bits moved
    // (the producers of both key lists also count their sort digits)
    const DepthKeysOut dk = view_depth_keys(w, L);
    if (e == cudaSuccess && step1 == Step1::kProject) e = launch_preprocess(*g, cc, p, s, &dk, header);
    if (e == cudaSuccess) e = mark(1);
    if (e == cudaSuccess && overlap) e = fork_ranges();
    if (e == cudaSuccess && step1 == Step1::kRecordOnly) e = launch_depth_keys(p, g->n, dkeys, order, dk.hist, s);
    if (e == cudaSuccess)
        e = launch_sort32_split(dkeys, order, dkeys_alt, order_alt, nullptr, g->n, 32, header, w + L.depth_head,
                                w + L.depth_lb, g_spin_limit, s, true);
    if (e == cudaSuccess) e = mark(2);
    if (e == cudaSuccess)
        e = launch_bin_ordered(p, order, g->n, cc, nullptr, keys, vals, key_capacity, num_keys, header, w + L.bin, s,
                               tile_hist, tbits, &km);
    if (e == cudaSuccess) e = mark(3);
    if (e == cudaSuccess)
        e = launch_sort32_split(keys, vals, keys_alt, vals_alt, num_keys, key_capacity, tbits, header,
                                w + L.tile_head, w + L.tile_lb, g_spin_limit, s, true);
    if (e == cudaSuccess) e = mark(4);
    if (e == cudaSuccess) e = ranges_and_order();
    if (e == cudaSuccess) e = mark(5);
    if (e == cudaSuccess)
        e = launch_rasterize(p, g->n, vals, ranges, tile_order, cc, image, final_T, n_contrib, s);
    if (e == cudaSuccess) e = mark(6);
    return e;
}

gs_status render_impl(const gs_gaussians* g, const gs_camera* cam, int64_t key_capacity, void* ws, size_t ws_bytes,
                      float* image, float* final_T, uint32_t* n_contrib, void* stream, void* const* events) {
    if (!gaussians_ok(g) || !camera_ok(cam) || !image) return GS_ERR_INVALID_ARG;
    // the depth order sorts n keys: its look-back counts keep 30 bits
    if (g->n > kMaxKeyCapacity || key_capacity < 0 || key_capacity > kMaxKeyCapacity) return GS_ERR_INVALID_ARG;
    const RenderLayout L = render_layout(g->n, cam->width, cam->height, key_capacity);
    if (!ws || !aligned(ws, kAlign) || ws_bytes < L.total) return GS_ERR_WORKSPACE;
    return cuda_status(view_pipeline(g, cam, key_capacity, static_cast<char*>(ws), L, image, final_T, n_contrib,
                                     (cudaStream_t)stream, events, Step1::kProject));
}

// Fork/join events for gs_render_batch, created once per device on first use
// (timing disabled, so recording them costs no timestamp). g_batch_mutex is
// held by gs_render_batch from the lookup through its last join wait, so two
// host threads batching on one device cannot re-record each other's fork or
// join events between a record and the waits that depend on it.
constexpr int kMaxBatchStreams = 8;
struct BatchEvents {
    cudaEvent_t fork = nullptr;
    cudaEvent_t join[kMaxBatchStreams] = {};
};
std::mutex g_batch_mutex;
std::map<int, BatchEvents> g_batch_events;

// The calling thread must hold g_batch_mutex.
cudaError_t batch_events(BatchEvents** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto it = g_batch_events.find(dev);
    if (it == g_batch_events.end()) {
        BatchEvents be;
        e = cudaEventCreateWithFlags(&be.fork, cudaEventDisableTiming);
        for (int i = 0; e == cudaSuccess && i < kMaxBatchStreams; i++)
            e = cudaEventCreateWithFlags(&be.join[i], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            // release whatever was created; the next call tries again
            if (be.fork) cudaEventDestroy(be.fork);
            for (int i = 0; i < kMaxBatchStreams; i++)
                if (be.join[i]) cudaEventDestroy(be.join[i]);
            return e;
        }
        it = g_batch_events.emplace(dev, be).first;
    }
    *out = &it->second;
    return cudaSuccess;
}

}  // namespace
}  // namespace gs

using namespace gs;

extern "C" {

const char* gs_status_string(int32_t s) {
    switch (s) {
        case GS_OK: return "ok";
        case GS_ERR_INVALID_ARG: return "invalid argument";
        case GS_ERR_CAPACITY: return "key capacity exceeded";
        case GS_ERR_CUDA: return "CUDA error";
        case GS_ERR_TIMEOUT: return "device wait timed out";
        case GS_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        default: return "unknown status";
    }
}

int32_t gs_abi_version(void) { return GS_ABI_VERSION; }

void gs_set_spin_limit(int64_t iterations) { g_spin_limit = iterations > 0 ? iterations : kDefaultSpin; }

gs_status gs_preprocess(const gs_gaussians* g, const gs_camera* cam, const gs_projected* out, void* stream) {
    if (!gaussians_ok(g) || !camera_ok(cam) || !projected_ok(out, g ? g->n : 0)) return GS_ERR_INVALID_ARG;
    return cuda_status(launch_preprocess(*g, make_cam_const(*cam), *out, (cudaStream_t)stream));
}

size_t gs_bin_workspace_bytes(int64_t n) { return sizeof(StatusHeader) + bin_scratch_bytes(n < 0 ? 0 : n); }

gs_status gs_bin(const gs_projected* p, int64_t n, const gs_camera* cam, uint32_t* offsets, uint64_t* keys,
                 uint32_t* vals, int64_t key_capacity, uint64_t* num_keys, void* ws, size_t ws_bytes,
                 void* stream) {
    if (n < 0 || n > kMaxGaussians || !camera_ok(cam) || !projected_ok(p, n) || !num_keys) return GS_ERR_INVALID_ARG;
    if (key_capacity < 0 || key_capacity > kMaxKeyCapacity) return GS_ERR_INVALID_ARG;
    if (n > 0 && !offsets) return GS_ERR_INVALID_ARG;
    if (key_capacity > 0 && (!keys || !vals || !aligned(keys, 8) || !aligned(vals, 4))) return GS_ERR_INVALID_ARG;
    if (!aligned(num_keys, 8)) return GS_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < gs_bin_workspace_bytes(n)) return GS_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    auto* header = static_cast<StatusHeader*>(ws);
    cudaError_t e = cudaMemsetAsync(header, 0, sizeof(StatusHeader), s);
    if (e != cudaSuccess) return GS_ERR_CUDA;
    return cuda_status(launch_bin(*p, n, make_cam_const(*cam), offsets, keys, vals, key_capacity, num_keys, header,
                                  static_cast<char*>(ws) + sizeof(StatusHeader), s));
}

size_t gs_bin_ordered_workspace_bytes(int64_t n, int64_t key_capacity) {
    return sizeof(StatusHeader) + bin_ordered_scratch_bytes(n < 0 ? 0 : n, key_capacity < 0 ? 0 : key_capacity);
}

size_t gs_sort_workspace_bytes(int64_t key_capacity) {
    return sizeof(StatusHeader) + sort_scratch_bytes(key_capacity < 0 ? 0 : key_capacity);
}

gs_status gs_sort(uint64_t* keys, uint32_t* vals, uint64_t* keys_alt, uint32_t* vals_alt, const uint64_t* num_keys,
                  int64_t key_capacity, int32_t key_bits, void* ws, size_t ws_bytes, void* stream) {
    if (key_capacity < 0 || key_capacity > kMaxKeyCapacity || key_bits < 1 || key_bits > 64 || !num_keys)
        return GS_ERR_INVALID_ARG;
    if (key_capacity > 0 && (!keys || !vals || !keys_alt || !vals_alt || !aligned(keys, 8) || !aligned(keys_alt, 8) ||
                             !aligned(vals, 4) || !aligned(vals_alt, 4)))
        return GS_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < gs_sort_workspace_bytes(key_capacity)) return GS_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    auto* header = static_cast<StatusHeader*>(ws);
    cudaError_t e = cudaMemsetAsync(header, 0, sizeof(StatusHeader), s);
    if (e != cudaSuccess) return GS_ERR_CUDA;
    return cuda_status(launch_sort(keys, vals, keys_alt, vals_alt, num_keys, key_capacity, key_bits, header,
                                   static_cast<char*>(ws) + sizeof(StatusHeader), g_spin_limit, s));
}

gs_status gs_tile_ranges(const uint64_t* sorted_keys, const uint64_t* num_keys, int64_t key_capacity,
                         const gs_camera* cam, uint32_t* ranges, void* stream) {
    if (!camera_ok(cam) || !ranges || !num_keys || key_capacity < 0 || key_capacity > kMaxKeyCapacity)
        return GS_ERR_INVALID_ARG;
    if (key_capacity > 0 && !sorted_keys) return GS_ERR_INVALID_ARG;
    if (!aligned(ranges, 8)) return GS_ERR_INVALID_ARG;
    return cuda_status(launch_tile_ranges(sorted_keys, num_keys, key_capacity, tiles_x(*cam) * tiles_y(*cam), ranges,
                                          (cudaStream_t)stream));
}

gs_status gs_rasterize(const gs_projected* p, int64_t n, const uint32_t* sorted_vals, const uint32_t* ranges,
                       const gs_camera* cam, float* image, float* final_T, uint32_t* n_contrib, uint32_t* tile_order,
                       void* stream) {
    if (n < 0 || !camera_ok(cam) || !projected_ok(p, n) || !ranges || !image || !aligned(ranges, 8))
        return GS_ERR_INVALID_ARG;
    if (n > 0 && !p->raster) return GS_ERR_INVALID_ARG;
    if (n > 0 && !sorted_vals) return GS_ERR_INVALID_ARG;
    const CamConst cc = make_cam_const(*cam);
    if (tile_order) {
        const cudaError_t e = launch_tile_order(ranges, cc.tiles_x * cc.tiles_y, tile_order, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return cuda_status(
        launch_rasterize(*p, n, sorted_vals, ranges, tile_order, cc, image, final_T, n_contrib, (cudaStream_t)stream));
}

size_t gs_render_workspace_bytes(int64_t n, int32_t width, int32_t height, int64_t key_capacity) {
    if (n < 0 || width < 1 || height < 1 || key_capacity < 0) return 0;
    return render_layout(n, width, height, key_capacity).total;
}

gs_status gs_render(const gs_gaussians* g, const gs_camera* cam, int64_t key_capacity, void* ws, size_t ws_bytes,
                    float* image, float* final_T, uint32_t* n_contrib, void* stream) {
    return render_impl(g, cam, key_capacity, ws, ws_bytes, image, final_T, n_contrib, stream, nullptr);
}

int32_t gs_render_tile_first(int64_t n, int32_t width, int32_t height, int64_t key_capacity) {
    (void)n;
    if (width < 1 || height < 1 || key_capacity < 0) return 0;
    return tile_first(key_capacity, Step1::kProject) ? 1 : 0;
}

void gs_set_programmatic_launch(int32_t on) { g_programmatic_launch.store(on ? 1 : 0, std::memory_order_relaxed); }

int64_t gs_debug_tile_key(int32_t tiles_x_, int32_t tiles_y_, int32_t tx, int32_t ty) {
    if (tiles_x_ < 1 || tiles_y_ < 1 || tiles_x_ > 32768 || tiles_y_ > 32768 || tx < 0 || ty < 0 || tx >= tiles_x_ ||
        ty >= tiles_y_)
        return -1;
    return tile_key(frame_tile_keys(tiles_x_, tiles_y_), (uint32_t)tx, (uint32_t)ty);
}

int32_t gs_debug_tile_key_bits(int32_t tiles_x_, int32_t tiles_y_) {
    if (tiles_x_ < 1 || tiles_y_ < 1 || tiles_x_ > 32768 || tiles_y_ > 32768) return -1;
    return tile_key_bits(frame_tile_keys(tiles_x_, tiles_y_), tiles_x_ * tiles_y_);
}

int64_t gs_debug_tile_of_key(int32_t tiles_x_, int32_t tiles_y_, int64_t key) {
    if (tiles_x_ < 1 || tiles_y_ < 1 || tiles_x_ > 32768 || tiles_y_ > 32768 || key < 0) return -1;
    const TileKeyMap km = frame_tile_keys(tiles_x_, tiles_y_);
    if (key >= (1ll << tile_key_bits(km, tiles_x_ * tiles_y_))) return -1;
    const uint32_t t = tile_of_key(km, (uint32_t)key);
    const uint32_t tx = t % (uint32_t)tiles_x_, ty = t / (uint32_t)tiles_x_;
    if (ty >= (uint32_t)tiles_y_ || tile_key(km, tx, ty) != (uint32_t)key) return -1;
    return t;
}

gs_status gs_set_steps_order(int32_t order) {
    if (order < 0 || order > 2) return GS_ERR_INVALID_ARG;
    g_steps_order.store(order, std::memory_order_relaxed);
    return GS_OK;
}

gs_status gs_render_workspace_lists(const void* ws, int64_t n, int32_t width, int32_t height, int64_t key_capacity,
                                    const uint32_t** sorted_vals, const uint32_t** ranges) {
    if (!ws || !aligned(ws, kAlign)) return GS_ERR_WORKSPACE;
    if (n < 0 || width < 1 || height < 1 || key_capacity < 0 || !sorted_vals || !ranges) return GS_ERR_INVALID_ARG;
    const RenderLayout L = render_layout(n, width, height, key_capacity);
    const char* w = static_cast<const char*>(ws);
    *sorted_vals = reinterpret_cast<const uint32_t*>(w + L.vals);
    *ranges = reinterpret_cast<const uint32_t*>(w + L.ranges);
    return GS_OK;
}

gs_status gs_render_profiled(const gs_gaussians* g, const gs_camera* cam, int64_t key_capacity, void* ws,
                             size_t ws_bytes, float* image, float* final_T, uint32_t* n_contrib, void* stream,
                             void* const* events, int32_t n_events) {
    if (!events || n_events < GS_RENDER_STAGES + 1) return GS_ERR_INVALID_ARG;
    for (int i = 0; i <= GS_RENDER_STAGES; i++)
        if (!events[i]) return GS_ERR_INVALID_ARG;
    return render_impl(g, cam, key_capacity, ws, ws_bytes, image, final_T, n_contrib, stream, events);
}



size_t gs_depth_order_workspace_bytes(int64_t n) {
    const size_t un = (size_t)(n > 0 ? n : 0);
    return sizeof(StatusHeader) + 3 * align_up(4 * un) + sort_scratch_bytes(n > 0 ? n : 0);
}

gs_status gs_depth_order(const gs_projected* p, int64_t n, uint32_t* order, void* ws, size_t ws_bytes,
                         void* stream) {
    if (n < 0 || n > kMaxKeyCapacity || !p || (n > 0 && (!p->depth || !p->tiles_touched || !order)))
        return GS_ERR_INVALID_ARG;
    if (n > 0 && (!aligned(p->depth, 4) || !aligned(p->tiles_touched, 4) || !aligned(order, 4)))
        return GS_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < gs_depth_order_workspace_bytes(n)) return GS_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    char* w = static_cast<char*>(ws);
    auto* header = reinterpret_cast<StatusHeader*>(w);
    const size_t un = align_up(4 * (size_t)n);
    auto* keys = reinterpret_cast<uint32_t*>(w + sizeof(StatusHeader));
    auto* keys_alt = reinterpret_cast<uint32_t*>(w + sizeof(StatusHeader) + un);
    auto* order_alt = reinterpret_cast<uint32_t*>(w + sizeof(StatusHeader) + 2 * un);
    void* scratch = w + sizeof(StatusHeader) + 3 * un;
    cudaError_t e = cudaMemsetAsync(header, 0, sizeof(StatusHeader), s);
    if (e == cudaSuccess) e = sort_prepare_histogram(scratch, s);
    if (e == cudaSuccess) e = launch_depth_keys(*p, n, keys, order, sort_histogram_of(scratch), s);
    if (e == cudaSuccess)
        e = launch_sort32(keys, order, keys_alt, order_alt, nullptr, n, 32, header, scratch, g_spin_limit, s, true);
    return cuda_status(e);
}

gs_status gs_bin_ordered(const gs_projected* p, int64_t n, const uint32_t* order, const gs_camera* cam,
                         uint32_t* offsets, uint32_t* tile_keys, uint32_t* vals, int64_t key_capacity,
                         uint64_t* num_keys, void* ws, size_t ws_bytes, void* stream) {
    if (n < 0 || n > kMaxGaussians || !camera_ok(cam) || !projected_ok(p, n) || !num_keys) return GS_ERR_INVALID_ARG;
    if (key_capacity < 0 || key_capacity > kMaxKeyCapacity) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!order || !aligned(order, 4))) return GS_ERR_INVALID_ARG;
    if (key_capacity > 0 && (!tile_keys || !vals || !aligned(tile_keys, 4) || !aligned(vals, 4)))
        return GS_ERR_INVALID_ARG;
    if (!aligned(num_keys, 8)) return GS_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < gs_bin_ordered_workspace_bytes(n, key_capacity))
        return GS_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    auto* header = static_cast<StatusHeader*>(ws);
    cudaError_t e = cudaMemsetAsync(header, 0, sizeof(StatusHeader), s);
    if (e != cudaSuccess) return GS_ERR_CUDA;
    return cuda_status(launch_bin_ordered(*p, order, n, make_cam_const(*cam), offsets, tile_keys, vals, key_capacity,
                                          num_keys, header, static_cast<char*>(ws) + sizeof(StatusHeader), s));
}

gs_status gs_sort32(uint32_t* keys, uint32_t* vals, uint32_t* keys_alt, uint32_t* vals_alt, const uint64_t* num_keys,
                    int64_t key_capacity, int32_t key_bits, void* ws, size_t ws_bytes, void* stream) {
    if (key_capacity < 0 || key_capacity > kMaxKeyCapacity || key_bits < 1 || key_bits > 32)
        return GS_ERR_INVALID_ARG;
    if (key_capacity > 0 && (!keys || !vals || !keys_alt || !vals_alt || !aligned(keys, 4) || !aligned(keys_alt, 4) ||
                             !aligned(vals, 4) || !aligned(vals_alt, 4)))
        return GS_ERR_INVALID_ARG;
    if (num_keys && !aligned(num_keys, 8)) return GS_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < gs_sort_workspace_bytes(key_capacity)) return GS_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    auto* header = static_cast<StatusHeader*>(ws);
    cudaError_t e = cudaMemsetAsync(header, 0, sizeof(StatusHeader), s);
    if (e != cudaSuccess) return GS_ERR_CUDA;
    return cuda_status(launch_sort32(keys, vals, keys_alt, vals_alt, num_keys, key_capacity, key_bits, header,
                                     static_cast<char*>(ws) + sizeof(StatusHeader), g_spin_limit, s));
}

gs_status gs_tile_ranges32(const uint32_t* sorted_tiles, const uint64_t* num_keys, int64_t key_capacity,
                           const gs_camera* cam, uint32_t* ranges, void* stream) {
    if (!camera_ok(cam) || !ranges || !num_keys || key_capacity < 0 || key_capacity > kMaxKeyCapacity)
        return GS_ERR_INVALID_ARG;
    if (key_capacity > 0 && !sorted_tiles) return GS_ERR_INVALID_ARG;
    if (!aligned(ranges, 8)) return GS_ERR_INVALID_ARG;
    return cuda_status(launch_tile_ranges32(sorted_tiles, num_keys, key_capacity, tiles_x(*cam) * tiles_y(*cam),
                                            ranges, (cudaStream_t)stream));
}

gs_status gs_render_from_host(const gs_gaussians* hg, const gs_gaussians* dg, const gs_camera* cam,
                              int64_t key_capacity, void* ws, size_t ws_bytes, float* device_image,
                              float* host_image, void* stream) {
    if (!hg || !dg || hg->n != dg->n || hg->sh_degree != dg->sh_degree || !gaussians_ok(dg) || !host_image)
        return GS_ERR_INVALID_ARG;
    if (dg->n > 0 && (!hg->means || !hg->quats || !hg->log_scales || !hg->opacity_logits || !hg->sh))
        return GS_ERR_INVALID_ARG;
    if (!camera_ok(cam) || !device_image) return GS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t n = (size_t)dg->n, nk = (size_t)((dg->sh_degree + 1) * (dg->sh_degree + 1));
    struct { const void* src; const void* dst; size_t bytes; } cp[5] = {
        {hg->means, dg->means, 12 * n}, {hg->quats, dg->quats, 16 * n}, {hg->log_scales, dg->log_scales, 12 * n},
        {hg->opacity_logits, dg->opacity_logits, 4 * n}, {hg->sh, dg->sh, 12 * nk * n}};
    for (auto& c : cp) {
        if (c.bytes == 0) continue;
        if (cudaMemcpyAsync(const_cast<void*>(c.dst), c.src, c.bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return GS_ERR_CUDA;
    }
    gs_status st = gs_render(dg, cam, key_capacity, ws, ws_bytes, device_image, nullptr, nullptr, stream);
    if (st != GS_OK) return st;
    const size_t img = (size_t)cam->width * cam->height * 3 * sizeof(float);
    return cuda_status(cudaMemcpyAsync(host_image, device_image, img, cudaMemcpyDeviceToHost, s));
}

static bool pgrad_ok(const gs_projected_grad* g, int64_t n) {
    if (!g) return false;
    if (n == 0) return true;
    return g->mean2d && g->conic && g->opacity && g->rgb && aligned(g->mean2d, 8) && aligned(g->conic, 4) &&
           aligned(g->opacity, 4) && aligned(g->rgb, 4);
}

static bool ggrad_ok(const gs_gaussians_grad* g, int64_t n) {
    if (!g) return false;
    if (n == 0) return true;
    return g->means && g->quats && g->log_scales && g->opacity_logits && g->sh && aligned(g->means, 4) &&
           aligned(g->quats, 4) && aligned(g->log_scales, 4) && aligned(g->opacity_logits, 4) && aligned(g->sh, 4);
}

gs_status gs_rasterize_backward(const gs_projected* p, int64_t n, const uint32_t* sorted_vals, const uint32_t* ranges,
                                const gs_camera* cam, const float* final_T, const uint32_t* n_contrib,
                                const float* grad_image, const uint32_t* tile_order, const gs_projected_grad* grad,
                                void* stream) {
    if (n < 0 || n > kMaxGaussians || !camera_ok(cam) || !projected_ok(p, n) || !ranges || !aligned(ranges, 8))
        return GS_ERR_INVALID_ARG;
    if (!final_T || !n_contrib || !grad_image || !pgrad_ok(grad, n)) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!p->raster || !sorted_vals)) return GS_ERR_INVALID_ARG;
    return cuda_status(launch_rasterize_backward(*p, n, sorted_vals, ranges, tile_order, make_cam_const(*cam),
                                                 final_T, n_contrib, grad_image, *grad, (cudaStream_t)stream));
}

gs_status gs_preprocess_backward(const gs_gaussians* g, const gs_camera* cam, const gs_projected* p,
                                 const gs_projected_grad* grad_in, const gs_gaussians_grad* grad_out, void* stream) {
    if (!gaussians_ok(g) || !camera_ok(cam) || !p || (g->n > 0 && !p->tiles_touched)) return GS_ERR_INVALID_ARG;
    if (!pgrad_ok(grad_in, g->n) || !ggrad_ok(grad_out, g->n)) return GS_ERR_INVALID_ARG;
    return cuda_status(launch_preprocess_backward(*g, make_cam_const(*cam), p->tiles_touched, *grad_in, *grad_out,
                                                  (cudaStream_t)stream));
}

gs_status gs_render_backward(const gs_gaussians* g, const gs_camera* cam, int64_t key_capacity, void* ws,
                             size_t ws_bytes, const float* final_T, const uint32_t* n_contrib, const float* grad_image,
                             const gs_gaussians_grad* grad_out, void* stream) {
    if (!gaussians_ok(g) || !camera_ok(cam)) return GS_ERR_INVALID_ARG;
    if (key_capacity < 0 || key_capacity > kMaxKeyCapacity) return GS_ERR_INVALID_ARG;
    if (!final_T || !n_contrib || !grad_image || !ggrad_ok(grad_out, g->n)) return GS_ERR_INVALID_ARG;
    const RenderLayout L = render_layout(g->n, cam->width, cam->height, key_capacity);
    if (!ws || !aligned(ws, kAlign) || ws_bytes < L.total) return GS_ERR_WORKSPACE;
    if (g->n == 0) return GS_OK;
    cudaStream_t s = (cudaStream_t)stream;
    char* w = static_cast<char*>(ws);
    const gs_projected p = view_projected(w, L);
    const size_t n = (size_t)g->n;
    float* pg = reinterpret_cast<float*>(w + L.pgrad);
    gs_projected_grad pgr;
    pgr.mean2d = pg;
    pgr.conic = pg + 2 * n;
    pgr.opacity = pg + 5 * n;
    pgr.rgb = pg + 6 * n;
    const CamConst cc = make_cam_const(*cam);
    cudaError_t e = launch_rasterize_backward(p, g->n, reinterpret_cast<const uint32_t*>(w + L.vals),
                                              reinterpret_cast<const uint32_t*>(w + L.ranges),
                                              reinterpret_cast<const uint32_t*>(w + L.tile_order), cc, final_T,
                                              n_contrib, grad_image, pgr, s);
    if (e == cudaSuccess) e = launch_preprocess_backward(*g, cc, p.tiles_touched, pgr, *grad_out, s);
    return cuda_status(e);
}

static gs_camera camera_2d(int32_t width, int32_t height) {
    gs_camera c;
    memset(&c, 0, sizeof(c));
    c.R[0] = c.R[4] = c.R[8] = 1.0f;
    c.fx = c.fy = 1.0f;
    c.near_z = 1.0f;
    c.width = width;
    c.height = height;
    return c;
}

gs_status gs_rasterize_2d(const float* means, const float* covs, const float* colours, const float* opacities,
                          const float* depths, int64_t n, int32_t width, int32_t height, int64_t key_capacity,
                          void* ws, size_t ws_bytes, float* image, float* final_T, uint32_t* n_contrib,
                          void* stream) {
    if (n < 0 || n > kMaxKeyCapacity || width < 1 || height < 1 || width > 32768 || height > 32768 || !image)
        return GS_ERR_INVALID_ARG;
    if (n > 0 && (!means || !covs || !colours || !opacities || !depths || !aligned(means, 8)))
        return GS_ERR_INVALID_ARG;
    if (key_capacity < 0 || key_capacity > kMaxKeyCapacity) return GS_ERR_INVALID_ARG;
    const RenderLayout L = render_layout(n, width, height, key_capacity);
    if (!ws || !aligned(ws, kAlign) || ws_bytes < L.total) return GS_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    char* w = static_cast<char*>(ws);
    const gs_camera cam = camera_2d(width, height);
    gs_gaussians g;
    memset(&g, 0, sizeof(g));
    g.n = n;
    if (launch_preprocess2d(means, covs, colours, opacities, depths, n, width, height, view_projected(w, L), s) !=
        cudaSuccess)
        return GS_ERR_CUDA;
    return cuda_status(
        view_pipeline(&g, &cam, key_capacity, w, L, image, final_T, n_contrib, s, nullptr, Step1::kRecordOnly));
}

gs_status gs_rasterize_2d_backward(const float* covs, int64_t n, int32_t width, int32_t height, int64_t key_capacity,
                                   void* ws, size_t ws_bytes, const float* final_T, const uint32_t* n_contrib,
                                   const float* grad_image, float* grad_means, float* grad_covs, float* grad_colours,
                                   float* grad_opacities, void* stream) {
    if (n < 0 || n > kMaxGaussians || width < 1 || height < 1 || width > 32768 || height > 32768)
        return GS_ERR_INVALID_ARG;
    if (!final_T || !n_contrib || !grad_image) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!covs || !grad_means || !grad_covs || !grad_colours || !grad_opacities || !aligned(grad_means, 8)))
        return GS_ERR_INVALID_ARG;
    if (key_capacity < 0 || key_capacity > kMaxKeyCapacity) return GS_ERR_INVALID_ARG;
    const RenderLayout L = render_layout(n, width, height, key_capacity);
    if (!ws || !aligned(ws, kAlign) || ws_bytes < L.total) return GS_ERR_WORKSPACE;
    if (n == 0) return GS_OK;
    cudaStream_t s = (cudaStream_t)stream;
    char* w = static_cast<char*>(ws);
    const gs_projected p = view_projected(w, L);
    gs_projected_grad pgr;
    pgr.mean2d = grad_means;
    pgr.conic = reinterpret_cast<float*>(w + L.pgrad);
    pgr.opacity = grad_opacities;
    pgr.rgb = grad_colours;
    const gs_camera cam = camera_2d(width, height);
    cudaError_t e = launch_rasterize_backward(p, n, reinterpret_cast<const uint32_t*>(w + L.vals),
                                              reinterpret_cast<const uint32_t*>(w + L.ranges),
                                              reinterpret_cast<const uint32_t*>(w + L.tile_order),
                                              make_cam_const(cam), final_T, n_contrib, grad_image, pgr, s);
    if (e == cudaSuccess) e = launch_conic_to_cov_grad(covs, p.tiles_touched, pgr.conic, n, grad_covs, s);
    return cuda_status(e);
}

gs_status gs_densify_stats(const float* grad_mean2d, const uint32_t* tiles_touched, int64_t n, float* accum,
                           uint32_t* count, void* stream) {
    if (n < 0 || n > kMaxGaussians) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!grad_mean2d || !tiles_touched || !accum || !count || !aligned(grad_mean2d, 8)))
        return GS_ERR_INVALID_ARG;
    return cuda_status(launch_densify_stats(grad_mean2d, tiles_touched, n, accum, count, (cudaStream_t)stream));
}

size_t gs_densify_workspace_bytes(int64_t n) {
    if (n < 0 || n > kMaxGaussians) return 0;
    return densify_scratch_bytes(n);
}

gs_status gs_densify(const gs_gaussians* in, const float* accum, const uint32_t* count, const float* xi,
                     float grad_threshold, float scale_threshold, float prune_opacity, const gs_gaussians_out* out,
                     uint64_t* out_count, uint8_t* action, void* ws, size_t ws_bytes, void* stream) {
    if (!gaussians_ok(in) || !out || !out_count) return GS_ERR_INVALID_ARG;
    if (out->sh_degree != in->sh_degree || out->n < 0 || out->n > kMaxGaussians) return GS_ERR_INVALID_ARG;
    if (in->n > 0 && (!accum || !count || !xi)) return GS_ERR_INVALID_ARG;
    if (out->n > 0 && (!out->means || !out->quats || !out->log_scales || !out->opacity_logits || !out->sh))
        return GS_ERR_INVALID_ARG;
    if (!(prune_opacity > 0.0f && prune_opacity < 1.0f) || !(scale_threshold > 0.0f) || !isfinite(grad_threshold))
        return GS_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < densify_scratch_bytes(in->n)) return GS_ERR_WORKSPACE;
    const double t = prune_opacity;
    const float logit_thr = (float)log(t / (1.0 - t));
    const float log_scale_thr = (float)log((double)scale_threshold);
    return cuda_status(launch_densify(*in, *out, out->n, accum, count, xi, grad_threshold, log_scale_thr, logit_thr,
                                      action, out_count, ws, (cudaStream_t)stream));
}

size_t gs_render_batch_workspace_bytes(int64_t n, int32_t width, int32_t height, int64_t key_capacity,
                                       int32_t views) {
    if (views < 1 || views > GS_MAX_BATCH_VIEWS) return 0;
    return (size_t)views * gs_render_workspace_bytes(n, width, height, key_capacity);
}

gs_status gs_render_batch(const gs_gaussians* g, const gs_camera* cams, int32_t views, int64_t key_capacity,
                          void* ws, size_t ws_bytes, float* images, float* final_T, uint32_t* n_contrib,
                          void* const* streams, int32_t n_streams) {
    if (!gaussians_ok(g) || !cams || views < 1 || views > GS_MAX_BATCH_VIEWS || !images) return GS_ERR_INVALID_ARG;
    if (g->n > kMaxKeyCapacity) return GS_ERR_INVALID_ARG;
    if (!streams || n_streams < 1 || n_streams > kMaxBatchStreams) return GS_ERR_INVALID_ARG;
    if (key_capacity < 0 || key_capacity > kMaxKeyCapacity) return GS_ERR_INVALID_ARG;
    for (int v = 0; v < views; v++) {
        if (!camera_ok(cams + v)) return GS_ERR_INVALID_ARG;
        if (cams[v].width != cams[0].width || cams[v].height != cams[0].height) return GS_ERR_INVALID_ARG;
    }
    const RenderLayout L = render_layout(g->n, cams[0].width, cams[0].height, key_capacity);
    const size_t stride = L.total;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < stride * (size_t)views) return GS_ERR_WORKSPACE;
    // held until the last join wait is enqueued (the calls below only enqueue work)
    std::lock_guard<std::mutex> lock(g_batch_mutex);
    BatchEvents* ev = nullptr;
    if (batch_events(&ev) != cudaSuccess) return GS_ERR_CUDA;
    char* w0 = static_cast<char*>(ws);
    const size_t pix = (size_t)cams[0].width * cams[0].height;
    cudaStream_t s0 = (cudaStream_t)streams[0];
    // step 1 for all views, one pass over the parameters (chunks of kMaxBatchViews)
    for (int v0 = 0; v0 < views; v0 += kMaxBatchViews) {
        const int nv = views - v0 < kMaxBatchViews ? views - v0 : kMaxBatchViews;
        CamConst cc[kMaxBatchViews];
        gs_projected pr[kMaxBatchViews];
        DepthKeysOut dk[kMaxBatchViews];
        for (int i = 0; i < nv; i++) {
            char* wv = w0 + (size_t)(v0 + i) * stride;
            cc[i] = make_cam_const(cams[v0 + i]);
            pr[i] = view_projected(wv, L);
            dk[i] = view_depth_keys(wv, L);
            if (sort_prepare_histogram(wv + L.depth_head, s0) != cudaSuccess) return GS_ERR_CUDA;
        }
        if (launch_preprocess_batch(*g, cc, pr, dk, nv, s0) != cudaSuccess) return GS_ERR_CUDA;
    }
    // steps 2-5 per view, round-robin over the streams, forked from and joined into streams[0]
    if (n_streams > 1) {
        if (cudaEventRecord(ev->fork, s0) != cudaSuccess) return GS_ERR_CUDA;
        for (int i = 1; i < n_streams; i++)
            if (cudaStreamWaitEvent((cudaStream_t)streams[i], ev->fork, 0) != cudaSuccess) return GS_ERR_CUDA;
    }
    for (int v = 0; v < views; v++) {
        cudaStream_t s = (cudaStream_t)streams[v % n_streams];
        const cudaError_t e = view_pipeline(g, cams + v, key_capacity, w0 + (size_t)v * stride, L,
                                            images + (size_t)v * pix * 3, final_T ? final_T + (size_t)v * pix : nullptr,
                                            n_contrib ? n_contrib + (size_t)v * pix : nullptr, s, nullptr,
                                            Step1::kKeysReady);
        if (e != cudaSuccess) return GS_ERR_CUDA;
    }
    for (int i = 1; i < n_streams; i++) {
        if (cudaEventRecord(ev->join[i], (cudaStream_t)streams[i]) != cudaSuccess) return GS_ERR_CUDA;
        if (cudaStreamWaitEvent(s0, ev->join[i], 0) != cudaSuccess) return GS_ERR_CUDA;
    }
    return GS_OK;
}

gs_status gs_render_from_host_async(const gs_gaussians* hg, const gs_gaussians* device_sets, int64_t frame,
                                    const gs_camera* cam, int64_t key_capacity, void* ws, size_t ws_bytes,
                                    float* device_image, float* host_image, void* const* streams,
                                    void* const* events) {
    if (!hg || !device_sets || frame < 0 || !streams || !events || !host_image || !device_image)
        return GS_ERR_INVALID_ARG;
    for (int i = 0; i < 3; i++)
        if (!streams[i]) return GS_ERR_INVALID_ARG;
    for (int i = 0; i < 6; i++)
        if (!events[i]) return GS_ERR_INVALID_ARG;
    const int set = (int)(frame & 1);
    const gs_gaussians* dg = device_sets + set;
    if (hg->n != dg->n || hg->sh_degree != dg->sh_degree || !gaussians_ok(dg) || !camera_ok(cam))
        return GS_ERR_INVALID_ARG;
    if (dg->n > 0 && (!hg->means || !hg->quats || !hg->log_scales || !hg->opacity_logits || !hg->sh))
        return GS_ERR_INVALID_ARG;
    cudaStream_t s_render = (cudaStream_t)streams[0], s_h2d = (cudaStream_t)streams[1],
                 s_d2h = (cudaStream_t)streams[2];
    cudaEvent_t h2d_done = (cudaEvent_t)events[set], render_done = (cudaEvent_t)events[2 + set],
                img_ready = (cudaEvent_t)events[4], img_copied = (cudaEvent_t)events[5];
    const size_t n = (size_t)dg->n, nk = (size_t)((dg->sh_degree + 1) * (dg->sh_degree + 1));
    struct { const void* src; const void* dst; size_t bytes; } cp[5] = {
        {hg->means, dg->means, 12 * n}, {hg->quats, dg->quats, 16 * n}, {hg->log_scales, dg->log_scales, 12 * n},
        {hg->opacity_logits, dg->opacity_logits, 4 * n}, {hg->sh, dg->sh, 12 * nk * n}};
    // 1. parameters into this frame's device set, once the frame two back has
    //    finished rendering from it
    if (frame >= 2 && cudaStreamWaitEvent(s_h2d, render_done, 0) != cudaSuccess) return GS_ERR_CUDA;
    for (auto& c : cp) {
        if (c.bytes == 0) continue;
        if (cudaMemcpyAsync(const_cast<void*>(c.dst), c.src, c.bytes, cudaMemcpyHostToDevice, s_h2d) != cudaSuccess)
            return GS_ERR_CUDA;
    }
    if (cudaEventRecord(h2d_done, s_h2d) != cudaSuccess) return GS_ERR_CUDA;
    // 2. render once the copy is in and the previous image has been read back
    if (cudaStreamWaitEvent(s_render, h2d_done, 0) != cudaSuccess) return GS_ERR_CUDA;
    if (frame >= 1 && cudaStreamWaitEvent(s_render, img_copied, 0) != cudaSuccess) return GS_ERR_CUDA;
    gs_status st = gs_render(dg, cam, key_capacity, ws, ws_bytes, device_image, nullptr, nullptr, s_render);
    if (st != GS_OK) return st;
    if (cudaEventRecord(render_done, s_render) != cudaSuccess) return GS_ERR_CUDA;
    if (cudaEventRecord(img_ready, s_render) != cudaSuccess) return GS_ERR_CUDA;
    // 3. the image back to the host
    if (cudaStreamWaitEvent(s_d2h, img_ready, 0) != cudaSuccess) return GS_ERR_CUDA;
    const size_t img = (size_t)cam->width * cam->height * 3 * sizeof(float);
    if (cudaMemcpyAsync(host_image, device_image, img, cudaMemcpyDeviceToHost, s_d2h) != cudaSuccess)
        return GS_ERR_CUDA;
    return cuda_status(cudaEventRecord(img_copied, s_d2h));
}

int32_t gs_debug_checks_enabled(void) {
#ifdef GS_DEBUG_CHECKS
    return 1;
#else
    return 0;
#endif
}

gs_status gs_debug_set_check_counter(uint64_t* device_counter) {
    unsigned long long* p = reinterpret_cast<unsigned long long*>(device_counter);
    cudaError_t e = set_check_counter_preprocess(p);
    if (e == cudaSuccess) e = set_check_counter_binning(p);
    if (e == cudaSuccess) e = set_check_counter_sort(p);
    if (e == cudaSuccess) e = set_check_counter_rasterize(p);
    if (e == cudaSuccess) e = set_check_counter_backward(p);
    if (e == cudaSuccess) e = set_check_counter_splat2d(p);
    if (e == cudaSuccess) e = set_check_counter_densify(p);
    if (e == cudaSuccess) e = set_check_counter_tiledepth(p);
    if (e == cudaSuccess) e = set_check_counter_tilelen(p);
    return cuda_status(e);
}

gs_status gs_read_status(const void* ws, void* stream, uint32_t* flags, uint64_t* num_keys) {
    if (!ws || !aligned(ws, kAlign)) return GS_ERR_WORKSPACE;
    StatusHeader h;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return GS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GS_ERR_CUDA;
    if (flags) *flags = h.flags;
    if (num_keys) *num_keys = h.num_keys;
    if (h.flags & GS_FLAG_TIMEOUT) return GS_ERR_TIMEOUT;
    if (h.flags & GS_FLAG_CAPACITY) return GS_ERR_CAPACITY;
    return GS_OK;
}

size_t gs_workspace_bytes(int64_t n, int32_t width, int32_t height, int64_t key_capacity) {
    return gs_render_workspace_bytes(n, width, height, key_capacity);
}

gs_status gs_last_device_status(const void* ws) {
    if (!ws || !aligned(ws, kAlign)) return GS_ERR_WORKSPACE;
    if (cudaDeviceSynchronize() != cudaSuccess) return GS_ERR_CUDA;
    return gs_read_status(ws, nullptr, nullptr, nullptr);
}

gs_status gs_test_spin_timeout(void* ws, int64_t iterations, void* stream) {
    if (!ws || !aligned(ws, kAlign) || iterations < 0) return GS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    auto* header = static_cast<StatusHeader*>(ws);
    if (cudaMemsetAsync(header, 0, sizeof(StatusHeader), s) != cudaSuccess) return GS_ERR_CUDA;
    return cuda_status(launch_spin_timeout_test(header, iterations, s));
}

}  // extern "C"
