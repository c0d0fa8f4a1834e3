/*
 * gs.h -- C ABI of the B300 forward renderer for 3D Gaussian Splatting.
 *
 * The method is the one on the lesson page "3D Gaussian Splatting à partir de
 * zéro": each Gaussian carries a mean, a unit quaternion, log-scales, an
 * opacity logit and spherical-harmonic colour (section "Ce qu'un Gaussien
 * porte"); a frame is rendered in five steps -- project to 2D, assign to 16x16
 * screen tiles, depth-sort per tile, alpha-composite front to back, pixel
 * colour (section "Rastérisation, non rayée", flowchart).
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA global-memory addresses on the current
 *     device; the caller owns every buffer. The library never allocates, frees
 *     or synchronises, except where an entry point says so.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All work is enqueued on it in order; results are ready when the
 *     stream is.
 *   - Argument errors are found on the host before anything is enqueued and
 *     return GS_ERR_INVALID_ARG (or GS_ERR_WORKSPACE for a short workspace).
 *     A failed launch returns GS_ERR_CUDA. Device-side conditions (key
 *     capacity exceeded, a bounded wait that ran out) set flags in the
 *     workspace status header, read with gs_read_status.
 *   - Nothing throws across the ABI.
 *   - All per-Gaussian arrays are C-contiguous float32 (int32/uint32 where
 *     stated). Images are HWC float32.
 *   - Tiles are 16x16 pixels, tiles_x = ceil(width/16), tiles_y =
 *     ceil(height/16), tile id = ty * tiles_x + tx.
 *   - Host threads: entry points may be called from several host threads on
 *     different workspaces. gs_render_batch enqueues under one process-wide
 *     lock (its fork/join events are shared per device); gs_set_spin_limit is
 *     not thread-safe.
 *   - cudaDeviceReset: gs_render_batch keeps per-device fork/join events, and
 *     gs_render a per-thread second stream with its events, that a reset
 *     destroys; do not call them on a device after resetting that device
 *     in the same process. (gs_bin_static looks its scratch address up again
 *     on every call made outside stream capture.)
 */
#ifndef GS_B300_H
#define GS_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GS_ABI_VERSION 2

typedef enum gs_status {
    GS_OK = 0,
    GS_ERR_INVALID_ARG = 1,  /* bad pointer, size, degree, camera */
    GS_ERR_CAPACITY = 2,     /* more keys than key_capacity (count still reported) */
    GS_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    GS_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out */
    GS_ERR_WORKSPACE = 5     /* workspace missing, misaligned or too small */
} gs_status;

/* Workspace status flags (bit set). */
#define GS_FLAG_CAPACITY 1u
#define GS_FLAG_TIMEOUT 2u

/* Pinhole camera (host memory). x_cam = R x_world + t with R row-major;
 * camera x right, y down, z forward. Pixel (x, y) is sampled at the integer
 * coordinates (x, y), as the integer grid of rasterise_2d ("Étape 2") does.
 * near_z > 0: Gaussians with camera z <= near_z are culled. bg is the
 * background colour added with the final transmittance. */
typedef struct gs_camera {
    float R[9];
    float t[3];
    float fx, fy, cx, cy, near_z;
    int32_t width, height;   /* 1 .. 32768 */
    float bg[3];
} gs_camera;

/* Gaussian parameters (section "Ce qu'un Gaussien porte"). All device
 * pointers, 16-byte aligned (quats is read as float4).
 *   means          [n][3]  world-space centres mu
 *   quats          [n][4]  (w, x, y, z); normalised on the fly, so any
 *                          non-zero quaternion is accepted (zero -> culled)
 *   log_scales     [n][3]  s, scale = exp(s) at render time
 *   opacity_logits [n]     opacity = sigmoid(logit)
 *   sh             [n][(D+1)^2][3]  SH coefficient k of colour channel c
 *   sh_degree      D in 0..3 */
typedef struct gs_gaussians {
    const float* means;
    const float* quats;
    const float* log_scales;
    const float* opacity_logits;
    const float* sh;
    int64_t n;
    int32_t sh_degree;
} gs_gaussians;

/* Per-Gaussian output of the projection step (device pointers, caller
 * allocated, each [n] rows). depth, tiles_touched and rect are required; the
 * others may be NULL, and are then not written (gs_render writes only the
 * fields binning and compositing read). Alignment: mean2d 8 bytes,
 * conic_opacity and raster 16 bytes, rect 8 bytes.
 *   mean2d         [n][2]  projected centre mu' (pixels), the binary32 value of
 *                          the decision program (rectangles are cut from it)
 *   conic_opacity  [n][4]  (A, B, C, o): Sigma'^-1 = [[A, B], [B, C]], opacity o
 *   rgb            [n][3]  colour from SH along the view direction, + 0.5, >= 0
 *   depth          [n]     camera-space z (the sort key's low 32 bits)
 *   radius         [n]     ceil(3 sqrt(lambda_max(Sigma'))) pixels, 0 if culled
 *   tiles_touched  [n]     number of 16x16 tiles the pixel rectangle
 *                          [u-r, u+r] x [v-r, v+r] (clipped) covers, 0 if culled
 *   rect           [n][4]  uint16 tile rectangle (tx0, ty0, tx1, ty1), inclusive
 *   raster         [n][12] the compositor's packed record, written for
 *                          Gaussians with tiles_touched > 0 (required by
 *                          gs_rasterize): {u, v, du, dv} with mu' = (u + du,
 *                          v + dv) from a compensated (double-float) evaluation
 *                          of the projection, good to ~1e-9 px; {k1, k2, k3,
 *                          log2 o} with log2(alpha) = log2 o - (k1 dx)^2 -
 *                          (k2 dy + k3 dx)^2, the Gaussian's quadratic form as
 *                          a sum of two squares; {r, g, b, h} with h the bits of
 *                          a half2 holding the half-extents (rounded up) of a
 *                          box that contains every pixel offset where alpha can
 *                          reach 1/255 (+inf: no box, -1: never reaches it).
 * For culled Gaussians only radius and tiles_touched are defined (both 0). */
typedef struct gs_projected {
    float* mean2d;
    float* conic_opacity;
    float* rgb;
    float* depth;
    int32_t* radius;
    uint32_t* tiles_touched;
    uint16_t* rect;
    float* raster;
} gs_projected;

/* gs_status_string: a static, NUL-terminated English description of a
 * gs_status value ("unknown status" for any other number); never NULL, never
 * to be freed. gs_abi_version: GS_ABI_VERSION of the library that was loaded,
 * so a caller can refuse a library built from another version of this header.
 * Neither touches the GPU. */
const char* gs_status_string(int32_t status);
int32_t gs_abi_version(void);

/* Step 1 -- projection (sections "L'étape de projection", "Étape 5",
 * "Étape 6"). Per Gaussian: R from the normalised quaternion,
 * Sigma = R S S^T R^T, camera-space centre, near-plane cull, mu', the EWA
 * screen covariance Sigma' = J W Sigma W^T J^T, its inverse (the conic), the
 * 3-sigma radius, the pixel and tile rectangles, opacity = sigmoid(logit) and
 * the SH colour. The integer results (culling, depth bits, radius, rectangles)
 * come from a fixed binary32 program with no fused multiply-add, so they are
 * reproducible bit for bit on any IEEE machine.
 * Errors: GS_ERR_INVALID_ARG for null/misaligned pointers, n < 0,
 * sh_degree outside 0..3, a bad camera. */
gs_status gs_preprocess(const gs_gaussians* gaussians, const gs_camera* camera,
                        const gs_projected* out, void* stream);

/* Step 2 -- tile binning (flowchart box "Assign to tiles (16x16
 * screen-space)"). A device prefix scan of tiles_touched gives
 * offsets[i] = sum_{j<=i} tiles_touched[j] (inclusive) and the key count
 * K = offsets[n-1], written to *num_keys (device uint64). Then each Gaussian
 * i writes one key per touched tile, in row-major order over its tile
 * rectangle, at positions offsets[i]-tiles_touched[i] ...:
 *     key = (uint64)tile_id << 32 | float_bits(depth[i]),   value = i.
 * Keys beyond key_capacity are not written; K is still reported and
 * GS_FLAG_CAPACITY is set in the workspace header.
 * ws: device scratch of at least gs_bin_workspace_bytes(n), 256-byte aligned.
 * keys/vals: device, key_capacity entries each. */
size_t gs_bin_workspace_bytes(int64_t n);
gs_status gs_bin(const gs_projected* projected, int64_t n, const gs_camera* camera,
                 uint32_t* offsets, uint64_t* keys, uint32_t* vals, int64_t key_capacity,
                 uint64_t* num_keys, void* ws, size_t ws_bytes, void* stream);

/* Binning that allocates nothing (the pages have no counterpart: this is a
 * deployment variant of gs_bin). For callers that cannot allocate device
 * memory -- plugins whose host application owns all GPU memory through its
 * own pools, real-time loops that forbid cudaMalloc after start-up because it
 * can synchronise the device. Same inputs, outputs and results as gs_bin, but
 * the scratch lives in a file-scope device array of the library (65,792
 * bytes per device that loads the library, held until the process exits), so
 * there is no ws argument.
 *   - n must be <= GS_BIN_STATIC_MAX_GAUSSIANS, else GS_ERR_INVALID_ARG.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress with that device current); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array. Calls whose work overlaps
 *     on the GPU (e.g. issued on different streams without ordering) race and
 *     give wrong results; order them on one stream.
 *   - Capacity overflow is visible in the outputs: *num_keys > key_capacity
 *     means only the first key_capacity keys were written. */
#define GS_BIN_STATIC_MAX_GAUSSIANS 16777216
gs_status gs_bin_static(const gs_projected* projected, int64_t n, const gs_camera* camera,
                        uint32_t* offsets, uint64_t* keys, uint32_t* vals, int64_t key_capacity,
                        uint64_t* num_keys, void* stream);

/* Step 3 -- sort (flowchart box "Depth-sort per tile"). Stable ascending
 * least-significant-digit radix sort of the first min(K, key_capacity) (key,
 * value) pairs, K read from *num_keys on the device. Only the low key_bits
 * bits of the keys take part (1..64; the binning keys need 32 +
 * ceil(log2(tiles))). Equal keys keep their input order, which for binning
 * output is Gaussian-index order. The sorted pairs end in keys/vals;
 * keys_alt/vals_alt are ping-pong buffers of the same capacity.
 * ws: device scratch of at least gs_sort_workspace_bytes(key_capacity).
 * A bounded wait that runs out sets GS_FLAG_TIMEOUT (the output is then
 * unspecified but every access stays in bounds). */
size_t gs_sort_workspace_bytes(int64_t key_capacity);
gs_status gs_sort(uint64_t* keys, uint32_t* vals, uint64_t* keys_alt, uint32_t* vals_alt,
                  const uint64_t* num_keys, int64_t key_capacity, int32_t key_bits,
                  void* ws, size_t ws_bytes, void* stream);

/* Step 4 -- per-tile ranges: ranges[t] = [first, one past last) position of
 * tile id t in the sorted keys, (0, 0) for tiles without keys.
 * ranges: device uint32 [tiles_y * tiles_x][2]. */
gs_status gs_tile_ranges(const uint64_t* sorted_keys, const uint64_t* num_keys,
                         int64_t key_capacity, const gs_camera* camera, uint32_t* ranges,
                         void* stream);

/* Depth-first variant of steps 2-4, used by gs_render. Sorting the N
 * Gaussians by depth once, then emitting each Gaussian's tiles in that order
 * and sorting stably by tile id alone, gives exactly the per-tile order of
 * steps 2-4 (tile, then depth bits, then Gaussian index) while moving 32-bit
 * keys of ceil(log2(tiles)) bits instead of 64-bit keys of 32 + that many.
 *
 * gs_depth_order: order[0..n) = the Gaussian indices sorted by (float bits of
 * depth, index) -- a stable sort of the depth bits -- with the Gaussians that
 * touch no tile (tiles_touched == 0) last, in index order. Reads depth and
 * tiles_touched of `projected`. ws: >= gs_depth_order_workspace_bytes(n).
 *
 * gs_bin_ordered: step 2 over the Gaussians in the given order (n entries of
 * `order`): for each, in order, one 32-bit key per touched tile holding the
 * tile id (row-major over the rectangle), value = Gaussian index. K goes to
 * *num_keys; offsets (nullable) receives the inclusive prefix sums in list
 * order. Capacity rules as gs_bin; ws: >= gs_bin_ordered_workspace_bytes(n,
 * key_capacity). The keys are written load-balanced by key slot (one block
 * per 2048 slots), so Gaussians with many tiles do not stall a block.
 *
 * gs_sort32: gs_sort for 32-bit keys (key_bits 1..32). num_keys may be NULL,
 * in which case key_capacity is the key count. ws: >= gs_sort_workspace_bytes.
 *
 * gs_tile_ranges32: step 4 (as gs_tile_ranges) for sorted 32-bit tile-id
 * keys: sorted_tiles is device uint32 [key_capacity], of which the first
 * min(*num_keys, key_capacity) are read; any 4-byte alignment (16-byte
 * aligned arrays are read with vector loads). ranges: device uint32
 * [tiles_y * tiles_x][2], 8-byte aligned. */
size_t gs_depth_order_workspace_bytes(int64_t n);
size_t gs_bin_ordered_workspace_bytes(int64_t n, int64_t key_capacity);
gs_status gs_depth_order(const gs_projected* projected, int64_t n, uint32_t* order, void* ws,
                         size_t ws_bytes, void* stream);
gs_status gs_bin_ordered(const gs_projected* projected, int64_t n, const uint32_t* order,
                         const gs_camera* camera, uint32_t* offsets, uint32_t* tile_keys,
                         uint32_t* vals, int64_t key_capacity, uint64_t* num_keys, void* ws,
                         size_t ws_bytes, void* stream);
gs_status gs_sort32(uint32_t* keys, uint32_t* vals, uint32_t* keys_alt, uint32_t* vals_alt,
                    const uint64_t* num_keys, int64_t key_capacity, int32_t key_bits, void* ws,
                    size_t ws_bytes, void* stream);
gs_status gs_tile_ranges32(const uint32_t* sorted_tiles, const uint64_t* num_keys,
                           int64_t key_capacity, const gs_camera* camera, uint32_t* ranges,
                           void* stream);

/* Step 5 -- composite (sections "La règle de composition alpha", "Étape 2").
 * Each pixel walks its tile's sorted list front to back:
 *     alpha = min(0.99, o exp(-0.5 d^T Sigma'^-1 d)), d = pixel - mu';
 *     skipped if alpha < 1/255; C += alpha T c; T *= (1 - alpha);
 *     the pixel stops once T < 1e-4 (after that Gaussian);
 *     image = C + T * bg.
 * image: device float [height][width][3]. final_T (device float [h][w]) and
 * n_contrib (device uint32 [h][w], 1 + list position of the last
 * contributing Gaussian, 0 if none) may be NULL.
 * tile_order: NULL, or device uint32 [tiles_x * tiles_y] scratch (caller
 * owned, contents on entry ignored); when given, a first kernel orders the
 * tiles by decreasing list length (bucketed by floor(log2 length)) and the
 * tiles are launched in that order, which shortens the last wave. The image
 * does not depend on it. */
gs_status gs_rasterize(const gs_projected* projected, int64_t n, const uint32_t* sorted_vals,
                       const uint32_t* ranges, const gs_camera* camera, float* image,
                       float* final_T, uint32_t* n_contrib, uint32_t* tile_order, void* stream);

/* The whole frame: step 1, steps 2-4 in one of two orders, and step 5, chained
 * on `stream` with no host synchronisation (so the call can be captured into a
 * CUDA graph). Depth-first (as gs_depth_order, gs_bin_ordered, gs_sort32,
 * gs_tile_ranges32): the Gaussians are sorted by depth, binned in that order
 * and stably sorted by tile. From 4096 tiles up the tile sort's keys number
 * the 8x4-tile block in their low digit and the tile inside it above, which
 * orders the tiles' lists differently in the array, not their contents. For
 * frames of at most 2^21 Gaussians whose tile grid's difference array fits in
 * 96 KB of shared memory (up to about 2560x1440), the tile ranges and the
 * tiles' launch order are computed from the tile rectangles on a second
 * stream that the library owns (one per host thread and device, created on
 * the thread's first such frame outside a stream capture), forked from
 * `stream` after the projection and joined back before they are needed;
 * inside a CUDA graph capture the fork and the join become graph edges. A
 * frame captured before its thread has that stream runs on `stream` alone. Tile-first, for short tile lists (see
 * gs_render_tile_first): binned in index order, stably sorted by tile, then
 * each tile's list is sorted by (depth bits, index) on its own. Both give the
 * same per-tile lists bit for bit. The image equals the one of the staged path
 * gs_preprocess/gs_bin/gs_sort/gs_tile_ranges/gs_rasterize bit for bit. All
 * intermediates live in ws (device, 256-byte aligned, at least
 * gs_render_workspace_bytes(n, width, height, key_capacity) bytes); the first
 * 256 bytes of ws are the status header read by gs_read_status.
 * key_capacity bounds the (Gaussian, tile) pairs of the frame; if the frame
 * needs more, GS_FLAG_CAPACITY is set, the image is unspecified and
 * gs_read_status reports the count needed. */
/* Limits: n and key_capacity at most 2^30 - 1 (the radix sort's look-back
 * words keep 30-bit counts); GS_ERR_INVALID_ARG above. */
size_t gs_render_workspace_bytes(int64_t n, int32_t width, int32_t height, int64_t key_capacity);
gs_status gs_render(const gs_gaussians* gaussians, const gs_camera* camera, int64_t key_capacity,
                    void* ws, size_t ws_bytes, float* image, float* final_T,
                    uint32_t* n_contrib, void* stream);

/* 1 if gs_render takes the tile-first order of steps 2-4 for these sizes, 0 if
 * depth-first: tile-first when key_capacity is at most 2^20 pairs (the
 * frame's four global depth-sort passes would be short, latency-bound
 * launches), unless gs_set_steps_order pins an order. Host-only arithmetic
 * (no CUDA call). */
int32_t gs_render_tile_first(int64_t n, int32_t width, int32_t height, int64_t key_capacity);

/* Programmatic dependent launch (on by default): every kernel is launched
 * with the programmatic-serialisation attribute, so that its launch overlaps
 * the end of the kernel before it on the stream (inside a CUDA graph the
 * dependencies become programmatic edges); each kernel waits in hardware for
 * its predecessor's completion before it touches memory, so results are the
 * same bit for bit either way. 0 turns the attribute off for launches made
 * after the call (for measurement and tests). Process-wide; not thread-safe
 * against concurrent launches. */
void gs_set_programmatic_launch(int32_t on);

/* Pins the order of steps 2-4 for gs_render, gs_render_profiled and
 * gs_render_batch frames enqueued after the call: 0 automatic (the default,
 * gs_render_tile_first), 1 depth-first, 2 tile-first. Either order gives the
 * same lists and image bit for bit; the pin is for tests and measurement.
 * Process-wide; GS_ERR_INVALID_ARG for other values. */
gs_status gs_set_steps_order(int32_t order);

/* Where a gs_render (or one view of gs_render_batch) workspace keeps the
 * frame's per-tile lists: *sorted_vals receives the device address of the
 * frame's K Gaussian indices -- valid after a frame, K as gs_read_status
 * reports it -- and *ranges that of the tile ranges (uint32 [tiles_y *
 * tiles_x][2], [start, end) into the sorted list). Tile t's list is
 * sorted_vals[ranges[t][0] .. ranges[t][1]), sorted by (depth bits, index),
 * and the lists tile [0, K). From 4096 tiles up the lists are laid out in the
 * order of the frame's tile keys (8x4-tile blocks in the low digit), not by
 * tile id; below that, by tile id. n, width, height and key_capacity must be those the workspace
 * was sized with (gs_render_workspace_bytes). Host-only arithmetic on ws; no
 * CUDA call. The lists are the ones the pages' step "Depth-sort per tile"
 * produces (section "Rastérisation, non rayée"). */
gs_status gs_render_workspace_lists(const void* ws, int64_t n, int32_t width, int32_t height,
                                    int64_t key_capacity, const uint32_t** sorted_vals,
                                    const uint32_t** ranges);

/* gs_render that also records CUDA events at its stage boundaries, for
 * per-stage timing of the very launches a frame makes. events[0..6] are
 * caller-created cudaEvent_t handles (as void*), recorded on `stream`, in the
 * order of the steps the frame takes (gs_render_tile_first):
 *   depth-first: 0 start (after the frame's setup memsets: status header and
 *   the depth digits' histograms), 1 after projection, 2 after the depth order
 *   of the Gaussians, 3 after binning, 4 after the tile sort, 5 after the
 *   ranges and the tiles' launch order, 6 after compositing (the compositing
 *   kernel alone);
 *   tile-first: 0 start, 1 after projection, 2 after binning, 3 after the tile
 *   sort, 4 after the ranges and the tiles' launch order, 5 after the per-tile
 *   depth sort, 6 after compositing.
 * n_events must be >= GS_RENDER_STAGES + 1. */
#define GS_RENDER_STAGES 6
gs_status gs_render_profiled(const gs_gaussians* gaussians, const gs_camera* camera,
                             int64_t key_capacity, void* ws, size_t ws_bytes, float* image,
                             float* final_T, uint32_t* n_contrib, void* stream,
                             void* const* events, int32_t n_events);

/* Several views of the same Gaussians in one call (the multi-view workloads:
 * orbit poses of one scene). Step 1 runs once for all views: one pass over
 * the parameters projects each Gaussian for every camera (the 236 B per
 * Gaussian are read from HBM once, not once per view). Steps 2-5 of each view
 * then run on streams[v % n_streams], so the views' latency-bound passes (the
 * radix sorts' look-back chains) overlap on the GPU.
 * cameras[views]: same width and height. images: device float
 * [views][h][w][3]; final_T / n_contrib: NULL or [views][h][w].
 * ws: views consecutive gs_render workspaces; view v's (and its status header,
 * read with gs_read_status) starts at ws + v * gs_render_workspace_bytes(n,
 * width, height, key_capacity); key_capacity applies to each view.
 * streams[0..n_streams-1] (1 <= n_streams <= 8): the call is ordered after
 * the work already queued on streams[0], and everything it launches is joined
 * back into streams[0] (fork/join events are created once per device on first
 * use). Each view's image equals gs_render's for that camera bit for bit.
 * 1 <= views <= GS_MAX_BATCH_VIEWS. */
#define GS_MAX_BATCH_VIEWS 64
size_t gs_render_batch_workspace_bytes(int64_t n, int32_t width, int32_t height, int64_t key_capacity,
                                       int32_t views);
gs_status gs_render_batch(const gs_gaussians* gaussians, const gs_camera* cameras, int32_t views,
                          int64_t key_capacity, void* ws, size_t ws_bytes, float* images, float* final_T,
                          uint32_t* n_contrib, void* const* streams, int32_t n_streams);

/* The whole frame from host memory: copies the five parameter arrays from
 * host to the caller's device buffers in `device_gaussians` (same n and
 * degree), renders with gs_render, and copies the image back to host_image
 * (host float [h][w][3]). All copies are cudaMemcpyAsync on `stream`; host
 * buffers should be page-locked for them to overlap. device_image is the
 * device image buffer. The call does not wait for the stream. */
gs_status gs_render_from_host(const gs_gaussians* host_gaussians,
                              const gs_gaussians* device_gaussians, const gs_camera* camera,
                              int64_t key_capacity, void* ws, size_t ws_bytes,
                              float* device_image, float* host_image, void* stream);

/* ---------------------------------------------------------------- backward
 * Section "Rastérisation, non rayée": every stage of the renderer is
 * differentiable, so the parameters can be fitted by gradient descent. The
 * calls below return the gradient of a scalar loss L(image) given
 * grad_image = dL/dimage (device float [h][w][3]), by the chain rule through
 * the forward's functions with its discrete decisions (culling, tile lists,
 * the 1/255 skip, the 1e-4 stop) held fixed. The forward's 0.99 cap gives a
 * zero derivative where it is active. Gradient sums over pixels use float
 * atomics, so their rounding order (not their value beyond rounding) varies
 * between runs. All arrays are device arrays owned by the caller. */

/* dL/d of the per-Gaussian projected quantities (step 1 outputs):
 *   mean2d  [n][2] dL/d(u, v)
 *   conic   [n][3] dL/d(A, B, C) of conic = Sigma'^-1 = [[A, B], [B, C]]
 *   opacity [n]    dL/do, o = sigmoid(logit)
 *   rgb     [n][3] dL/dc (the clamped SH colour) */
typedef struct gs_projected_grad {
    float* mean2d;
    float* conic;
    float* opacity;
    float* rgb;
} gs_projected_grad;

/* dL/d of the parameters, same layouts as gs_gaussians (quats (w, x, y, z),
 * sh [n][(D+1)^2][3]); every entry is written (zero for Gaussians that
 * touch no tile). */
typedef struct gs_gaussians_grad {
    float* means;
    float* quats;
    float* log_scales;
    float* opacity_logits;
    float* sh;
} gs_gaussians_grad;

/* Step 5 backward. projected, sorted_vals, ranges: as given to gs_rasterize
 * (after the forward of the same frame); final_T and n_contrib: the forward's
 * outputs (device [h][w]). tile_order: NULL, or the tile_order scratch the
 * forward filled (launch order only). Zeroes the four arrays of `grad`, then
 * accumulates into them. */
gs_status gs_rasterize_backward(const gs_projected* projected, int64_t n, const uint32_t* sorted_vals,
                                const uint32_t* ranges, const gs_camera* camera,
                                const float* final_T, const uint32_t* n_contrib,
                                const float* grad_image, const uint32_t* tile_order,
                                const gs_projected_grad* grad, void* stream);

/* Step 1 backward: maps grad_in (from gs_rasterize_backward) to the
 * parameters. projected->tiles_touched (from gs_preprocess of the same frame)
 * marks the Gaussians that enter the image. */
gs_status gs_preprocess_backward(const gs_gaussians* gaussians, const gs_camera* camera,
                                 const gs_projected* projected, const gs_projected_grad* grad_in,
                                 const gs_gaussians_grad* grad_out, void* stream);

/* Backward of a gs_render frame: uses the intermediates that gs_render left
 * in ws (same gaussians, camera and key_capacity, ws not reused in between)
 * and the final_T / n_contrib it wrote. Chains gs_rasterize_backward and
 * gs_preprocess_backward on `stream`; the projected gradients live in ws. */
gs_status gs_render_backward(const gs_gaussians* gaussians, const gs_camera* camera,
                             int64_t key_capacity, void* ws, size_t ws_bytes, const float* final_T,
                             const uint32_t* n_contrib, const float* grad_image,
                             const gs_gaussians_grad* grad_out, void* stream);

/* ---------------------------------------------------------------- 2D splats
 * Section "Étape 2" (rasterise_2d) and "Étape 3" (a trainable 2D scene): n
 * Gaussians given directly in image space, composited on the tile pipeline.
 *   means     [n][2]    (x, y) in pixels (8-byte aligned)
 *   covs      [n][2][2] image-space covariance (the off-diagonal is taken as
 *                       the mean of the two entries)
 *   colours   [n][3]    in [0, 1];  opacities [n] in (0, 1]
 *   depths    [n]       any real; only orders the Gaussians, smallest first
 *                       (ties by index)
 * alpha = min(0.99, o exp(-0.5 d^T cov^-1 d)) at the integer pixel (x, y);
 * out = sum alpha_i T_i c_i with no background term (zero background). The
 * tile renderer's cut-offs apply: each Gaussian covers the tiles of its
 * 3-sigma rectangle, alpha < 1/255 is skipped, a pixel stops once T < 1e-4.
 * ws: >= gs_render_workspace_bytes(n, width, height, key_capacity), key
 * capacity and status header as for gs_render. image [h][w][3]; final_T and
 * n_contrib may be NULL (the backward needs them). */
gs_status gs_rasterize_2d(const float* means, const float* covs, const float* colours,
                          const float* opacities, const float* depths, int64_t n, int32_t width,
                          int32_t height, int64_t key_capacity, void* ws, size_t ws_bytes, float* image,
                          float* final_T, uint32_t* n_contrib, void* stream);

/* Backward of the last gs_rasterize_2d on ws (same inputs, ws not reused in
 * between): dL/dmeans [n][2], dL/dcovs [n][2][2] (the off-diagonal gradient
 * split evenly over the two entries), dL/dcolours [n][3], dL/dopacities [n],
 * all written (zero for Gaussians that touch no tile). The depths get no
 * gradient: they only order the Gaussians. */
gs_status gs_rasterize_2d_backward(const float* covs, int64_t n, int32_t width, int32_t height,
                                   int64_t key_capacity, void* ws, size_t ws_bytes,
                                   const float* final_T, const uint32_t* n_contrib,
                                   const float* grad_image, float* grad_means, float* grad_covs,
                                   float* grad_colours, float* grad_opacities, void* stream);

/* ---------------------------------------------------------------- densify / prune
 * Section "Densation et taille": every N iterations, clone a Gaussian whose
 * gradient magnitude is high but whose scale is small, split a large one with
 * a high gradient into two smaller ones, prune those whose opacity fell below
 * a threshold.
 *
 * gs_densify_stats: accumulates, for every Gaussian that touched a tile in
 * the frame (projected->tiles_touched > 0), |dL/d(u, v)| into accum[n] and 1
 * into count[n] (device; zero them at the start of a densification period).
 * grad_mean2d: the gs_projected_grad mean2d of the frame's backward [n][2]. */
gs_status gs_densify_stats(const float* grad_mean2d, const uint32_t* tiles_touched, int64_t n,
                           float* accum, uint32_t* count, void* stream);

/* Writable parameter arrays (layouts as gs_gaussians) with room for n
 * Gaussians. */
typedef struct gs_gaussians_out {
    float* means;
    float* quats;
    float* log_scales;
    float* opacity_logits;
    float* sh;
    int64_t n;
    int32_t sh_degree;
} gs_gaussians_out;

/* The densification step, as one stable compaction of `in` into `out`:
 *   prune  o < prune_opacity  (o = sigmoid(logit))
 *   else, with g = accum / count (0 if count = 0):
 *   clone  g >= grad_threshold and max(exp(log_scale)) <= scale_threshold:
 *          the Gaussian and an exact copy right after it
 *   split  g >= grad_threshold and max scale > scale_threshold: two children
 *          at mu + R S xi_c (c = 0, 1) with log_scales - log(1.6), the other
 *          parameters copied; xi: device float [in->n][2][3] standard normal
 *          samples supplied by the caller (only split Gaussians read theirs)
 *   keep   otherwise.
 * Survivors keep the input order; children replace their parent. The tests
 * are taken on logit < log(t/(1-t)) and max log_scale > log(scale_threshold)
 * (thresholds mapped on the host, in double, then rounded to float), so the
 * decisions are exact. out->n is the capacity (2 * in->n always suffices);
 * out->sh_degree must equal in->sh_degree. *out_count (device uint64) gets
 * the new count; if it exceeds the capacity GS_FLAG_CAPACITY is set in the
 * workspace header and the out arrays are unspecified. action (device uint8
 * [in->n], nullable): 0 keep, 1 clone, 2 split, 3 prune.
 * ws: >= gs_densify_workspace_bytes(in->n); the first 256 bytes are the status
 * header read by gs_read_status. */
size_t gs_densify_workspace_bytes(int64_t n);
gs_status gs_densify(const gs_gaussians* in, const float* accum, const uint32_t* count,
                     const float* xi, float grad_threshold, float scale_threshold,
                     float prune_opacity, const gs_gaussians_out* out, uint64_t* out_count,
                     uint8_t* action, void* ws, size_t ws_bytes, void* stream);

/* Frames from host memory with the copies overlapped: a two-deep pipeline
 * over a sequence of calls with frame = 0, 1, 2, ... . Frame k copies the
 * host parameters into device_sets[k % 2] on streams[1], renders from that set
 * with gs_render on streams[0] once the copy is in (and the previous frame's
 * image has been read back), and copies the image to host_image on streams[2]
 * once it is rendered. So frame k + 1's parameter upload runs during frame
 * k's render and read-back, and throughput is bound by the upload alone.
 * device_sets[2]: two device parameter sets with the same n and degree as
 * host_gaussians. streams[3]: render, upload, read-back (distinct). events[6]:
 * caller-created cudaEvent_t handles (timing may be disabled), reused across
 * the calls of one pipeline: upload done per set [0..1], render done per set
 * [2..3], image ready [4], image read back [5]. host buffers should be
 * page-locked. No call waits for the GPU; host_image of frame k is complete
 * once streams[2] has passed that frame (e.g. after a synchronisation). */
gs_status gs_render_from_host_async(const gs_gaussians* host_gaussians,
                                    const gs_gaussians* device_sets, int64_t frame,
                                    const gs_camera* camera, int64_t key_capacity, void* ws,
                                    size_t ws_bytes, float* device_image, float* host_image,
                                    void* const* streams, void* const* events);

/* Debug build (libgs_b300_debug.so, compiled with GS_DEBUG_CHECKS): the
 * kernels check their index invariants -- tile ranges ordered, list entries
 * naming a Gaussian of the scene, sort destinations inside the key count,
 * expansion slots inside the capacity, tile ids inside the image -- and add 1
 * to *device_counter (device uint64, zeroed by the caller) for each failure,
 * instead of trapping. gs_debug_set_check_counter sets the counter for the
 * current device (NULL turns counting off); gs_debug_checks_enabled returns 1
 * in the debug build and 0 in the release build (where the call does nothing). */
int32_t gs_debug_checks_enabled(void);
gs_status gs_debug_set_check_counter(uint64_t* device_counter);

/* The key gs_render's tile sort gives tile (tx, ty) of a tiles_x x tiles_y grid
 * (the tile id ty * tiles_x + tx below 4096 tiles; from 4096 tiles up the
 * block of 8 x 4 tiles in the low bits and the tile inside it above), the
 * number of key bits, and the tile id of a key (-1 for a key no tile has).
 * Host-only arithmetic, the device code's own functions; -1 for arguments
 * outside the grid. For tests of the key layout. */
int64_t gs_debug_tile_key(int32_t tiles_x, int32_t tiles_y, int32_t tx, int32_t ty);
int32_t gs_debug_tile_key_bits(int32_t tiles_x, int32_t tiles_y);
int64_t gs_debug_tile_of_key(int32_t tiles_x, int32_t tiles_y, int64_t key);

/* Reads the status header at the start of a gs_bin, gs_sort or gs_render
 * workspace. SYNCHRONISES `stream`. flags/num_keys may be NULL. Returns
 * GS_ERR_TIMEOUT, GS_ERR_CAPACITY or GS_OK from the flags. num_keys is the
 * key count of the last gs_bin/gs_render on that workspace. */
gs_status gs_read_status(const void* ws, void* stream, uint32_t* flags, uint64_t* num_keys);

/* The boundary's names for two of the calls above:
 *   gs_workspace_bytes(n, width, height, key_capacity) ==
 *       gs_render_workspace_bytes(n, width, height, key_capacity);
 *   gs_last_device_status(ws): the flags of a gs_render / gs_bin / gs_sort
 *       workspace as gs_read_status returns them, after a cudaDeviceSynchronize
 *       (so the work of every stream of the device is included). SYNCHRONISES
 *       the device. */
size_t gs_workspace_bytes(int64_t n, int32_t width, int32_t height, int64_t key_capacity);
gs_status gs_last_device_status(const void* ws);

/* FP32 peak probe (a measurement utility; the pages have no counterpart). The
 * compositing step is bound by FP32 issue, so its roofline needs the rate of
 * fused multiply-adds the device sustains. This launches `blocks` blocks of
 * 256 threads; each thread runs 16 independent FMA chains for `iterations`
 * steps, as one fma.rn.f32 per chain and step, or with packed != 0 as one
 * fma.rn.f32x2 per pair of chains. *fma_count (host, may be NULL) receives the
 * number of FMAs the launch executes (2 flops each). Time it with events on
 * `stream`. sink: device float[blocks * 256], never written in practice.
 * 1 <= blocks <= 2^20, iterations >= 1. */
gs_status gs_fp32_peak_probe(int32_t blocks, int32_t iterations, int32_t packed, float* sink,
                             int64_t* fma_count, void* stream);

/* Upper bound on the wait of every device-side spin (look-back of the radix
 * sort), in polling iterations; <= 0 restores the default (about a second).
 * Applies to launches made after the call; not thread-safe. */
void gs_set_spin_limit(int64_t iterations);

/* Test hook: launches one block whose wait on a flag in ws (which nothing
 * sets) runs out after `iterations` polls; sets GS_FLAG_TIMEOUT in the ws
 * status header. ws: at least 256 bytes. */
gs_status gs_test_spin_timeout(void* ws, int64_t iterations, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GS_B300_H */
