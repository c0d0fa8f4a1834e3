"""Benchmark: frames/s of the forward renderer on the 1M-Gaussian, SH degree 3,
1920x1080 workload (one orbit view), through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config 1M|100k|5M|stress|tiny] [--no-graph] [--no-cpu-baseline]

Prints ONE JSON line (rank 0). A step is one whole frame (projection, binning,
sort, ranges, compositing) of gs_render, replayed from a CUDA graph, with the
scene resident in HBM (236 MB of parameters: larger than the 126 MB L2, so no
flush is needed between frames). Per-stage CUDA-event times come from a
second pass of K frames through the stage entry points on the same stream.
`e2e` renders the same frames through gs_render_from_host: the parameters are
copied from pinned host memory and the image read back inside the timed
region. Under torchrun each rank renders its own replica (independent frames:
replicas only, no collective on the data path).

The FP32 roofline of the compositing step is taken against the FMA rate that
gs_fp32_peak_probe measures on the same GPU in the same run (scalar and packed
FMA chains; the higher rate). The `configs` block repeats the frame and stage
measurement for every view of every workload (tiny, 100k, 1M, 5M x 4 views,
stress x 8 views) with the per-view and mean figures; it runs at N=1 only.

--impl reference times the CPU oracle (the plain fp64 renderer) on the host
cores on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6400.0
# FP32 work per evaluated (pixel, Gaussian) pair, counted two ways:
# - the method's count: dx, dy, the quadratic form with its cross term, the -1/2 scale, the
#   opacity product, the 0.99 cap and the 1/255 test, 15 flops (an FMA is 2), against the
#   measured FMA rate x 2 flops;
FLOPS_PER_EVAL = 15
# - the kernel's count: dx, dy (2), the exponent with the conic pre-scaled (5), min with 0.99
#   (1), the 1/255 test (1), 9 FP32 lane operations, against the measured FMA rate (one
#   operation per lane and cycle).
OPS_PER_EVAL = 9
PARAM_BYTES_PER_G = 12 + 16 + 12 + 4 + 192       # SH degree 3
# what the projection writes per Gaussian: the method's record (mean2d 8, conic + opacity 16,
# rgb 12, depth 4, radius 4, tiles touched 4 = 48 B) ...
PROJ_BYTES_METHOD = 8 + 16 + 12 + 4 + 4 + 4
# ... and this implementation's (depth 4, tiles touched 4, tile rectangle 8, the 48-byte raster record)
PROJ_BYTES_PER_G = 4 + 4 + 8 + 48


def metric_name(cfg) -> str:
    n = f"{cfg.n // 10**6}M" if cfg.n >= 10**6 else f"{cfg.n // 1000}k" if cfg.n >= 1000 else str(cfg.n)
    return f"frames/s at {cfg.width}x{cfg.height}, {n} Gaussians SH{cfg.sh_degree}"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="1M")
    ap.add_argument("--view", type=int, default=0)
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-batch", action="store_true")
    ap.add_argument("--no-densify", action="store_true")
    ap.add_argument("--no-toy", action="store_true")
    ap.add_argument("--batch-streams", type=int, default=4)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-single-thread", action="store_true", help="skip the one-thread oracle frame")
    ap.add_argument("--configs", default="tiny,100k,1M,5M,stress",
                    help="workloads of the configs block (every view of each); empty for none")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the raw nvidia-smi samples of the timed region in this file "
                         "(a {rank} field is filled in); by default they go to a temporary file")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def rank_view(view0: int, rank: int, n_views: int) -> int:
    """The view a rank renders: replicas of a one-view scene, views dealt out
    round-robin for multi-view scenes (independent frames, no exchange)."""
    return (view0 + rank) % n_views


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank number over all ranks (the job takes as long as its slowest rank)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(frame_ms_max: float, world: int) -> float:
    """Whole-job frames/s: every rank renders one frame per step, a step lasts
    as long as the slowest rank's frame."""
    return world * 1e3 / frame_ms_max


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", d
    except Exception:
        return FALLBACK_HBM_GBS, "fallback", {}


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path=None):
        self.gpu = gpu_index
        self.proc = None
        self.fh = None
        self.keep = path is not None
        if path is None:
            fd, path = tempfile.mkstemp(prefix=f"gs_clocks_{gpu_index}_", suffix=".csv")
            os.close(fd)
        self.path = path

    def __enter__(self):
        try:
            d = os.path.dirname(self.path)
            if d:
                os.makedirs(d, exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.fh is not None:
            self.fh.close()
            self.fh = None

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    rows.append(parts)
        except Exception:
            pass
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        load = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        sm = [num(r[1]) for r in load if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in load:
            for i, n in enumerate(names):
                if r[6 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": sorted(reasons), "samples": len(rows),
                "samples_under_load": len(load),
                "power_w_max": max((num(r[3]) or 0) for r in rows)}


def sort_launches(key_bits: int) -> int:
    """Kernels of one 32-bit sort: the digit bases, one pass per 8-bit digit, a copy back after
    an odd pass count."""
    passes = (key_bits + 7) // 8
    return 1 + passes + passes % 2


def tile_depth_launches(key_capacity: int) -> int:
    """Kernels of a tile-first frame's per-tile depth sort: one per list-size class the key
    capacity allows (up to 512, 2048 and 8192 entries, and longer)."""
    if key_capacity <= 1:
        return 0
    return 1 + (key_capacity > 512) + (key_capacity > 2048) + (key_capacity > 8192)


def tile_key_bits(tiles_x: int, tiles_y: int) -> int:
    """Bits of the frame's tile-sort keys: the tile id below 4096 tiles, else the number of
    the block of 8 x 4 tiles and 5 bits for the tile inside the block."""
    tiles = tiles_x * tiles_y
    if tiles < 4096:
        return max(1, (tiles - 1).bit_length())
    blocks = -(-tiles_x // 8) * -(-tiles_y // 4)
    return max(1, (blocks - 1).bit_length()) + 5


def side_ranges(n: int, tiles_x: int, tiles_y: int) -> bool:
    """Whether a gs_render frame computes its tile ranges from the tile rectangles on a
    second stream: up to 2^21 Gaussians, when the tile grid's difference array fits in 96 KB
    of shared memory."""
    return n <= (1 << 21) and (tiles_x + 1) * (tiles_y + 1) * 4 <= 96 * 1024


def frame_launches(tiles: int, tile_first: bool = False, key_capacity: int = 1 << 20, tiles_xy=None,
                   n: int = 0) -> int:
    """Kernels one gs_render frame launches for an image of `tiles` 16x16 tiles (tiles_xy:
    its tiles_x, tiles_y, for the tile keys' width; without it, the tile id's): preprocess
    (which, depth-first, also writes the depth keys); depth-first, the depth sort (4 passes);
    5 binning kernels; the tile-key sort; ranges; the tile order (count and scatter kernels up
    to 186 blocks of 256 tiles, one kernel beyond); tile-first, the per-tile depth sort
    (tile_depth_launches); rasterize. The ranges and the order run on a second stream when
    side_ranges(n, *tiles_xy) holds; they are counted here all the same."""
    tile_bits = tile_key_bits(*tiles_xy) if tiles_xy else max(1, (tiles - 1).bit_length())
    order = 2 if -(-tiles // 256) <= 186 else 1
    depth = tile_depth_launches(key_capacity) if tile_first else sort_launches(32)
    # the ranges: one kernel over the sorted keys, or, when the tile grid's difference
    # array fits in 96 KB of shared memory, two on the side stream (lengths, then ranges)
    ranges = 2 if tiles_xy and side_ranges(n, *tiles_xy) else 1
    return 1 + depth + 5 + sort_launches(tile_bits) + ranges + order + 1


def code_hash(files) -> str:
    """sha256 (16 hex digits) of the code of the given csrc files, comments and whitespace
    removed, so that a comment edit does not void counters taken on the same code."""
    h = hashlib.sha256()
    for name in files:
        src = open(os.path.join(ROOT, "gaussian_splatting_tile_02_b300", "csrc", name)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def traffic_from_profile(profile: str, workload: str):
    """Per-launch DRAM bytes recorded in a committed ncu summary, if the summary was taken on
    this workload and the code of the files it names is unchanged since."""
    try:
        rec = {}
        with open(os.path.join(ROOT, "profiles", profile)) as f:
            for line in f:
                if ":" in line and line.startswith("- "):
                    k, v = line[2:].split(":", 1)
                    rec[k.strip()] = v.strip()
        if rec.get("workload") == workload and rec.get("code_sha256_16") == code_hash(rec["code_files"].split()):
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def backward_summary(bwd, n, hbm_peak, fp32_peak):
    """Backward of one frame (gs_render_backward): whole time, and its two steps.
    Step 1 backward is HBM-bound: 236 B of parameters + 36 B of projected
    gradients + 4 B tile count read, 236 B of parameter gradients written per
    Gaussian. Step 5 backward walks every pixel's list up to its last
    contributor; 9 FP32 ops per walked entry (the forward's exponent) is a
    lower bound on its arithmetic, the gradient terms of contributing pairs
    come on top."""
    if bwd is None:
        return None
    pre_ms = bwd["preprocess_backward_ms"]
    ras_ms = max(bwd["ms"] - pre_ms, 1e-9)
    pre_bytes = (PARAM_BYTES_PER_G + 36 + 4 + PARAM_BYTES_PER_G) * n
    walked = bwd["n_contrib_sum"]
    ras_tops = OPS_PER_EVAL * walked / (ras_ms * 1e-3) / 1e12
    return {"ms": bwd["ms"], "frames_per_s": 1e3 / bwd["ms"], "steps": bwd["steps"],
            "preprocess_backward": {"ms": pre_ms, "bound": "hbm", "bytes": pre_bytes,
                                    "GB/s": pre_bytes / (pre_ms * 1e-3) / 1e9,
                                    "frac": pre_bytes / (pre_ms * 1e-3) / 1e9 / hbm_peak},
            "rasterize_backward": {"ms": ras_ms, "bound": "alu", "walked_entries": walked,
                                   "ops_lower_bound": OPS_PER_EVAL * walked, "Top/s": ras_tops,
                                   "frac": ras_tops / fp32_peak}}


def densify_summary(dens, sh_degree, hbm_peak):
    """Densification step, per input Gaussian: the decision pass reads the
    logit and log-scales (16 B) and the statistics (8 B); the scatter reads
    the parameters once and the split samples (24 B), and writes the
    parameters once per output copy."""
    if dens is None:
        return None
    p = 4 * (3 + 4 + 3 + 1 + 3 * (sh_degree + 1) ** 2)
    nbytes = dens["n_in"] * (16 + 8 + p + 24) + dens["n_out"] * p
    return {"ms": dens["ms"], "n_in": dens["n_in"], "n_out": dens["n_out"], "bound": "hbm", "bytes": nbytes,
            "GB/s": nbytes / (dens["ms"] * 1e-3) / 1e9, "frac": nbytes / (dens["ms"] * 1e-3) / 1e9 / hbm_peak}


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from gaussian_splatting_tile_02_b300 import scenes
    cfg = scenes.CONFIGS[args.config]
    scene = scenes.make_scene(cfg)
    cam = scenes.make_cameras(cfg)[args.view]
    oracle.build()
    cores = oracle.get_threads()
    # warm-up (one frame at most), then full frames until K are done or ~90 s pass
    for _ in range(min(args.warmup, 1)):
        oracle.render(scene, cam)
    t0 = time.perf_counter()
    done = 0
    budget = 90.0
    while done < args.steps:
        oracle.render(scene, cam)
        done += 1
        if time.perf_counter() - t0 > budget:
            break
    dt = time.perf_counter() - t0
    fps = done / dt
    line = {"impl": "reference", "metric": metric_name(cfg),
            "value": fps, "unit": "frames/s", "n_gpus": args.gpus, "steps": done, "warmup": min(args.warmup, 1),
            "ms_per_step": 1e3 * dt / done, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.description, "n": cfg.n, "width": cfg.width, "height": cfg.height,
                       "sh_degree": cfg.sh_degree, "view": args.view},
            "cpu_baseline": {"value": fps, "unit": "frames/s", "cores": cores, "kind": "oracle",
                             "sample": f"{done} full frame(s) of the {args.steps} requested steps "
                                       f"(capped at ~{budget:.0f} s), all stages, fp64 oracle"},
            "e2e": {"value": fps, "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm

def fp32_peak_probe(torch, L, native, stream, dev):
    """The measured FMA rate of this GPU: gs_fp32_peak_probe (16 independent FMA chains per
    thread, 8 blocks of 256 threads per SM), scalar and packed, best of 5 timed launches each."""
    import ctypes
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks = sms * 8
    sink = torch.zeros(blocks * 256, device=dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    iters = 1 << 16
    out = {"sms": sms, "blocks": blocks, "threads": 256, "chains": 16, "iterations": iters}
    for packed in (0, 1):
        n = ctypes.c_int64(0)

        def launch():
            native.check(L.gs_fp32_peak_probe(blocks, iters, packed, sink.data_ptr(), ctypes.byref(n), sp),
                         "gs_fp32_peak_probe")
        best = None
        with torch.cuda.stream(stream):
            for _ in range(3):
                launch()
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                launch()
                b.record(stream)
                b.synchronize()
                ms = a.elapsed_time(b)
                best = ms if best is None else min(best, ms)
        out["packed_f32x2" if packed else "scalar"] = {"ms": best, "fmas": n.value,
                                                      "fma_per_s": n.value / (best * 1e-3)}
    fma = max(out["scalar"]["fma_per_s"], out["packed_f32x2"]["fma_per_s"])
    out["fma_per_s"] = fma
    out["TFLOP/s"] = 2 * fma / 1e12          # an FMA is 2 flops
    out["T_lane_ops/s"] = fma / 1e12         # one FMA per lane and cycle
    del sink
    return out


def param_bytes(sh_degree: int) -> int:
    return 4 * (3 + 4 + 3 + 1 + 3 * (sh_degree + 1) ** 2)


def evaluation_count(torch, gs, g, cam, final_T, n_contrib, dev) -> int:
    """The rasterizer's algorithmic count: over pixels, the list entries walked before T < 1e-4
    (all of the tile's list, or n_contrib for a pixel that stopped). The per-tile list lengths
    are recounted from the per-Gaussian tile rectangles (the sorted order is the oracle-checked
    one) with a 2D difference array."""
    tx, ty = gs.tiles_xy(cam)
    p_dev = gs.preprocess(g, cam)
    rect = p_dev["rect"].to(torch.int64) & 0xFFFF
    tt = p_dev["tiles_touched"].to(torch.int64)
    has = torch.nonzero(tt > 0).flatten()
    diff = torch.zeros((ty + 1, tx + 1), dtype=torch.int64, device=dev)
    rr = rect[has]
    ones = torch.ones(rr.shape[0], dtype=torch.int64, device=dev)
    diff.index_put_((rr[:, 1], rr[:, 0]), ones, accumulate=True)
    diff.index_put_((rr[:, 1], rr[:, 2] + 1), -ones, accumulate=True)
    diff.index_put_((rr[:, 3] + 1, rr[:, 0]), -ones, accumulate=True)
    diff.index_put_((rr[:, 3] + 1, rr[:, 2] + 1), ones, accumulate=True)
    cover = diff.cumsum(0).cumsum(1)[:ty, :tx]
    lens = cover.cpu().numpy()
    L_pix = np.kron(lens, np.ones((16, 16), np.int64))[: cam["height"], : cam["width"]]
    nc = n_contrib.cpu().numpy().astype(np.int64)
    Tf = final_T.cpu().numpy()
    del p_dev
    return int(np.where(Tf < 1e-4, nc, L_pix).sum())


STAGE_NAMES = ["preprocess", "depth_order", "bin", "tile_sort", "ranges", "rasterize"]
# the event order of a tile-first frame: the depth sort runs per tile, after the ranges
STAGE_NAMES_TILE_FIRST = ["preprocess", "bin", "tile_sort", "ranges", "depth_order", "rasterize"]


def measure_view(torch, gs, native, g, cam, r, stream, dev, steps, warmup, use_graph, world=1):
    """One view: K graph-replayed frames of gs_render (the frame time), K more through
    gs_render_profiled (per-stage CUDA-event times of the very launches a frame makes), and one
    frame with the per-pixel outputs (the rasterizer's evaluation count)."""
    import ctypes

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            r.render(cam, stream=stream, aux=False)
        stream.synchronize()
        st, flags, k = r.status(stream)
        if st != native.GS_OK:
            raise RuntimeError(f"render status {st} flags {flags} keys {k}")
        graph = None
        if use_graph:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                r.render(cam, stream=stream, aux=False)
            for _ in range(3):
                graph.replay()
            stream.synchronize()
    # --- the timed region: K whole frames, a barrier and a device synchronisation on both sides
    barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(40e6))
        e0.record(stream)
        for _ in range(steps):
            if graph is not None:
                graph.replay()
            else:
                r.render(cam, stream=stream, aux=False)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    frame_ms = e0.elapsed_time(e1) / steps
    del graph

    # --- per-stage times
    L = gs.lib()
    cs = gs.camera_struct(cam)
    sp = ctypes.c_void_p(stream.cuda_stream)
    n_stage = max(3, min(steps, 20))

    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(STAGE_NAMES) + 1)]
        for ev in evs:
            ev.record(stream)   # creates the underlying CUDA event
        arr = (ctypes.c_void_p * len(evs))(*[ctypes.c_void_p(ev.cuda_event) for ev in evs])
        return evs, arr

    def profiled(arr):
        native.check(L.gs_render_profiled(ctypes.byref(r._gs), ctypes.byref(cs), r.key_capacity,
                                          r.ws.data_ptr(), r.ws_bytes, r.image.data_ptr(), None, None, sp,
                                          arr, len(arr)), "gs_render_profiled")

    tile_first = bool(L.gs_render_tile_first(int(g["n"]), int(cam["width"]), int(cam["height"]), r.key_capacity))
    names = STAGE_NAMES_TILE_FIRST if tile_first else STAGE_NAMES
    st_ms = {k: 0.0 for k in STAGE_NAMES}
    with torch.cuda.stream(stream):
        pool = [new_events() for _ in range(n_stage)]
        for evs, arr in pool[:3]:
            profiled(arr)
        stream.synchronize()
        # a fixed-length device sleep first, so the host queues frames ahead of the GPU
        # and no stage time includes host launch latency
        torch.cuda._sleep(int(40e6))
        for evs, arr in pool:
            profiled(arr)
    torch.cuda.synchronize(dev)
    for evs, _ in pool:
        for i, k in enumerate(names):
            st_ms[k] += evs[i].elapsed_time(evs[i + 1]) / n_stage
    # --- one frame with the per-pixel outputs, for the evaluation count
    with torch.cuda.stream(stream):
        r.render(cam, stream=stream, aux=True)
    torch.cuda.synchronize(dev)
    st, flags, K = r.status(stream)
    if st != native.GS_OK:
        raise RuntimeError(f"render status {st} flags {flags} keys {K}")
    evals = evaluation_count(torch, gs, g, cam, r.final_T, r.n_contrib, dev)
    return {"frame_ms": frame_ms, "stage_ms": st_ms, "stage_steps": n_stage, "keys": int(K),
            "evaluations": evals, "graph": use_graph, "tile_first": tile_first}


def stage_summary(st_ms, n, sh_degree, K, tiles_x, tiles_y, evals, hbm_peak, fp32, tile_first=False, side=False):
    """Per-stage achieved rates and roofline fractions. HBM-bound stages: algorithmic bytes per
    unit (preprocess also in the method's count: parameters read + the 48-byte projected record
    written). Rasterize: evaluations x 15 flops (the method's count) against the measured FMA
    rate x 2, and evaluations x 9 FP32 lane operations (the kernel's count) against the measured
    FMA rate."""
    tile_bits = max(1, (tiles_x * tiles_y - 1).bit_length())
    tpasses = (tile_bits + 7) // 8
    pb = param_bytes(sh_degree)
    stage_bytes = {
        # (depth-first: + the depth keys and indices)
        "preprocess": (pb + PROJ_BYTES_PER_G + (0 if tile_first else 8)) * n,
        # depth-first: the keys and indices written, 4 passes of 16 B; tile-first: each list entry
        # read, its depth gathered and the entry written back (12 B)
        "depth_order": 12 * K if tile_first else 4 * 16 * n,
        "bin": 24 * n + 8 * K,
        "tile_sort": tpasses * 16 * K,
        "ranges": 4 * K + 8 * tiles_x * tiles_y + 12 * tiles_x * tiles_y,   # + the launch order
    }
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9 if ms > 0 else 0.0
    out = {}
    for k, b in stage_bytes.items():
        out[k] = {"ms": st_ms[k], "bound": "hbm", "GB/s": gbs(b, st_ms[k]), "frac": gbs(b, st_ms[k]) / hbm_peak,
                  "bytes": b}
    if side:
        # the ranges and the launch order ran on the second stream during the sorts; the stage
        # times the frame's wait for them, so it has no rate of its own
        out["ranges"] = {"ms": st_ms["ranges"], "bound": "overlapped", "frac": None, "bytes": stage_bytes["ranges"],
                         "note": "computed from the tile rectangles on a second stream; the stage is the join"}
    mb = (pb + PROJ_BYTES_METHOD) * n
    out["preprocess"].update({"bytes_method": mb, "GB/s_method": gbs(mb, st_ms["preprocess"]),
                              "frac_method": gbs(mb, st_ms["preprocess"]) / hbm_peak})
    ras_ms = st_ms["rasterize"]
    flops = FLOPS_PER_EVAL * evals
    lane_ops = OPS_PER_EVAL * evals
    tf = flops / (ras_ms * 1e-3) / 1e12 if ras_ms > 0 else 0.0
    lo = lane_ops / (ras_ms * 1e-3) / 1e12 if ras_ms > 0 else 0.0
    out["rasterize"] = {"ms": ras_ms, "bound": "alu", "evaluations": evals,
                        "flops": flops, "TFLOP/s": tf, "frac": tf / fp32["TFLOP/s"],
                        "lane_ops": lane_ops, "T_lane_ops/s": lo, "frac_lane_ops": lo / fp32["T_lane_ops/s"]}
    return out


def run_ours(args, rank, local_rank, world):
    import torch
    import gaussian_splatting_tile_02_b300 as gs
    from gaussian_splatting_tile_02_b300 import native, scenes

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = scenes.CONFIGS[args.config]
    scene = scenes.make_scene(cfg)
    cams = scenes.make_cameras(cfg)
    cam = cams[rank_view(args.view, rank, len(cams))]
    g = gs.gaussians_to_device(scene, dev)
    r = gs.Renderer.for_scene(g, cam, headroom=1.1)
    stream = torch.cuda.Stream(device=dev)
    L = gs.lib()
    sp = None

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    hbm_peak, peak_kind, peaks = measured_peaks()
    sampler = ClockSampler(local_rank, args.clocks_csv.format(rank=rank) if args.clocks_csv else None)
    with sampler:
        time.sleep(0.3)
        # --- the FP32 rate the compositing kernel is measured against
        fp32 = fp32_peak_probe(torch, L, native, stream, dev)
        # --- the headline workload (timed region inside, max over ranks)
        head = measure_view(torch, gs, native, g, cam, r, stream, dev, args.steps, args.warmup,
                            not args.no_graph, world)
        frame_ms_max = max_over_ranks(head["frame_ms"], world, dev)
        st_ms = head["stage_ms"]
        stage_total = sum(st_ms.values())
        import ctypes
        sp = ctypes.c_void_p(stream.cuda_stream)
        tx, ty = gs.tiles_xy(cam)

        # --- end to end from host memory
        e2e = None
        if not args.no_e2e:
            host = {k: torch.from_numpy(np.ascontiguousarray(scene[k])).pin_memory()
                    for k in ("means", "quats", "log_scales", "opacity_logits", "sh")}
            dst = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
            dst.update(n=g["n"], sh_degree=g["sh_degree"])
            r2 = gs.Renderer(dst, cam["width"], cam["height"], r.key_capacity)
            himg = torch.empty((cam["height"], cam["width"], 3), dtype=torch.float32).pin_memory()
            n_e2e = max(3, min(args.steps, 50))
            # one call after another (upload, render, read-back in sequence)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    gs.render_from_host(host, r2, cam, himg, stream=stream)
                stream.synchronize()
                barrier()
                t0 = time.perf_counter()
                for _ in range(n_e2e):
                    gs.render_from_host(host, r2, cam, himg, stream=stream)
                stream.synchronize()
                t_seq = max_over_ranks(time.perf_counter() - t0, world, dev)
                barrier()
            # the pipelined call: frame k + 1's upload overlaps frame k's render and read-back
            pipe = gs.HostPipeline(r2)
            for _ in range(3):
                pipe.submit(host, cam, himg)
            pipe.synchronize()
            barrier()
            t0 = time.perf_counter()
            for _ in range(n_e2e):
                pipe.submit(host, cam, himg)
            pipe.synchronize()
            t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
            barrier()
            h2d = sum(v.numel() * v.element_size() for v in host.values())
            d2h = himg.numel() * himg.element_size()
            e2e = {"value": world * n_e2e / t_e2e, "unit": "frames/s", "h2d_bytes_per_step": int(h2d),
                   "d2h_bytes_per_step": int(d2h), "steps": n_e2e, "call": "gs_render_from_host_async",
                   "sequential_value": world * n_e2e / t_seq, "sequential_call": "gs_render_from_host",
                   "h2d_GB_per_s": h2d * n_e2e / t_e2e / 1e9}
            del dst, r2, pipe
        # --- backward of the same frame: gs_render_backward replayed on the
        # forward's workspace (one forward with final T / n_contrib first)
        bwd = None
        if not args.no_backward:
            gen = torch.Generator(device=dev)
            gen.manual_seed(1234)
            gimg = torch.randn((cam["height"], cam["width"], 3), device=dev, generator=gen)
            grads = gs.alloc_param_grads(g)
            nb = max(3, min(args.steps, 50))
            with torch.cuda.stream(stream):
                r.render(cam, stream=stream, aux=True)
                for _ in range(3):
                    r.render_backward(cam, gimg, grads, stream=stream)
                stream.synchronize()
                b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda._sleep(int(40e6))
                b0.record(stream)
                for _ in range(nb):
                    r.render_backward(cam, gimg, grads, stream=stream)
                b1.record(stream)
                # step 1 backward alone (the same launch gs_render_backward makes)
                p_b = gs.preprocess(g, cam, stream=stream)
                n_g = int(g["n"])
                pg = {"mean2d": torch.zeros((n_g, 2), device=dev), "conic": torch.zeros((n_g, 3), device=dev),
                      "opacity": torch.zeros(n_g, device=dev), "rgb": torch.zeros((n_g, 3), device=dev)}
                for _ in range(3):
                    gs.preprocess_backward(g, cam, p_b, pg, stream=stream)
                b2, b3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda._sleep(int(40e6))
                b2.record(stream)
                for _ in range(nb):
                    gs.preprocess_backward(g, cam, p_b, pg, stream=stream)
                b3.record(stream)
            torch.cuda.synchronize(dev)
            bwd = {"ms": b0.elapsed_time(b1) / nb, "preprocess_backward_ms": b2.elapsed_time(b3) / nb,
                   "steps": nb, "n_contrib_sum": int(r.n_contrib.to(torch.int64).sum().item())}
            del grads, pg, p_b
        # --- several views per call: gs_render_batch against the same views
        # rendered one gs_render after another
        batch = None
        if not args.no_batch:
            bcams = cams if len(cams) > 1 else [scenes.orbit_camera(th, cfg.cam_distance, cfg.focal, cfg.width,
                                                                    cfg.height, cfg.near, cfg.bg)
                                                for th in (0.0, 90.0, 180.0, 270.0)]
            br = gs.BatchRenderer.for_scene(g, bcams, headroom=1.1, n_streams=args.batch_streams)
            single = gs.Renderer(g, cfg.width, cfg.height, br.key_capacity)
            nbt = max(3, min(args.steps // len(bcams), 20))
            with torch.cuda.stream(stream):
                for _ in range(2):
                    br.render(stream=stream)
                    for c in bcams:
                        single.render(c, stream=stream, aux=False)
                stream.synchronize()
                c0, c1, c2, c3 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
                torch.cuda._sleep(int(40e6))
                c0.record(stream)
                for _ in range(nbt):
                    for c in bcams:
                        single.render(c, stream=stream, aux=False)
                c1.record(stream)
                torch.cuda._sleep(int(40e6))
                c2.record(stream)
                for _ in range(nbt):
                    br.render(stream=stream)
                c3.record(stream)
            torch.cuda.synchronize(dev)
            for v in range(len(bcams)):
                if br.status(v)[0] != native.GS_OK:
                    raise RuntimeError(f"batch view {v} status {br.status(v)}")
            seq_ms, bat_ms = c0.elapsed_time(c1) / nbt, c2.elapsed_time(c3) / nbt
            batch = {"views": len(bcams), "streams": args.batch_streams, "steps": nbt,
                     "ms_per_batch": bat_ms, "views_per_s": len(bcams) * 1e3 / bat_ms,
                     "sequential_ms": seq_ms, "sequential_views_per_s": len(bcams) * 1e3 / seq_ms,
                     "speedup": seq_ms / bat_ms}
            del br, single
        # --- densification step on this scene (synthetic statistics): one
        # stable compaction pass over the parameters
        dens = None
        if not args.no_densify:
            n_g = int(g["n"])
            gen = torch.Generator(device=dev)
            gen.manual_seed(7)
            acc = torch.rand(n_g, device=dev, generator=gen) * 4e-4
            cnt = torch.ones(n_g, dtype=torch.int32, device=dev)
            xi = torch.randn((n_g, 2, 3), device=dev, generator=gen)
            with torch.cuda.stream(stream):
                n_new = gs.densify(g, acc, cnt, xi, 2e-4, 0.01, 0.005, stream=stream)["n"]
                # the C call alone, into preallocated arrays (no host reads)
                k3 = (cfg.sh_degree + 1) ** 2
                ob = {"means": torch.empty((2 * n_g, 3), device=dev), "quats": torch.empty((2 * n_g, 4), device=dev),
                      "log_scales": torch.empty((2 * n_g, 3), device=dev),
                      "opacity_logits": torch.empty(2 * n_g, device=dev),
                      "sh": torch.empty((2 * n_g, k3, 3), device=dev)}
                o = native.GsGaussiansOut()
                for k, v in ob.items():
                    setattr(o, k, v.data_ptr())
                o.n, o.sh_degree = 2 * n_g, cfg.sh_degree
                new_n = torch.zeros(1, dtype=torch.int64, device=dev)
                dwsb = int(L.gs_densify_workspace_bytes(n_g))
                dws = torch.empty(dwsb, dtype=torch.uint8, device=dev)
                gstruct = gs.gaussians_struct(g)

                def densify_call():
                    native.check(L.gs_densify(ctypes.byref(gstruct), acc.data_ptr(), cnt.data_ptr(), xi.data_ptr(),
                                              2e-4, 0.01, 0.005, ctypes.byref(o), new_n.data_ptr(), None,
                                              dws.data_ptr(), dwsb, sp), "gs_densify")
                for _ in range(3):
                    densify_call()
                d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                nd = 10
                stream.synchronize()
                torch.cuda._sleep(int(40e6))
                d0.record(stream)
                for _ in range(nd):
                    densify_call()
                d1.record(stream)
            torch.cuda.synchronize(dev)
            assert int(new_n.item()) == n_new
            dens = {"ms": d0.elapsed_time(d1) / nd, "n_in": n_g, "n_out": n_new}
            del acc, cnt, xi, ob, dws
        # --- the pages' 2D toy fit on the tile kernels (64 splats, 64x64, 200 Adam steps)
        toy = None
        if not args.no_toy:
            from gaussian_splatting_tile_02_b300 import splat2d
            splat2d.fit(steps=5)
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fit = splat2d.fit(steps=200)
            torch.cuda.synchronize(dev)
            toy = {"steps": 200, "seconds": time.perf_counter() - t0, "mse_first": fit["losses"][0],
                   "mse_final": fit["final_mse"]}
            toy["steps_per_s"] = 200 / toy["seconds"]
        # --- every workload of the benchmark, each view (one GPU only)
        configs = None
        if world == 1 and not args.no_configs:
            configs = {}
            names = [c for c in args.configs.split(",") if c]
            for name in names:
                if name == args.config and len(cams) == 1:
                    cfg_n, views = cfg, [(0, cam, head)]
                    g_n = g
                else:
                    cfg_n = scenes.CONFIGS[name]
                    sc = scenes.make_scene(cfg_n)
                    cams_n = scenes.make_cameras(cfg_n)
                    g_n = gs.gaussians_to_device(sc, dev)
                    del sc
                    r_n = gs.Renderer.for_scene(g_n, cams_n, headroom=1.1)
                    views = []
                    for v, c in enumerate(cams_n):
                        views.append((v, c, measure_view(torch, gs, native, g_n, c, r_n, stream, dev, args.steps,
                                                         args.warmup, not args.no_graph)))
                    del r_n
                recs = []
                for v, c, m in views:
                    ctx, cty = gs.tiles_xy(c)
                    recs.append({"view": v, "frame_ms": m["frame_ms"], "fps": 1e3 / m["frame_ms"], "keys": m["keys"],
                                 "tile_first": m["tile_first"],
                                 "stages": stage_summary(m["stage_ms"], cfg_n.n, cfg_n.sh_degree, m["keys"], ctx, cty,
                                                         m["evaluations"], hbm_peak, fp32, m["tile_first"],
                                                         side_ranges(cfg_n.n, ctx, cty))})
                mean_ms = statistics.mean(x["frame_ms"] for x in recs)
                mean_st = {}
                for k in recs[0]["stages"]:
                    mean_st[k] = {kk: statistics.mean(x["stages"][k][kk] for x in recs)
                                  for kk in recs[0]["stages"][k] if isinstance(recs[0]["stages"][k][kk], (int, float))}
                configs[name] = {"workload": cfg_n.description, "n": cfg_n.n, "width": cfg_n.width,
                                 "height": cfg_n.height, "sh_degree": cfg_n.sh_degree, "steps": args.steps,
                                 "views": recs,
                                 "mean": {"frame_ms": mean_ms, "fps": 1e3 / mean_ms, "stages": mean_st}}
                if g_n is not g:
                    del g_n
                torch.cuda.empty_cache()
    clocks = sampler.summary()

    n = int(g["n"])
    K = head["keys"]
    stages_out = stage_summary(st_ms, n, cfg.sh_degree, K, tx, ty, head["evaluations"], hbm_peak, fp32,
                               head["tile_first"], side_ranges(n, tx, ty))
    launches_per_frame = frame_launches(tx * ty, head["tile_first"], r.key_capacity, (tx, ty), int(g["n"]))
    ras = stages_out["rasterize"]
    evals = head["evaluations"]
    dominant = max(stages_out, key=lambda k: stages_out[k]["ms"])
    if dominant == "rasterize":
        roof = {"kernel": "rasterize_kernel", "bound": "alu", "achieved": ras["TFLOP/s"], "peak": fp32["TFLOP/s"],
                "unit": "TFLOP/s", "frac": ras["frac"],
                "peak_kind": "measured: FFMA probe (gs_fp32_peak_probe), 2 flops per FMA, of measured",
                "traffic": traffic_from_profile("rasterize_1M.md", args.config),
                "units": f"{evals} pixel-Gaussian evaluations x {FLOPS_PER_EVAL} flops",
                "lane_ops": {"achieved": ras["T_lane_ops/s"], "peak": fp32["T_lane_ops/s"], "frac": ras["frac_lane_ops"],
                             "unit": "T FP32 lane-ops/s",
                             "units": f"{evals} evaluations x {OPS_PER_EVAL} FP32 lane operations"}}
    else:
        d = stages_out[dominant]
        roof = {"kernel": dominant, "bound": "hbm", "achieved": d["GB/s"], "peak": hbm_peak, "unit": "GB/s",
                "frac": d["frac"], "peak_kind": peak_kind, "traffic": None}

    result = {
        "metric": metric_name(cfg),
        "value": job_value(frame_ms_max, world), "unit": "frames/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": frame_ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": cfg.description, "n": cfg.n, "width": cfg.width, "height": cfg.height,
                   "sh_degree": cfg.sh_degree, "view": args.view, "keys": K, "key_capacity": r.key_capacity,
                   "graph": not args.no_graph,
                   "steps_order": "tile-first" if head["tile_first"] else "depth-first",
                   "l2": "inputs larger than L2: 236 MB of Gaussian parameters per frame (L2 126 MB)",
                   "parallelism": f"replicas x{world}"},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches_per_frame * args.steps,
        "roofline": roof,
        "stages": stages_out,
        "stage_sum_ms": stage_total,
        "hbm_peak_gbs": hbm_peak,
        "fp32_peak_measured": fp32,
        "backward": backward_summary(bwd, int(g["n"]), hbm_peak, fp32["T_lane_ops/s"]),
        "batch": batch,
        "densify": densify_summary(dens, cfg.sh_degree, hbm_peak),
        "toy2d": toy,
        "configs": configs,
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cores = oracle.get_threads()
        t0 = time.perf_counter()
        frames = 0
        while frames < 5:
            oracle.render(scene, cam)
            frames += 1
            if time.perf_counter() - t0 > args.cpu_seconds:
                break
        dt = time.perf_counter() - t0
        result["cpu_baseline"] = {"value": frames / dt, "unit": "frames/s", "cores": cores, "kind": "oracle",
                                  "sample": f"{frames} full frame(s) of this workload, all stages, fp64"}
        if not args.no_single_thread:
            # the same oracle on one thread, one full frame
            oracle.set_threads(1)
            t0 = time.perf_counter()
            oracle.render(scene, cam)
            dt1 = time.perf_counter() - t0
            oracle.set_threads(cores)
            result["cpu_baseline"]["single_thread"] = {
                "value": 1.0 / dt1, "unit": "frames/s", "cores": 1,
                "sample": "1 full frame of this workload, all stages, fp64, one thread"}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    main()
