"""B300 forward renderer for 3D Gaussian Splatting.

Python front end of the C-ABI library ``libgs_b300.so`` (include/gs.h). The
five steps of the lesson page "3D Gaussian Splatting à partir de zéro"
(section "Rastérisation, non rayée": project to 2D, assign to 16x16 tiles,
depth-sort per tile, alpha-composite front to back, pixel colour) each run as
hand-written sm_103a CUDA kernels; this module only allocates device memory
with PyTorch, passes pointers and the current stream, and checks status codes.

    from gaussian_splatting_tile_02_b300 import Renderer, scenes
    scene = scenes.make_scene("1M"); cam = scenes.make_cameras("1M")[0]
    r = Renderer.for_scene(scene, cam)          # device copy + workspace
    image = r.render(cam)                      # [H, W, 3] float32 on cuda

Stage-wise calls (preprocess, bin_keys, sort_pairs, tile_ranges, rasterize)
expose each step for testing and composition.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import native
from .native import GsCamera, GsGaussians, GsGaussiansGrad, GsProjected, GsProjectedGrad, check, lib

__all__ = ["GsCamera", "camera_struct", "gaussians_to_device", "gaussians_struct", "preprocess",
           "bin_keys", "sort_pairs", "tile_ranges", "rasterize", "Renderer", "read_status",
           "key_bits", "tiles_xy", "lib", "render_from_host", "rasterize_backward", "preprocess_backward",
           "alloc_param_grads", "BatchRenderer", "densify_stats", "densify", "HostPipeline"]


def _torch():
    import torch
    return torch


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def tiles_xy(cam: dict) -> tuple:
    return (int(cam["width"]) + 15) // 16, (int(cam["height"]) + 15) // 16


def key_bits(cam: dict) -> int:
    tx, ty = tiles_xy(cam)
    return 32 + max(0, (tx * ty - 1).bit_length())


def camera_struct(cam: dict) -> GsCamera:
    c = GsCamera()
    R = np.asarray(cam["R"], np.float32).reshape(9)
    t = np.asarray(cam["t"], np.float32).reshape(3)
    bg = np.asarray(cam.get("bg", (0.0, 0.0, 0.0)), np.float32).reshape(3)
    for i in range(9):
        c.R[i] = float(R[i])
    for i in range(3):
        c.t[i] = float(t[i])
        c.bg[i] = float(bg[i])
    c.fx, c.fy, c.cx, c.cy = (float(np.float32(cam[k])) for k in ("fx", "fy", "cx", "cy"))
    c.near_z = float(np.float32(cam["near"]))
    c.width, c.height = int(cam["width"]), int(cam["height"])
    return c


_FIELDS = ("means", "quats", "log_scales", "opacity_logits", "sh")


def gaussians_to_device(scene: dict, device="cuda") -> dict:
    torch = _torch()
    out = {k: torch.from_numpy(np.ascontiguousarray(scene[k], np.float32)).to(device) for k in _FIELDS}
    out["sh_degree"] = int(scene["sh_degree"])
    out["n"] = int(scene["means"].shape[0])
    return out


def gaussians_struct(g: dict) -> GsGaussians:
    s = GsGaussians()
    for k in _FIELDS:
        setattr(s, k, _ptr(g[k]))
    s.n = int(g["n"])
    s.sh_degree = int(g["sh_degree"])
    return s


def alloc_projected(n: int, device="cuda") -> dict:
    torch = _torch()
    return {"mean2d": torch.empty((n, 2), dtype=torch.float32, device=device),
            "conic_opacity": torch.empty((n, 4), dtype=torch.float32, device=device),
            "rgb": torch.empty((n, 3), dtype=torch.float32, device=device),
            "depth": torch.empty(n, dtype=torch.float32, device=device),
            "radius": torch.empty(n, dtype=torch.int32, device=device),
            "tiles_touched": torch.empty(n, dtype=torch.int32, device=device),
            "rect": torch.empty((n, 4), dtype=torch.int16, device=device),
            "raster": torch.empty((n, 12), dtype=torch.float32, device=device)}


def projected_struct(p: dict) -> GsProjected:
    s = GsProjected()
    for k in ("mean2d", "conic_opacity", "rgb", "depth", "radius", "tiles_touched", "rect", "raster"):
        setattr(s, k, _ptr(p.get(k)))
    return s


# ------------------------------------------------------------------------------ stages

def preprocess(g: dict, cam: dict, stream=None) -> dict:
    """Step 1: projection. Returns the projected record (device tensors)."""
    p = alloc_projected(int(g["n"]), g["means"].device)
    check(lib().gs_preprocess(ctypes.byref(gaussians_struct(g)), ctypes.byref(camera_struct(cam)),
                              ctypes.byref(projected_struct(p)), _stream_ptr(stream)), "gs_preprocess")
    return p


def bin_keys(p: dict, cam: dict, key_capacity: int, stream=None) -> dict:
    """Step 2: scan + duplication into 64-bit tile|depth keys (device tensors)."""
    torch = _torch()
    n = int(p["depth"].shape[0])
    dev = p["depth"].device
    cap = int(key_capacity)
    out = {"offsets": torch.empty(n, dtype=torch.int32, device=dev),
           "keys": torch.empty(max(cap, 1), dtype=torch.int64, device=dev),
           "vals": torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
           "num_keys": torch.zeros(1, dtype=torch.int64, device=dev)}
    wsb = int(lib().gs_bin_workspace_bytes(n))
    out["ws"] = torch.empty(wsb, dtype=torch.uint8, device=dev)
    check(lib().gs_bin(ctypes.byref(projected_struct(p)), n, ctypes.byref(camera_struct(cam)),
                       _ptr(out["offsets"]), _ptr(out["keys"]), _ptr(out["vals"]), cap,
                       _ptr(out["num_keys"]), _ptr(out["ws"]), wsb, _stream_ptr(stream)), "gs_bin")
    return out


def sort_pairs(keys, vals, num_keys, key_bits_: int, key_capacity: int | None = None, stream=None,
               ws=None) -> dict:
    """Step 3: stable radix sort in place (keys/vals end sorted). Returns scratch for status reads."""
    torch = _torch()
    cap = int(keys.shape[0] if key_capacity is None else key_capacity)
    dev = keys.device
    keys_alt = torch.empty_like(keys)
    vals_alt = torch.empty_like(vals)
    wsb = int(lib().gs_sort_workspace_bytes(cap))
    if ws is None:
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    check(lib().gs_sort(_ptr(keys), _ptr(vals), _ptr(keys_alt), _ptr(vals_alt), _ptr(num_keys), cap,
                        int(key_bits_), _ptr(ws), wsb, _stream_ptr(stream)), "gs_sort")
    return {"keys": keys, "vals": vals, "ws": ws, "keys_alt": keys_alt, "vals_alt": vals_alt}


def tile_ranges(sorted_keys, num_keys, cam: dict, key_capacity: int | None = None, stream=None):
    """Step 4: [start, end) of every tile in the sorted keys, [tiles, 2] int32 (uint32 values)."""
    torch = _torch()
    tx, ty = tiles_xy(cam)
    ranges = torch.empty((tx * ty, 2), dtype=torch.int32, device=sorted_keys.device)
    cap = int(sorted_keys.shape[0] if key_capacity is None else key_capacity)
    check(lib().gs_tile_ranges(_ptr(sorted_keys), _ptr(num_keys), cap, ctypes.byref(camera_struct(cam)),
                               _ptr(ranges), _stream_ptr(stream)), "gs_tile_ranges")
    return ranges


def rasterize(p: dict, sorted_vals, ranges, cam: dict, stream=None, want_aux: bool = True,
              heavy_first: bool = True) -> dict:
    """Step 5: composite. Returns image [H,W,3], final_T [H,W], n_contrib [H,W].

    heavy_first launches the tiles in decreasing list length (the image does not change)."""
    torch = _torch()
    H, W = int(cam["height"]), int(cam["width"])
    dev = ranges.device
    out = {"image": torch.empty((H, W, 3), dtype=torch.float32, device=dev)}
    if want_aux:
        out["final_T"] = torch.empty((H, W), dtype=torch.float32, device=dev)
        out["n_contrib"] = torch.empty((H, W), dtype=torch.int32, device=dev)
    tx, ty = tiles_xy(cam)
    order = torch.empty(tx * ty, dtype=torch.int32, device=dev) if heavy_first else None
    n = int(p["depth"].shape[0])
    check(lib().gs_rasterize(ctypes.byref(projected_struct(p)), n, _ptr(sorted_vals), _ptr(ranges),
                             ctypes.byref(camera_struct(cam)), _ptr(out["image"]), _ptr(out.get("final_T")),
                             _ptr(out.get("n_contrib")), _ptr(order), _stream_ptr(stream)), "gs_rasterize")
    return out


# ------------------------------------------------------------------------------ backward

def _pgrad_struct(d: dict) -> GsProjectedGrad:
    s = GsProjectedGrad()
    for k in ("mean2d", "conic", "opacity", "rgb"):
        setattr(s, k, _ptr(d[k]))
    return s


def alloc_param_grads(g: dict) -> dict:
    """Gradient arrays shaped like the Gaussian parameters (device, float32)."""
    torch = _torch()
    return {k: torch.empty_like(g[k]) for k in _FIELDS}


def _ggrad_struct(d: dict) -> GsGaussiansGrad:
    s = GsGaussiansGrad()
    for k in _FIELDS:
        setattr(s, k, _ptr(d[k]))
    return s


def rasterize_backward(p: dict, sorted_vals, ranges, cam: dict, final_T, n_contrib, grad_image,
                       tile_order=None, stream=None) -> dict:
    """Step 5 backward: dL/d(u, v), dL/d(conic A, B, C), dL/do, dL/dc per Gaussian."""
    torch = _torch()
    n = int(p["depth"].shape[0])
    dev = ranges.device
    out = {"mean2d": torch.empty((n, 2), dtype=torch.float32, device=dev),
           "conic": torch.empty((n, 3), dtype=torch.float32, device=dev),
           "opacity": torch.empty(n, dtype=torch.float32, device=dev),
           "rgb": torch.empty((n, 3), dtype=torch.float32, device=dev)}
    check(lib().gs_rasterize_backward(ctypes.byref(projected_struct(p)), n, _ptr(sorted_vals), _ptr(ranges),
                                      ctypes.byref(camera_struct(cam)), _ptr(final_T), _ptr(n_contrib),
                                      _ptr(grad_image), _ptr(tile_order), ctypes.byref(_pgrad_struct(out)),
                                      _stream_ptr(stream)), "gs_rasterize_backward")
    return out


def preprocess_backward(g: dict, cam: dict, p: dict, pgrad: dict, stream=None) -> dict:
    """Step 1 backward: parameter gradients from the projected ones."""
    out = alloc_param_grads(g)
    check(lib().gs_preprocess_backward(ctypes.byref(gaussians_struct(g)), ctypes.byref(camera_struct(cam)),
                                       ctypes.byref(projected_struct(p)), ctypes.byref(_pgrad_struct(pgrad)),
                                       ctypes.byref(_ggrad_struct(out)), _stream_ptr(stream)),
          "gs_preprocess_backward")
    return out


# ------------------------------------------------------------------------------ densify / prune

def densify_stats(grad_mean2d, tiles_touched, accum, count, stream=None) -> None:
    """accum += |dL/d(u, v)|, count += 1 for Gaussians that touched a tile."""
    n = int(accum.shape[0])
    check(lib().gs_densify_stats(_ptr(grad_mean2d), _ptr(tiles_touched), n, _ptr(accum), _ptr(count),
                                 _stream_ptr(stream)), "gs_densify_stats")


def densify(g: dict, accum, count, xi, grad_threshold: float = 2e-4, scale_threshold: float = 0.01,
            prune_opacity: float = 0.005, capacity: int | None = None, stream=None) -> dict:
    """Clone / split / prune (section "Densation et taille"). Returns the new
    device parameter dict (n = new count; synchronises to read it) and
    ``action`` (uint8 per input Gaussian: 0 keep, 1 clone, 2 split, 3 prune)."""
    torch = _torch()
    n = int(g["n"])
    dev = g["means"].device
    cap = 2 * n if capacity is None else int(capacity)
    k3 = (int(g["sh_degree"]) + 1) ** 2
    out = {"means": torch.empty((max(cap, 1), 3), dtype=torch.float32, device=dev),
           "quats": torch.empty((max(cap, 1), 4), dtype=torch.float32, device=dev),
           "log_scales": torch.empty((max(cap, 1), 3), dtype=torch.float32, device=dev),
           "opacity_logits": torch.empty(max(cap, 1), dtype=torch.float32, device=dev),
           "sh": torch.empty((max(cap, 1), k3, 3), dtype=torch.float32, device=dev)}
    o = native.GsGaussiansOut()
    for k in _FIELDS:
        setattr(o, k, _ptr(out[k]))
    o.n = cap
    o.sh_degree = int(g["sh_degree"])
    new_n = torch.zeros(1, dtype=torch.int64, device=dev)
    action = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
    wsb = int(lib().gs_densify_workspace_bytes(n))
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    check(lib().gs_densify(ctypes.byref(gaussians_struct(g)), _ptr(accum), _ptr(count), _ptr(xi),
                           float(grad_threshold), float(scale_threshold), float(prune_opacity), ctypes.byref(o),
                           _ptr(new_n), _ptr(action), _ptr(ws), wsb, _stream_ptr(stream)), "gs_densify")
    st, flags, _ = read_status(ws, stream)
    check(st, "gs_densify (capacity)")
    m = int(new_n.item())
    res = {k: v[:m] for k, v in out.items()}
    res.update(n=m, sh_degree=int(g["sh_degree"]), action=action[:n])
    return res


def read_status(ws, stream=None) -> tuple:
    """(status, flags, num_keys) from a workspace header; synchronises the stream."""
    flags = ctypes.c_uint32(0)
    nk = ctypes.c_uint64(0)
    st = lib().gs_read_status(_ptr(ws), _stream_ptr(stream), ctypes.byref(flags), ctypes.byref(nk))
    return int(st), int(flags.value), int(nk.value)


# ------------------------------------------------------------------------------ whole frame

def workspace_lists(ws, n: int, width: int, height: int, key_capacity: int, num_keys: int) -> tuple:
    """(sorted_vals [num_keys] int32, ranges [tiles, 2] int32): views into a gs_render workspace
    tensor (uint8) of the frame's per-tile lists, located by gs_render_workspace_lists."""
    vp, rp = ctypes.c_void_p(), ctypes.c_void_p()
    check(lib().gs_render_workspace_lists(_ptr(ws), int(n), int(width), int(height), int(key_capacity),
                                          ctypes.byref(vp), ctypes.byref(rp)), "gs_render_workspace_lists")
    base = ws.data_ptr()
    num_keys = min(int(num_keys), int(key_capacity))
    tx, ty = (int(width) + 15) // 16, (int(height) + 15) // 16
    vo, ro = vp.value - base, rp.value - base
    vals = ws[vo: vo + 4 * int(num_keys)].view(_torch().int32)
    ranges = ws[ro: ro + 8 * tx * ty].view(_torch().int32).view(tx * ty, 2)
    return vals, ranges


class Renderer:
    """Owns a device copy of a scene and a gs_render workspace sized for it."""

    def __init__(self, g: dict, width: int, height: int, key_capacity: int):
        torch = _torch()
        self.g = g
        self.width, self.height = int(width), int(height)
        self.key_capacity = int(key_capacity)
        self.ws_bytes = int(lib().gs_render_workspace_bytes(int(g["n"]), self.width, self.height,
                                                           self.key_capacity))
        dev = g["means"].device
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.image = torch.empty((self.height, self.width, 3), dtype=torch.float32, device=dev)
        self.final_T = torch.empty((self.height, self.width), dtype=torch.float32, device=dev)
        self.n_contrib = torch.empty((self.height, self.width), dtype=torch.int32, device=dev)
        self._gs = gaussians_struct(g)

    @staticmethod
    def count_keys(g: dict, cam: dict) -> int:
        """K for one view (runs preprocess + binning with zero capacity; synchronises)."""
        p = preprocess(g, cam)
        b = bin_keys(p, cam, 0)
        return int(b["num_keys"].item())

    @classmethod
    def for_scene(cls, scene: dict, cams, headroom: float = 1.25, device="cuda") -> "Renderer":
        g = gaussians_to_device(scene, device) if isinstance(scene["means"], np.ndarray) else scene
        cams = cams if isinstance(cams, (list, tuple)) else [cams]
        k = max(cls.count_keys(g, c) for c in cams)
        w = max(int(c["width"]) for c in cams)
        h = max(int(c["height"]) for c in cams)
        return cls(g, w, h, int(k * headroom) + 1024)

    def render(self, cam: dict, stream=None, aux: bool = True):
        """Renders one frame into self.image (no host synchronisation)."""
        assert int(cam["width"]) == self.width and int(cam["height"]) == self.height
        c = camera_struct(cam)
        check(lib().gs_render(ctypes.byref(self._gs), ctypes.byref(c), self.key_capacity, _ptr(self.ws),
                              self.ws_bytes, _ptr(self.image), _ptr(self.final_T) if aux else None,
                              _ptr(self.n_contrib) if aux else None, _stream_ptr(stream)), "gs_render")
        return self.image

    def status(self, stream=None) -> tuple:
        return read_status(self.ws, stream)

    def lists(self, stream=None) -> tuple:
        """(sorted_vals [K], ranges [tiles, 2]) of the last frame (synchronises the stream)."""
        K = self.status(stream)[2]
        return workspace_lists(self.ws, int(self.g["n"]), self.width, self.height, self.key_capacity, K)

    def render_backward(self, cam: dict, grad_image, grads: dict | None = None, stream=None) -> dict:
        """Parameter gradients of sum(grad_image * image) for the frame last
        rendered with render(cam, aux=True) (no host synchronisation)."""
        grads = alloc_param_grads(self.g) if grads is None else grads
        check(lib().gs_render_backward(ctypes.byref(self._gs), ctypes.byref(camera_struct(cam)), self.key_capacity,
                                       _ptr(self.ws), self.ws_bytes, _ptr(self.final_T), _ptr(self.n_contrib),
                                       _ptr(grad_image), ctypes.byref(_ggrad_struct(grads)), _stream_ptr(stream)),
              "gs_render_backward")
        return grads


class BatchRenderer:
    """Several views of one scene per call (gs_render_batch): one projection
    pass over the parameters for all views, then each view's steps 2-5 on one
    of ``n_streams`` streams so that the views overlap on the GPU."""

    def __init__(self, g: dict, cams: list, key_capacity: int, n_streams: int = 4):
        torch = _torch()
        self.g = g
        self.cams = list(cams)
        self.views = len(self.cams)
        self.width, self.height = int(self.cams[0]["width"]), int(self.cams[0]["height"])
        self.key_capacity = int(key_capacity)
        n = int(g["n"])
        self.ws_bytes = int(lib().gs_render_batch_workspace_bytes(n, self.width, self.height, self.key_capacity,
                                                                 self.views))
        if self.ws_bytes == 0:
            raise ValueError("unsupported batch")
        self.view_ws_bytes = int(lib().gs_render_workspace_bytes(n, self.width, self.height, self.key_capacity))
        dev = g["means"].device
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        V, H, W = self.views, self.height, self.width
        self.images = torch.empty((V, H, W, 3), dtype=torch.float32, device=dev)
        self.final_T = torch.empty((V, H, W), dtype=torch.float32, device=dev)
        self.n_contrib = torch.empty((V, H, W), dtype=torch.int32, device=dev)
        self.extra_streams = [torch.cuda.Stream(device=dev) for _ in range(max(0, n_streams - 1))]
        self._gs = gaussians_struct(g)
        self._cams = (GsCamera * V)(*[camera_struct(c) for c in self.cams])

    @classmethod
    def for_scene(cls, scene: dict, cams: list, headroom: float = 1.25, n_streams: int = 4,
                  device="cuda") -> "BatchRenderer":
        g = gaussians_to_device(scene, device) if isinstance(scene["means"], np.ndarray) else scene
        k = max(Renderer.count_keys(g, c) for c in cams)
        return cls(g, cams, int(k * headroom) + 1024, n_streams)

    def render(self, stream=None, aux: bool = False):
        """Renders every view into self.images [V, H, W, 3] (no host synchronisation)."""
        torch = _torch()
        s0 = stream if stream is not None else torch.cuda.current_stream()
        handles = [s0.cuda_stream] + [s.cuda_stream for s in self.extra_streams]
        arr = (ctypes.c_void_p * len(handles))(*handles)
        check(lib().gs_render_batch(ctypes.byref(self._gs), self._cams, self.views, self.key_capacity,
                                    _ptr(self.ws), self.ws_bytes, _ptr(self.images),
                                    _ptr(self.final_T) if aux else None, _ptr(self.n_contrib) if aux else None,
                                    arr, len(handles)), "gs_render_batch")
        return self.images

    def status(self, view: int, stream=None) -> tuple:
        """(status, flags, num_keys) of one view; synchronises the stream."""
        return read_status(self.ws[view * self.view_ws_bytes:], stream)

    def lists(self, view: int, stream=None) -> tuple:
        """(sorted_vals [K], ranges [tiles, 2]) of one view of the last batch (synchronises the stream)."""
        K = self.status(view, stream)[2]
        w = self.ws[view * self.view_ws_bytes: (view + 1) * self.view_ws_bytes]
        return workspace_lists(w, int(self.g["n"]), self.width, self.height, self.key_capacity, K)


class HostPipeline:
    """Frames from pinned host parameters with the copies overlapped
    (gs_render_from_host_async): two device parameter sets, and render,
    upload and read-back streams, so that frame k + 1's upload runs during
    frame k's render and image read-back."""

    def __init__(self, renderer: Renderer):
        torch = _torch()
        self.r = renderer
        g = renderer.g
        dev = g["means"].device
        self.sets = [{k: torch.empty_like(g[k]) for k in _FIELDS} for _ in range(2)]
        structs = []
        for d in self.sets:
            d.update(n=g["n"], sh_degree=g["sh_degree"])
            structs.append(gaussians_struct(d))
        self._sets = (GsGaussians * 2)(*structs)
        self.streams = [torch.cuda.Stream(device=dev) for _ in range(3)]
        self.events = [torch.cuda.Event() for _ in range(6)]
        for e in self.events:
            e.record(self.streams[0])   # creates the underlying CUDA events
        torch.cuda.synchronize(dev)
        self._streams = (ctypes.c_void_p * 3)(*[s.cuda_stream for s in self.streams])
        self._events = (ctypes.c_void_p * 6)(*[e.cuda_event for e in self.events])
        self.frame = 0

    def submit(self, host: dict, cam: dict, host_image) -> None:
        hs = GsGaussians()
        for k in _FIELDS:
            setattr(hs, k, host[k].data_ptr())
        hs.n = int(self.r.g["n"])
        hs.sh_degree = int(self.r.g["sh_degree"])
        check(lib().gs_render_from_host_async(ctypes.byref(hs), self._sets, self.frame,
                                              ctypes.byref(camera_struct(cam)), self.r.key_capacity,
                                              _ptr(self.r.ws), self.r.ws_bytes, _ptr(self.r.image),
                                              host_image.data_ptr(), self._streams, self._events),
              "gs_render_from_host_async")
        self.frame += 1

    def synchronize(self) -> None:
        for s in self.streams:
            s.synchronize()


def render_from_host(host: dict, renderer: Renderer, cam: dict, host_image, stream=None) -> None:
    """One frame from host (pinned) parameter arrays into a host image through gs_render_from_host."""
    hs = GsGaussians()
    for k in _FIELDS:
        setattr(hs, k, host[k].data_ptr())
    hs.n = int(renderer.g["n"])
    hs.sh_degree = int(renderer.g["sh_degree"])
    check(lib().gs_render_from_host(ctypes.byref(hs), ctypes.byref(renderer._gs),
                                    ctypes.byref(camera_struct(cam)), renderer.key_capacity,
                                    _ptr(renderer.ws), renderer.ws_bytes, _ptr(renderer.image),
                                    host_image.data_ptr(), _stream_ptr(stream)), "gs_render_from_host")
