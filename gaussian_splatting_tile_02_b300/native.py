"""ctypes binding of libgs_b300.so (the C ABI in include/gs.h).

Argument marshalling only: every step of the rendering path runs in the
library's CUDA kernels. Loading fails loudly if the library is missing and
cannot be built; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

c_void_p = ctypes.c_void_p


class GsCamera(ctypes.Structure):
    _fields_ = [("R", ctypes.c_float * 9), ("t", ctypes.c_float * 3),
                ("fx", ctypes.c_float), ("fy", ctypes.c_float), ("cx", ctypes.c_float),
                ("cy", ctypes.c_float), ("near_z", ctypes.c_float),
                ("width", ctypes.c_int32), ("height", ctypes.c_int32), ("bg", ctypes.c_float * 3)]


class GsGaussians(ctypes.Structure):
    _fields_ = [("means", c_void_p), ("quats", c_void_p), ("log_scales", c_void_p),
                ("opacity_logits", c_void_p), ("sh", c_void_p), ("n", ctypes.c_int64),
                ("sh_degree", ctypes.c_int32)]


class GsProjected(ctypes.Structure):
    _fields_ = [("mean2d", c_void_p), ("conic_opacity", c_void_p), ("rgb", c_void_p),
                ("depth", c_void_p), ("radius", c_void_p), ("tiles_touched", c_void_p),
                ("rect", c_void_p), ("raster", c_void_p)]


class GsProjectedGrad(ctypes.Structure):
    _fields_ = [("mean2d", c_void_p), ("conic", c_void_p), ("opacity", c_void_p), ("rgb", c_void_p)]


class GsGaussiansGrad(ctypes.Structure):
    _fields_ = [("means", c_void_p), ("quats", c_void_p), ("log_scales", c_void_p),
                ("opacity_logits", c_void_p), ("sh", c_void_p)]


class GsGaussiansOut(ctypes.Structure):
    _fields_ = [("means", c_void_p), ("quats", c_void_p), ("log_scales", c_void_p),
                ("opacity_logits", c_void_p), ("sh", c_void_p), ("n", ctypes.c_int64), ("sh_degree", ctypes.c_int32)]


GS_OK, GS_ERR_INVALID_ARG, GS_ERR_CAPACITY, GS_ERR_CUDA, GS_ERR_TIMEOUT, GS_ERR_WORKSPACE = range(6)
GS_FLAG_CAPACITY, GS_FLAG_TIMEOUT = 1, 2

# every function the header declares, with its ctypes signature
_SIGNATURES = {
    "gs_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "gs_abi_version": (ctypes.c_int32, []),
    "gs_preprocess": (ctypes.c_int, [ctypes.POINTER(GsGaussians), ctypes.POINTER(GsCamera),
                                     ctypes.POINTER(GsProjected), c_void_p]),
    "gs_bin_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64]),
    "gs_bin": (ctypes.c_int, [ctypes.POINTER(GsProjected), ctypes.c_int64, ctypes.POINTER(GsCamera),
                              c_void_p, c_void_p, c_void_p, ctypes.c_int64, c_void_p, c_void_p,
                              ctypes.c_size_t, c_void_p]),
    "gs_bin_static": (ctypes.c_int, [ctypes.POINTER(GsProjected), ctypes.c_int64, ctypes.POINTER(GsCamera),
                                     c_void_p, c_void_p, c_void_p, ctypes.c_int64, c_void_p, c_void_p]),
    "gs_sort_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64]),
    "gs_sort": (ctypes.c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, ctypes.c_int64,
                               ctypes.c_int32, c_void_p, ctypes.c_size_t, c_void_p]),
    "gs_tile_ranges": (ctypes.c_int, [c_void_p, c_void_p, ctypes.c_int64, ctypes.POINTER(GsCamera),
                                      c_void_p, c_void_p]),
    "gs_depth_order_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64]),
    "gs_bin_ordered_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "gs_depth_order": (ctypes.c_int, [ctypes.POINTER(GsProjected), ctypes.c_int64, c_void_p, c_void_p,
                                      ctypes.c_size_t, c_void_p]),
    "gs_bin_ordered": (ctypes.c_int, [ctypes.POINTER(GsProjected), ctypes.c_int64, c_void_p,
                                      ctypes.POINTER(GsCamera), c_void_p, c_void_p, c_void_p, ctypes.c_int64,
                                      c_void_p, c_void_p, ctypes.c_size_t, c_void_p]),
    "gs_sort32": (ctypes.c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, ctypes.c_int64,
                                 ctypes.c_int32, c_void_p, ctypes.c_size_t, c_void_p]),
    "gs_tile_ranges32": (ctypes.c_int, [c_void_p, c_void_p, ctypes.c_int64, ctypes.POINTER(GsCamera),
                                        c_void_p, c_void_p]),
    "gs_rasterize": (ctypes.c_int, [ctypes.POINTER(GsProjected), ctypes.c_int64, c_void_p, c_void_p,
                                    ctypes.POINTER(GsCamera), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "gs_render_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                    ctypes.c_int64]),
    "gs_render_tile_first": (ctypes.c_int32, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64]),
    "gs_render_workspace_lists": (ctypes.c_int, [c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int64, ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p)]),
    "gs_render": (ctypes.c_int, [ctypes.POINTER(GsGaussians), ctypes.POINTER(GsCamera), ctypes.c_int64,
                                 c_void_p, ctypes.c_size_t, c_void_p, c_void_p, c_void_p, c_void_p]),
    "gs_render_profiled": (ctypes.c_int, [ctypes.POINTER(GsGaussians), ctypes.POINTER(GsCamera), ctypes.c_int64,
                                          c_void_p, ctypes.c_size_t, c_void_p, c_void_p, c_void_p, c_void_p,
                                          ctypes.POINTER(c_void_p), ctypes.c_int32]),
    "gs_render_from_host": (ctypes.c_int, [ctypes.POINTER(GsGaussians), ctypes.POINTER(GsGaussians),
                                           ctypes.POINTER(GsCamera), ctypes.c_int64, c_void_p,
                                           ctypes.c_size_t, c_void_p, c_void_p, c_void_p]),
    "gs_render_batch_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                          ctypes.c_int64, ctypes.c_int32]),
    "gs_render_batch": (ctypes.c_int, [ctypes.POINTER(GsGaussians), ctypes.POINTER(GsCamera), ctypes.c_int32,
                                       ctypes.c_int64, c_void_p, ctypes.c_size_t, c_void_p, c_void_p, c_void_p,
                                       ctypes.POINTER(c_void_p), ctypes.c_int32]),
    "gs_rasterize_2d": (ctypes.c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, ctypes.c_int64,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, c_void_p, ctypes.c_size_t,
                                       c_void_p, c_void_p, c_void_p, c_void_p]),
    "gs_rasterize_2d_backward": (ctypes.c_int, [c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                ctypes.c_int64, c_void_p, ctypes.c_size_t, c_void_p, c_void_p,
                                                c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "gs_densify_stats": (ctypes.c_int, [c_void_p, c_void_p, ctypes.c_int64, c_void_p, c_void_p, c_void_p]),
    "gs_densify_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64]),
    "gs_densify": (ctypes.c_int, [ctypes.POINTER(GsGaussians), c_void_p, c_void_p, c_void_p, ctypes.c_float,
                                  ctypes.c_float, ctypes.c_float, ctypes.POINTER(GsGaussiansOut), c_void_p, c_void_p,
                                  c_void_p, ctypes.c_size_t, c_void_p]),
    "gs_render_from_host_async": (ctypes.c_int, [ctypes.POINTER(GsGaussians), ctypes.POINTER(GsGaussians),
                                                 ctypes.c_int64, ctypes.POINTER(GsCamera), ctypes.c_int64, c_void_p,
                                                 ctypes.c_size_t, c_void_p, c_void_p, ctypes.POINTER(c_void_p),
                                                 ctypes.POINTER(c_void_p)]),
    "gs_debug_checks_enabled": (ctypes.c_int32, []),
    "gs_debug_set_check_counter": (ctypes.c_int, [c_void_p]),
    "gs_rasterize_backward": (ctypes.c_int, [ctypes.POINTER(GsProjected), ctypes.c_int64, c_void_p, c_void_p,
                                             ctypes.POINTER(GsCamera), c_void_p, c_void_p, c_void_p, c_void_p,
                                             ctypes.POINTER(GsProjectedGrad), c_void_p]),
    "gs_preprocess_backward": (ctypes.c_int, [ctypes.POINTER(GsGaussians), ctypes.POINTER(GsCamera),
                                              ctypes.POINTER(GsProjected), ctypes.POINTER(GsProjectedGrad),
                                              ctypes.POINTER(GsGaussiansGrad), c_void_p]),
    "gs_render_backward": (ctypes.c_int, [ctypes.POINTER(GsGaussians), ctypes.POINTER(GsCamera), ctypes.c_int64,
                                          c_void_p, ctypes.c_size_t, c_void_p, c_void_p, c_void_p,
                                          ctypes.POINTER(GsGaussiansGrad), c_void_p]),
    "gs_read_status": (ctypes.c_int, [c_void_p, c_void_p, ctypes.POINTER(ctypes.c_uint32),
                                      ctypes.POINTER(ctypes.c_uint64)]),
    "gs_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64]),
    "gs_last_device_status": (ctypes.c_int, [c_void_p]),
    "gs_fp32_peak_probe": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, c_void_p,
                                          ctypes.POINTER(ctypes.c_int64), c_void_p]),
    "gs_set_spin_limit": (None, [ctypes.c_int64]),
    "gs_set_steps_order": (ctypes.c_int32, [ctypes.c_int32]),
    "gs_set_programmatic_launch": (None, [ctypes.c_int32]),
    "gs_debug_tile_key": (ctypes.c_int64, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    "gs_debug_tile_key_bits": (ctypes.c_int32, [ctypes.c_int32, ctypes.c_int32]),
    "gs_debug_tile_of_key": (ctypes.c_int64, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64]),
    "gs_test_spin_timeout": (ctypes.c_int, [c_void_p, ctypes.c_int64, c_void_p]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libgs_b300.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not _build.up_to_date():
            try:
                _build.build()
            except Exception as exc:  # no silent fallback: the product path needs the library
                raise RuntimeError(f"libgs_b300.so is missing or stale and could not be built: {exc}") from exc
        if not os.path.exists(path):
            raise RuntimeError(f"libgs_b300.so not found at {path}")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


_debug_lib = None


def debug_lib() -> ctypes.CDLL:
    """Load libgs_b300_debug.so: the same library with the kernels' index checks
    on (gs_debug_set_check_counter), building it in-tree first if needed."""
    global _debug_lib
    if _debug_lib is None:
        path = _build.DEBUG_LIB
        if not _build.up_to_date(path):
            _build.build(debug=True)
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _debug_lib = L
    return _debug_lib


class GsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib().gs_status_string(status)
        super().__init__(f"{what}: {msg.decode() if msg else status}")


def check(status: int, what: str) -> None:
    if status != GS_OK:
        raise GsError(status, what)
