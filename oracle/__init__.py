"""CPU oracle for the 3D Gaussian Splatting forward renderer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package. It is a plain, slow, fp64 restatement
of the method on the lesson page "3D Gaussian Splatting à partir de zéro"
(sections "Ce qu'un Gaussien porte", "L'étape de projection", "La règle de
composition alpha", "Étape 2", "Étape 5", "Étape 6"), plus the binary32
decision program that fixes the integer results (culling, key bits, tile
rectangles) in the precision the pages' own code uses. The arithmetic lives in
``gs_oracle.c``; this module only builds it, marshals numpy arrays and
assembles the stages. It never imports the CUDA package.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, invariants, brute force, the printed constants; the
threshold-flip helper ``composite_pixel_flipped`` by closed-form pixels in
``tests/test_oracle_flip_pins.py``) except the sign
convention of SH band 3, which the pages leave out: band 3 is parity
unpinned (its orthonormality and harmonicity are pinned, its signs are a
reading).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gs_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")

# -ffp-contract=off: the decision program must round every product and sum on
# its own (gcc contracts a*b+c into an FMA by default in GNU C modes).
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math", "-mno-fma", "-fexcess-precision=standard"]

EV_SKIP = 1
EV_STOP = 2
ALPHA_MIN = 1.0 / 255.0
T_MIN = 1e-4


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class Camera(ctypes.Structure):
    _fields_ = [("R", ctypes.c_float * 9), ("t", ctypes.c_float * 3),
                ("fx", ctypes.c_float), ("fy", ctypes.c_float), ("cx", ctypes.c_float),
                ("cy", ctypes.c_float), ("near_z", ctypes.c_float),
                ("width", ctypes.c_int32), ("height", ctypes.c_int32), ("bg", ctypes.c_float * 3)]


def make_camera(cam: dict) -> Camera:
    c = Camera()
    R = np.asarray(cam["R"], dtype=np.float32).reshape(9)
    t = np.asarray(cam["t"], dtype=np.float32).reshape(3)
    bg = np.asarray(cam.get("bg", (0, 0, 0)), dtype=np.float32).reshape(3)
    for i in range(9):
        c.R[i] = float(R[i])
    for i in range(3):
        c.t[i] = float(t[i])
        c.bg[i] = float(bg[i])
    c.fx, c.fy, c.cx, c.cy = (float(np.float32(cam[k])) for k in ("fx", "fy", "cx", "cy"))
    c.near_z = float(np.float32(cam["near"]))
    c.width, c.height = int(cam["width"]), int(cam["height"])
    return c


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.or_scan.restype = ctypes.c_uint64
        _lib.or_get_threads.restype = ctypes.c_int
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def set_threads(n: int) -> None:
    lib().or_set_threads(ctypes.c_int(int(n)))


def get_threads() -> int:
    return int(lib().or_get_threads())


def tiles_xy(cam: dict) -> tuple:
    return (int(cam["width"]) + 15) // 16, (int(cam["height"]) + 15) // 16


# --------------------------------------------------------------------------- stages

def sh_basis(dirs: np.ndarray) -> np.ndarray:
    """Real SH basis (16 functions) at unit directions, [M, 16]."""
    dirs = np.ascontiguousarray(dirs, dtype=np.float64).reshape(-1, 3)
    out = np.empty((dirs.shape[0], 16), dtype=np.float64)
    L = lib()
    for i in range(dirs.shape[0]):
        L.or_sh_basis(ctypes.c_double(dirs[i, 0]), ctypes.c_double(dirs[i, 1]),
                      ctypes.c_double(dirs[i, 2]), _p(out[i]))
    return out


def eval_sh(sh: np.ndarray, degree: int, dirs: np.ndarray) -> np.ndarray:
    sh = _f32(sh)
    dirs = np.ascontiguousarray(dirs, dtype=np.float64)
    n = dirs.shape[0]
    out = np.empty((n, 3), dtype=np.float64)
    lib().or_eval_sh(ctypes.c_int64(n), _p(sh), ctypes.c_int(degree), _p(dirs), _p(out))
    return out


def project_f64(scene: dict, cam: dict) -> dict:
    n = int(scene["means"].shape[0])
    means, quats, ls, lg, sh = (_f32(scene[k]) for k in ("means", "quats", "log_scales",
                                                          "opacity_logits", "sh"))
    out = {"mean2d": np.empty((n, 2)), "conic": np.empty((n, 3)), "opacity": np.empty(n),
           "rgb": np.empty((n, 3)), "depth": np.empty(n), "cov2d": np.empty((n, 3)),
           "lam_max": np.empty(n), "valid": np.empty(n, dtype=np.uint8)}
    c = make_camera(cam)
    lib().or_project_f64(ctypes.c_int64(n), _p(means), _p(quats), _p(ls), _p(lg), _p(sh),
                         ctypes.c_int(int(scene["sh_degree"])), ctypes.byref(c),
                         _p(out["mean2d"]), _p(out["conic"]), _p(out["opacity"]), _p(out["rgb"]),
                         _p(out["depth"]), _p(out["cov2d"]), _p(out["lam_max"]), _p(out["valid"]))
    return out


def decide_f32(scene: dict, cam: dict) -> dict:
    n = int(scene["means"].shape[0])
    means, quats, ls = (_f32(scene[k]) for k in ("means", "quats", "log_scales"))
    out = {"valid": np.empty(n, dtype=np.uint8), "depth": np.empty(n, dtype=np.float32),
           "mean2d": np.empty((n, 2), dtype=np.float32), "cov2d": np.empty((n, 3), dtype=np.float32),
           "radius": np.empty(n, dtype=np.int32), "pix_rect": np.empty((n, 4), dtype=np.int32),
           "tile_rect": np.empty((n, 4), dtype=np.int32),
           "tiles_touched": np.empty(n, dtype=np.uint32)}
    c = make_camera(cam)
    lib().or_decide_f32(ctypes.c_int64(n), _p(means), _p(quats), _p(ls), ctypes.byref(c),
                        _p(out["valid"]), _p(out["depth"]), _p(out["mean2d"]), _p(out["cov2d"]),
                        _p(out["radius"]), _p(out["pix_rect"]), _p(out["tile_rect"]),
                        _p(out["tiles_touched"]))
    return out


def exp32(x: np.ndarray) -> np.ndarray:
    """The decision program's binary32 exp (Cody-Waite reduction + degree-7 Taylor)."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    y = np.empty_like(x)
    lib().or_exp32_batch(ctypes.c_int64(x.shape[0]), _p(x), _p(y))
    return y


def rect_f64(proj: dict, cam: dict) -> dict:
    n = proj["mean2d"].shape[0]
    radius = np.empty(n, dtype=np.int32)
    pix = np.empty((n, 4), dtype=np.int32)
    lib().or_rect_f64(ctypes.c_int64(n), _p(proj["mean2d"]), _p(proj["lam_max"]), _p(proj["valid"]),
                      ctypes.c_int32(int(cam["width"])), ctypes.c_int32(int(cam["height"])),
                      _p(radius), _p(pix))
    return {"radius": radius, "pix_rect": pix}


def scan(tiles_touched: np.ndarray) -> tuple:
    tt = np.ascontiguousarray(tiles_touched, dtype=np.uint32)
    off = np.empty(tt.shape[0], dtype=np.uint64)
    k = lib().or_scan(ctypes.c_int64(tt.shape[0]), _p(tt), _p(off))
    return off, int(k)


def duplicate(dec: dict, cam: dict, k: int) -> tuple:
    n = dec["depth"].shape[0]
    keys = np.empty(k, dtype=np.uint64)
    vals = np.empty(k, dtype=np.uint32)
    lib().or_duplicate(ctypes.c_int64(n), _p(dec["tiles_touched"]), _p(dec["tile_rect"]),
                       _p(dec["depth"]), ctypes.c_int32(tiles_xy(cam)[0]), _p(keys), _p(vals))
    return keys, vals


def sort_pairs(keys: np.ndarray, vals: np.ndarray) -> tuple:
    keys = np.array(keys, dtype=np.uint64, copy=True)
    vals = np.array(vals, dtype=np.uint32, copy=True)
    lib().or_sort(ctypes.c_int64(keys.shape[0]), _p(keys), _p(vals))
    return keys, vals


def tile_ranges(sorted_keys: np.ndarray, n_tiles: int) -> np.ndarray:
    sk = np.ascontiguousarray(sorted_keys, dtype=np.uint64)
    r = np.empty((n_tiles, 2), dtype=np.uint32)
    lib().or_tile_ranges(ctypes.c_int64(sk.shape[0]), _p(sk), ctypes.c_int64(n_tiles), _p(r))
    return r


def composite(proj: dict, sorted_vals: np.ndarray, ranges: np.ndarray, cam: dict,
              band: float = 0.0, max_ev: int = 8) -> dict:
    W, H = int(cam["width"]), int(cam["height"])
    P = W * H
    out = {"image": np.empty((H, W, 3)), "final_T": np.empty((H, W)),
           "n_contrib": np.empty((H, W), dtype=np.uint32), "n_eval": np.empty((H, W), dtype=np.uint32),
           "n_used": np.empty((H, W), dtype=np.uint32), "n_events": np.empty((H, W), dtype=np.int32)}
    ev_pos = np.zeros((P, max_ev), dtype=np.int32) if band > 0 else None
    ev_type = np.zeros((P, max_ev), dtype=np.int8) if band > 0 else None
    c = make_camera(cam)
    sv = np.ascontiguousarray(sorted_vals, dtype=np.uint32)
    rg = np.ascontiguousarray(ranges, dtype=np.uint32)
    lib().or_composite(ctypes.byref(c), _p(proj["mean2d"]), _p(proj["conic"]), _p(proj["opacity"]),
                       _p(proj["rgb"]), _p(sv), _p(rg), ctypes.c_double(band), ctypes.c_int(max_ev),
                       _p(out["image"]), _p(out["final_T"]), _p(out["n_contrib"]), _p(out["n_eval"]),
                       _p(out["n_used"]), _p(out["n_events"]),
                       _p(ev_pos) if ev_pos is not None else None,
                       _p(ev_type) if ev_type is not None else None)
    if band > 0:
        out["ev_pos"] = ev_pos.reshape(H, W, max_ev)
        out["ev_type"] = ev_type.reshape(H, W, max_ev)
    return out


def composite_pixel_flipped(proj: dict, sorted_vals, ranges, cam: dict, x: int, y: int,
                            flips: list) -> tuple:
    c = make_camera(cam)
    fp = np.array([f[0] for f in flips] or [0], dtype=np.int32)
    ft = np.array([f[1] for f in flips] or [0], dtype=np.int8)
    rgb = np.empty(3)
    T = np.empty(1)
    lib().or_composite_pixel_flipped(ctypes.byref(c), ctypes.c_int32(x), ctypes.c_int32(y),
                                     _p(proj["mean2d"]), _p(proj["conic"]), _p(proj["opacity"]),
                                     _p(proj["rgb"]), _p(np.ascontiguousarray(sorted_vals, dtype=np.uint32)),
                                     _p(np.ascontiguousarray(ranges, dtype=np.uint32)), _p(fp), _p(ft),
                                     ctypes.c_int(len(flips)), _p(rgb), _p(T))
    return rgb, float(T[0])


def render_untiled(proj: dict, dec: dict, cam: dict, tile_filter: bool = True,
                   window=None) -> tuple:
    W, H = int(cam["width"]), int(cam["height"])
    x0, y0, x1, y1 = window if window is not None else (0, 0, W, H)
    img = np.empty((y1 - y0, x1 - x0, 3))
    T = np.empty((y1 - y0, x1 - x0))
    c = make_camera(cam)
    n = dec["depth"].shape[0]
    lib().or_render_untiled(ctypes.byref(c), ctypes.c_int64(n), _p(dec["valid"]), _p(dec["depth"]),
                            _p(dec["tile_rect"]), _p(dec["tiles_touched"]), _p(proj["mean2d"]),
                            _p(proj["conic"]), _p(proj["opacity"]), _p(proj["rgb"]),
                            ctypes.c_int(1 if tile_filter else 0), ctypes.c_int32(x0), ctypes.c_int32(y0),
                            ctypes.c_int32(x1), ctypes.c_int32(y1), _p(img), _p(T))
    return img, T


def render(scene: dict, cam: dict, band: float = 0.0, max_ev: int = 8, timings: dict | None = None) -> dict:
    """The whole path: fp64 projection + fp32 decisions -> keys -> sort -> ranges -> composite."""
    t0 = time.perf_counter()
    proj = project_f64(scene, cam)
    dec = decide_f32(scene, cam)
    t1 = time.perf_counter()
    offsets, k = scan(dec["tiles_touched"])
    keys, vals = duplicate(dec, cam, k)
    t2 = time.perf_counter()
    skeys, svals = sort_pairs(keys, vals)
    tx, ty = tiles_xy(cam)
    ranges = tile_ranges(skeys, tx * ty)
    t3 = time.perf_counter()
    comp = composite(proj, svals, ranges, cam, band=band, max_ev=max_ev)
    t4 = time.perf_counter()
    if timings is not None:
        timings.update({"project": t1 - t0, "bin": t2 - t1, "sort": t3 - t2, "composite": t4 - t3,
                        "total": t4 - t0})
    return {"proj": proj, "dec": dec, "offsets": offsets, "num_keys": k, "keys": keys, "vals": vals,
            "sorted_keys": skeys, "sorted_vals": svals, "ranges": ranges, **comp}


def covariance3d(quats: np.ndarray, log_scales: np.ndarray) -> tuple:
    """Rotation R and Sigma = R S S^T R^T per Gaussian (fp64), [n,3,3] each."""
    q = _f32(quats).reshape(-1, 4)
    ls = _f32(log_scales).reshape(-1, 3)
    n = q.shape[0]
    R = np.empty((n, 3, 3))
    S = np.empty((n, 3, 3))
    lib().or_covariance3d(ctypes.c_int64(n), _p(q), _p(ls), _p(R), _p(S))
    return R, S
