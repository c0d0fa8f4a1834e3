"""Seeded synthetic scenes and pinhole cameras for the forward renderer.

This module only draws random inputs and builds camera poses; it contains none
of the renderer's arithmetic (no projection, covariance, colour or compositing),
so both the CUDA path and the CPU oracle can take their inputs from it.

Scene shapes follow the workloads described on the lesson page "3D Gaussian
Splatting à partir de zéro" (section "Ce qu'un Gaussien porte": per Gaussian a
mean (3), a unit quaternion (4), log-scales (3), an opacity and 3·(L+1)^2
spherical-harmonic coefficients; 1-5 M Gaussians per scene; SH degree 3).

Array layout (all float32, C-contiguous):
    means           [N, 3]      world-space centres
    quats           [N, 4]      (w, x, y, z)
    log_scales      [N, 3]
    opacity_logits  [N]
    sh              [N, (D+1)^2, 3]   coefficient k, colour channel c

Camera (dict): R [3,3] world->camera rotation (row-major), t [3] so that
x_cam = R x_world + t; fx, fy, cx, cy, near, width, height, bg [3].
Camera axes: x right, y down, z forward.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = ["CONFIGS", "SceneConfig", "make_scene", "make_cameras", "orbit_camera",
           "axis_camera", "scene_nbytes"]


@dataclass(frozen=True)
class SceneConfig:
    name: str
    n: int
    width: int
    height: int
    sh_degree: int
    seed: int
    focal: float
    means: str                   # "uniform", "clusters", "ball_mix"
    means_half: float            # half side of the uniform box / cluster box
    n_clusters: int = 0
    cluster_sigma: float = 0.0
    ball_fraction: float = 0.0
    ball_radius: float = 0.0
    log_scale_mu: float = 0.0
    log_scale_sigma: float = 0.0
    logit_mu: float = 0.0
    logit_sigma: float = 1.0
    dc: str = "sym"              # "unit": DC ~ U(0,1); "sym": DC ~ U(-1,1)
    rest_sigma: float = 0.05     # higher SH bands ~ N(0, rest_sigma)
    camera: str = "axis"         # "axis": on the -z axis looking +z; "orbit"
    cam_distance: float = 4.0
    views: tuple = (0.0,)        # orbit angles in degrees
    near: float = 0.2
    bg: tuple = (0.0, 0.0, 0.0)
    description: str = ""

    @property
    def n_coeffs(self) -> int:
        return (self.sh_degree + 1) ** 2


CONFIGS = {
    "tiny": SceneConfig(
        name="tiny", n=256, width=64, height=64, sh_degree=0, seed=0, focal=64.0,
        means="uniform", means_half=1.0, log_scale_mu=-2.5, log_scale_sigma=0.3,
        logit_mu=0.0, logit_sigma=1.0, dc="unit", camera="axis", cam_distance=4.0,
        description="256 Gaussians, 64x64, SH degree 0"),
    "100k": SceneConfig(
        name="100k", n=100_000, width=640, height=480, sh_degree=3, seed=1, focal=500.0,
        means="uniform", means_half=2.0, log_scale_mu=-4.0, log_scale_sigma=0.5,
        logit_mu=0.0, logit_sigma=1.5, dc="sym", camera="axis", cam_distance=6.0,
        description="100k Gaussians, 640x480, SH degree 3"),
    "1M": SceneConfig(
        name="1M", n=1_000_000, width=1920, height=1080, sh_degree=3, seed=2, focal=1100.0,
        means="clusters", means_half=5.0, n_clusters=64, cluster_sigma=0.3,
        log_scale_mu=-4.5, log_scale_sigma=0.6, logit_mu=0.5, logit_sigma=1.5, dc="sym",
        camera="orbit", cam_distance=12.0, views=(0.0,),
        description="1M Gaussians, 1920x1080, SH degree 3, 64 clusters, orbit radius 12"),
    "5M": SceneConfig(
        name="5M", n=5_000_000, width=1920, height=1080, sh_degree=3, seed=3, focal=1100.0,
        means="clusters", means_half=5.0, n_clusters=256, cluster_sigma=0.3,
        log_scale_mu=-4.5, log_scale_sigma=0.6, logit_mu=0.5, logit_sigma=1.5, dc="sym",
        camera="orbit", cam_distance=12.0, views=(0.0, 90.0, 180.0, 270.0),
        description="5M Gaussians, 1920x1080, SH degree 3, 256 clusters, 4 orbit views"),
    "stress": SceneConfig(
        name="stress", n=2_000_000, width=1920, height=1080, sh_degree=3, seed=4, focal=1100.0,
        means="ball_mix", means_half=5.0, ball_fraction=0.6, ball_radius=0.5,
        log_scale_mu=-3.5, log_scale_sigma=0.8, logit_mu=1.0, logit_sigma=1.0, dc="sym",
        camera="orbit", cam_distance=8.0, views=tuple(45.0 * k for k in range(8)),
        description="2M Gaussians, 60% in a radius-0.5 ball, 1920x1080, SH degree 3, 8 views"),
}


def _unit_quaternions(rng: np.random.Generator, n: int) -> np.ndarray:
    q = rng.standard_normal((n, 4), dtype=np.float32)
    norm = np.sqrt(np.sum(q.astype(np.float64) ** 2, axis=1, keepdims=True))
    norm[norm == 0] = 1.0
    return (q / norm).astype(np.float32)


def _means(cfg: SceneConfig, rng: np.random.Generator, n: int) -> np.ndarray:
    h = cfg.means_half
    if cfg.means == "uniform":
        return rng.uniform(-h, h, size=(n, 3)).astype(np.float32)
    if cfg.means == "clusters":
        centres = rng.uniform(-h, h, size=(cfg.n_clusters, 3))
        which = rng.integers(0, cfg.n_clusters, size=n)
        pts = centres[which] + cfg.cluster_sigma * rng.standard_normal((n, 3))
        return pts.astype(np.float32)
    if cfg.means == "ball_mix":
        n_ball = int(round(cfg.ball_fraction * n))
        d = rng.standard_normal((n_ball, 3))
        d /= np.linalg.norm(d, axis=1, keepdims=True)
        r = cfg.ball_radius * rng.random(n_ball) ** (1.0 / 3.0)
        ball = d * r[:, None]
        box = rng.uniform(-h, h, size=(n - n_ball, 3))
        pts = np.concatenate([ball, box], axis=0)
        return pts[rng.permutation(n)].astype(np.float32)
    raise ValueError(cfg.means)


def make_scene(cfg: SceneConfig | str, n: int | None = None, seed: int | None = None) -> dict:
    """Draw one scene. ``n`` overrides the Gaussian count (same distributions)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    n = cfg.n if n is None else int(n)
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    means = _means(cfg, rng, n)
    quats = _unit_quaternions(rng, n)
    log_scales = (cfg.log_scale_mu + cfg.log_scale_sigma *
                  rng.standard_normal((n, 3), dtype=np.float32)).astype(np.float32)
    logits = (cfg.logit_mu + cfg.logit_sigma *
              rng.standard_normal(n, dtype=np.float32)).astype(np.float32)
    k = cfg.n_coeffs
    sh = np.empty((n, k, 3), dtype=np.float32)
    if cfg.dc == "unit":
        sh[:, 0, :] = rng.random((n, 3), dtype=np.float32)
    else:
        sh[:, 0, :] = 2.0 * rng.random((n, 3), dtype=np.float32) - 1.0
    if k > 1:
        sh[:, 1:, :] = cfg.rest_sigma * rng.standard_normal((n, k - 1, 3), dtype=np.float32)
    return {"means": np.ascontiguousarray(means), "quats": quats,
            "log_scales": log_scales, "opacity_logits": logits, "sh": sh,
            "sh_degree": cfg.sh_degree, "n": n, "config": cfg.name}


def axis_camera(distance: float, focal: float, width: int, height: int,
                near: float = 0.2, bg=(0.0, 0.0, 0.0)) -> dict:
    """Camera at (0, 0, -distance) looking along +z (identity rotation)."""
    return {"R": np.eye(3, dtype=np.float32),
            "t": np.array([0.0, 0.0, distance], dtype=np.float32),
            "fx": float(focal), "fy": float(focal),
            "cx": width / 2.0, "cy": height / 2.0, "near": float(near),
            "width": int(width), "height": int(height),
            "bg": np.asarray(bg, dtype=np.float32)}


def orbit_camera(theta_deg: float, radius: float, focal: float, width: int, height: int,
                 near: float = 0.2, bg=(0.0, 0.0, 0.0)) -> dict:
    """Camera on a horizontal circle of ``radius`` around the origin, looking at it.

    Centre C = (r sin th, 0, -r cos th); camera axes x = (cos th, 0, sin th),
    y = (0, 1, 0), z = (-sin th, 0, cos th); t = -R C.  th = 0 gives the
    axis camera.
    """
    th = math.radians(theta_deg)
    R = np.array([[math.cos(th), 0.0, math.sin(th)],
                  [0.0, 1.0, 0.0],
                  [-math.sin(th), 0.0, math.cos(th)]], dtype=np.float64)
    C = np.array([radius * math.sin(th), 0.0, -radius * math.cos(th)])
    t = -R @ C
    return {"R": R.astype(np.float32), "t": t.astype(np.float32),
            "fx": float(focal), "fy": float(focal),
            "cx": width / 2.0, "cy": height / 2.0, "near": float(near),
            "width": int(width), "height": int(height),
            "bg": np.asarray(bg, dtype=np.float32)}


def make_cameras(cfg: SceneConfig | str, bg=None) -> list:
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    bg = cfg.bg if bg is None else bg
    if cfg.camera == "axis":
        return [axis_camera(cfg.cam_distance, cfg.focal, cfg.width, cfg.height, cfg.near, bg)]
    return [orbit_camera(th, cfg.cam_distance, cfg.focal, cfg.width, cfg.height, cfg.near, bg)
            for th in cfg.views]


def scene_nbytes(scene: dict) -> int:
    return sum(scene[k].nbytes for k in ("means", "quats", "log_scales", "opacity_logits", "sh"))
