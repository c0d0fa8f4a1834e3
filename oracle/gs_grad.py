"""Gradient oracle for the 3D Gaussian Splatting renderer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU legs may
import this module. It never imports the CUDA package.

The lesson page "3D Gaussian Splatting à partir de zéro" states that every stage
of the renderer is differentiable, which is what lets the parameters be fitted
by gradient descent (section "Rastérisation, non rayée"). The pages print no
backward formulas. The plain definition of the backward pass is therefore the
derivative of the forward function. This module restates the forward in plain
PyTorch float64 ops and lets autograd differentiate it:

- ``preprocess_t`` restates the projection of one Gaussian:
  - sections "Ce qu'un Gaussien porte" and "L'étape de projection":
    Sigma = R S S^T R^T, mu' = project(mu), Sigma' = J W Sigma W^T J^T,
    conic = Sigma'^-1, opacity = sigmoid(logit);
  - "Étape 5": quaternion rotation, camera-space depth;
  - "Étape 6": SH colour along the view direction, with the +0.5 offset and
    the clamp at 0.
- ``composite_t`` restates the compositing rule:
  - section "La règle de composition alpha": C = sum alpha_i T_i c_i,
    T_i = prod_{j<i} (1 - alpha_j);
  - section "Étape 2": alpha = min(0.99, o exp(-0.5 d^T Sigma'^-1 d)) at integer
    pixel coordinates;
  - the cut-offs: skip below alpha 1/255, stop once T < 1e-4, then
    image = C + T bg.
  - The list of each pixel is its tile's depth-sorted list, taken from the C
    oracle (``oracle.render``).

The discrete decisions are constants of the function, as they are for the renderer
itself: culling, tile membership, the 1/255 skip and the 1e-4 stop. They are
taken here in float64. Pixels with a decision within a relative ``band`` of a
threshold are reported in ``events`` (the same rule as the forward image test);
so are pixels where the 0.99 cap sits within the band, where the derivative
jumps. A test zeroes the upstream gradient there, because a float32 renderer may
take the other branch.

Pinned by ``tests/test_oracle_grad_pins.py``:
- the forward image equals the C oracle's fp64 composite;
- the SH basis equals the C oracle's;
- autograd matches central finite differences of this forward;
- closed forms for a single on-axis Gaussian.
"""
from __future__ import annotations

import math

import numpy as np

ALPHA_MAX = 0.99
ALPHA_MIN = 1.0 / 255.0
T_MIN = 1e-4


def _torch():
    import torch
    return torch


def sh_basis_t(d):
    """Real SH basis of bands 0..3 at unit directions d [M, 3] -> [M, 16].

    Bands 0-2 with the signs printed in eval_sh_degree_3 ("Étape 6"); band 3
    from the closed forms of the real harmonics with the band-1 sign pattern
    (odd m negative). Normalisations from their closed forms. Band 3's signs
    are parity unpinned (the pages print no band-3 code); this basis is pinned
    equal to the C oracle's."""
    torch = _torch()
    x, y, z = d[:, 0], d[:, 1], d[:, 2]
    pi = math.pi
    k0 = math.sqrt(1 / (4 * pi))
    k1 = math.sqrt(3 / (4 * pi))
    k2 = math.sqrt(15 / (4 * pi))
    k2z = math.sqrt(5 / (16 * pi))
    k2d = math.sqrt(15 / (16 * pi))
    k3a = math.sqrt(35 / (32 * pi))
    k3b = math.sqrt(105 / (4 * pi))
    k3c = math.sqrt(21 / (32 * pi))
    k3d = math.sqrt(7 / (16 * pi))
    k3e = math.sqrt(105 / (16 * pi))
    xx, yy, zz = x * x, y * y, z * z
    cols = [torch.full_like(x, k0),
            -k1 * y, k1 * z, -k1 * x,
            k2 * x * y, k2 * y * z, k2z * (2 * zz - xx - yy), k2 * x * z, k2d * (xx - yy),
            -k3a * y * (3 * xx - yy), k3b * x * y * z, -k3c * y * (4 * zz - xx - yy),
            k3d * z * (2 * zz - 3 * xx - 3 * yy), -k3c * x * (4 * zz - xx - yy), k3e * z * (xx - yy),
            -k3a * x * (xx - 3 * yy)]
    return torch.stack(cols, dim=1)


def _camera_t(cam):
    torch = _torch()
    W = torch.tensor(np.asarray(cam["R"], np.float32).reshape(3, 3).astype(np.float64))
    t = torch.tensor(np.asarray(cam["t"], np.float32).reshape(3).astype(np.float64))
    f = {k: float(np.float32(cam[k])) for k in ("fx", "fy", "cx", "cy")}
    return W, t, f


def preprocess_t(means, quats, log_scales, logits, sh, degree: int, cam) -> dict:
    """Per-Gaussian projection in float64 torch ops (differentiable)."""
    torch = _torch()
    W, t, f = _camera_t(cam)
    xc = means @ W.T + t                                     # x_c = W mu + t
    x, y, z = xc[:, 0], xc[:, 1], xc[:, 2]
    q = quats / torch.linalg.norm(quats, dim=1, keepdim=True)
    w, qx, qy, qz = q[:, 0], q[:, 1], q[:, 2], q[:, 3]
    R = torch.stack([
        torch.stack([1 - 2 * (qy * qy + qz * qz), 2 * (qx * qy - w * qz), 2 * (qx * qz + w * qy)], 1),
        torch.stack([2 * (qx * qy + w * qz), 1 - 2 * (qx * qx + qz * qz), 2 * (qy * qz - w * qx)], 1),
        torch.stack([2 * (qx * qz - w * qy), 2 * (qy * qz + w * qx), 1 - 2 * (qx * qx + qy * qy)], 1)], 1)
    S = torch.diag_embed(torch.exp(log_scales))
    RS = R @ S
    Sigma = RS @ RS.transpose(1, 2)                          # R S S^T R^T
    zero = torch.zeros_like(z)
    J = torch.stack([torch.stack([f["fx"] / z, zero, -f["fx"] * x / (z * z)], 1),
                     torch.stack([zero, f["fy"] / z, -f["fy"] * y / (z * z)], 1)], 1)
    JW = J @ W
    S2 = JW @ Sigma @ JW.transpose(1, 2)                     # J W Sigma W^T J^T
    a, b, c = S2[:, 0, 0], 0.5 * (S2[:, 0, 1] + S2[:, 1, 0]), S2[:, 1, 1]
    det = a * c - b * b
    conic = torch.stack([c / det, -b / det, a / det], 1)     # Sigma'^-1 as (A, B, C)
    u = f["fx"] * x / z + f["cx"]
    v = f["fy"] * y / z + f["cy"]
    opacity = torch.sigmoid(logits)
    centre = -(W.T @ t)                                      # camera centre
    d = means - centre
    d = d / torch.linalg.norm(d, dim=1, keepdim=True)
    nk = (degree + 1) ** 2
    Y = sh_basis_t(d)[:, :nk]
    rgb = torch.clamp(torch.einsum("gk,gkc->gc", Y, sh[:, :nk, :]) + 0.5, min=0.0)
    return {"mean2d": torch.stack([u, v], 1), "conic": conic, "opacity": opacity, "rgb": rgb, "depth": z}


def pixel_lists(sorted_vals: np.ndarray, ranges: np.ndarray, cam, px: np.ndarray, py: np.ndarray) -> np.ndarray:
    """[P, L] Gaussian indices of each pixel's tile list (in list order), -1 padded."""
    tx = (int(cam["width"]) + 15) // 16
    tiles = (py // 16) * tx + (px // 16)
    rg = ranges.astype(np.int64)
    lens = rg[tiles, 1] - rg[tiles, 0]
    L = int(lens.max()) if lens.size else 0
    idx = np.full((px.shape[0], max(L, 1)), -1, dtype=np.int64)
    for i in range(px.shape[0]):
        s, e = rg[tiles[i]]
        idx[i, : e - s] = sorted_vals[s:e]
    return idx


def composite_t(pre: dict, idx: np.ndarray, px: np.ndarray, py: np.ndarray, bg, band: float = 2e-3,
                cutoffs: bool = True):
    """Front-to-back composite of the listed pixels; returns (out [P,3], final T [P],
    n_contrib [P], events [P]). The skip/stop decisions are constants taken in
    float64 from the values themselves; ``events`` flags pixels with a skip, stop
    or cap decision within ``band`` (relative) of its threshold. cutoffs=False
    drops the 1/255 skip and the 1e-4 stop (the pages' dense rasterise_2d)."""
    torch = _torch()
    P, L = idx.shape
    valid = idx >= 0
    gi = torch.tensor(np.where(valid, idx, 0))
    u = pre["mean2d"][:, 0][gi]
    v = pre["mean2d"][:, 1][gi]
    A, B, C = pre["conic"][:, 0][gi], pre["conic"][:, 1][gi], pre["conic"][:, 2][gi]
    o = pre["opacity"][gi]
    rgb = pre["rgb"][gi]                                     # [P, L, 3]
    dx = torch.tensor(px.astype(np.float64))[:, None] - u
    dy = torch.tensor(py.astype(np.float64))[:, None] - v
    sigma = 0.5 * A * dx * dx + B * dx * dy + 0.5 * C * dy * dy
    araw = o * torch.exp(-sigma)
    alpha = torch.clamp(araw, max=ALPHA_MAX)
    # decisions (constants of the function), in list order
    a_np = alpha.detach().numpy()
    r_np = araw.detach().numpy()
    use = np.zeros((P, L), dtype=bool)
    active = np.ones(P, dtype=bool)
    T = np.ones(P)
    ev = np.zeros(P, dtype=bool)
    ncon = np.zeros(P, dtype=np.int64)
    for i in range(L):
        live = active & valid[:, i]
        ai = np.where(live, a_np[:, i], 0.0)
        ev |= live & (np.abs(ai - ALPHA_MIN) <= band * ALPHA_MIN)
        ev |= live & (np.abs(np.where(live, r_np[:, i], 0.0) - ALPHA_MAX) <= band * ALPHA_MAX)
        ui = live & (ai >= ALPHA_MIN) if cutoffs else live
        use[:, i] = ui
        T = np.where(ui, T * (1.0 - ai), T)
        ncon = np.where(ui, i + 1, ncon)
        if cutoffs:
            ev |= ui & (np.abs(T - T_MIN) <= band * T_MIN)
            active &= ~(ui & (T < T_MIN))
    w = alpha * torch.tensor(use.astype(np.float64))
    one_minus = 1.0 - w
    Tincl = torch.cumprod(one_minus, dim=1)
    Texcl = torch.cat([torch.ones((P, 1), dtype=torch.float64), Tincl[:, :-1]], dim=1)
    col = torch.einsum("pl,plc->pc", w * Texcl, rgb)
    Tfin = Tincl[:, -1]
    out = col + Tfin[:, None] * torch.tensor(np.asarray(bg, np.float64))[None, :]
    return out, Tfin, ncon, ev


def setup(scene: dict, cam: dict, grad_image: np.ndarray, ref: dict | None = None, pixels=None) -> dict:
    """The constants of one gradient evaluation: the pixels that enter (where
    grad_image is non-zero, or ``pixels`` = (px, py)), their tile lists (from the
    C oracle's sorted keys) and the Gaussians those lists use."""
    if ref is None:
        import oracle
        ref = oracle.render(scene, cam)
    gimg = np.asarray(grad_image, np.float64)
    if pixels is None:
        py, px = np.nonzero(np.any(gimg != 0.0, axis=2))
    else:
        px, py = (np.asarray(a, np.int64) for a in pixels)
    n = int(np.asarray(scene["means"]).shape[0])
    idx = pixel_lists(ref["sorted_vals"], ref["ranges"], cam, px, py)
    used = np.unique(idx[idx >= 0])
    remap = np.full(n, -1, dtype=np.int64)
    remap[used] = np.arange(used.shape[0])
    return {"px": px, "py": py, "g": gimg[py, px], "n": n, "used": used,
            "idx": np.where(idx >= 0, remap[np.maximum(idx, 0)], -1),
            "degree": int(scene["sh_degree"]),
            "bg": np.asarray(cam.get("bg", (0.0, 0.0, 0.0)), np.float32).astype(np.float64)}


PARAMS = ("means", "quats", "log_scales", "opacity_logits", "sh")


def params64(scene: dict) -> dict:
    """The scene's parameters as float64 arrays (the float32 values, exactly)."""
    return {k: np.asarray(scene[k], np.float32).astype(np.float64) for k in PARAMS}


def loss_t(st: dict, cam: dict, leaves: dict, band: float = 2e-3):
    """L = sum(grad_image * image) over the set-up pixels, for float64 parameter
    tensors ``leaves`` (full arrays); returns (L, pre, composite outputs)."""
    torch = _torch()
    ut = torch.tensor(st["used"])
    sub = {k: v[ut] for k, v in leaves.items()}
    pre = preprocess_t(sub["means"], sub["quats"], sub["log_scales"], sub["opacity_logits"], sub["sh"],
                       st["degree"], cam)
    out, Tfin, ncon, ev = composite_t(pre, st["idx"], st["px"], st["py"], st["bg"], band)
    return (torch.tensor(st["g"]) * out).sum(), pre, (out, Tfin, ncon, ev)


def loss_value(st: dict, cam: dict, p64: dict) -> float:
    """L at float64 parameter values (no gradient) -- for finite differences."""
    torch = _torch()
    with torch.no_grad():
        L, _, _ = loss_t(st, cam, {k: torch.tensor(v) for k, v in p64.items()})
    return float(L)


def render_grad(scene: dict, cam: dict, grad_image: np.ndarray, ref: dict | None = None, band: float = 2e-3,
                pixels=None, p64: dict | None = None) -> dict:
    """Gradients of L = sum(grad_image * image) with respect to the Gaussian
    parameters and the per-Gaussian projected quantities.

    grad_image: [H, W, 3]. Only pixels where it is non-zero (or the given
    ``pixels`` = (px, py) arrays) enter the composite.
    ref: the C oracle's render (for the sorted lists); computed if None.
    p64: float64 parameter values to differentiate at (default: the scene's).
    Returns numpy float64 arrays ``means``, ``quats``, ``log_scales``,
    ``opacity_logits``, ``sh`` (the parameter shapes); ``mean2d`` [N,2], ``conic`` [N,3]
    (dL/d(A, B, C) of conic = [[A, B], [B, C]]), ``opacity`` [N], ``rgb`` [N,3];
    plus ``image`` (the composite at those pixels), ``final_T``, ``n_contrib``,
    ``px``, ``py``, ``events``, ``used``, ``loss``."""
    torch = _torch()
    st = setup(scene, cam, grad_image, ref, pixels)
    p64 = params64(scene) if p64 is None else p64
    leaves = {k: torch.tensor(v, requires_grad=True) for k, v in p64.items()}
    loss, pre, (out, Tfin, ncon, ev) = loss_t(st, cam, leaves, band)
    inter = [pre["mean2d"], pre["conic"], pre["opacity"], pre["rgb"]]
    grads = torch.autograd.grad(loss, [leaves[k] for k in PARAMS] + inter, allow_unused=True)
    n, used = st["n"], st["used"]
    res = {}
    for k, gr in zip(PARAMS, grads[:5]):
        res[k] = np.zeros(p64[k].shape) if gr is None else gr.numpy()
    for k, gr, width in zip(("mean2d", "conic", "opacity", "rgb"), grads[5:], (2, 3, 1, 3)):
        full = np.zeros((n, width))
        if gr is not None:
            full[used] = gr.numpy().reshape(used.shape[0], width)
        res[k] = full[:, 0] if width == 1 else full
    res.update(image=out.detach().numpy(), final_T=Tfin.detach().numpy(), n_contrib=ncon, px=st["px"],
               py=st["py"], events=ev, used=used, loss=float(loss.detach()))
    return res


# --------------------------------------------------------------------------- 2D splats
# Section "Étape 2" (rasterise_2d) and "Étape 3" of the lesson page: Gaussians
# given directly in image space (mean, 2x2 covariance, colour, opacity) and a
# per-Gaussian scalar that only orders them; no background term.

def order_key(depths: np.ndarray) -> np.ndarray:
    """Order-preserving uint32 image of float32 values (sign bit flipped for
    non-negative values, all bits for negative ones)."""
    u = np.ascontiguousarray(depths, np.float32).view(np.uint32)
    return np.where(u & np.uint32(0x80000000), ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def decide2d_f32(means, covs, opacities, depths, width: int, height: int) -> dict:
    """The 2D tile rectangles as a binary32 program (numpy float32 element-wise
    ops, each rounded on its own, no FMA): b = (cov01 + cov10)/2, det = ac - bb,
    lam = (a+c)/2 + sqrt(((a-c)/2)^2 + b^2), r = ceil(3 sqrt(lam)); culled unless
    0 < det <= FLT_MAX, u, v, r finite, o > 0 and the depth is a number; pixel
    rectangle clipped to the image, tiles of 16x16."""
    f = np.float32
    m = np.asarray(means, f)
    c = np.asarray(covs, f).reshape(-1, 4)
    o = np.asarray(opacities, f)
    d = np.asarray(depths, f)
    with np.errstate(all="ignore"):
        a, cc = c[:, 0], c[:, 3]
        b = f(0.5) * (c[:, 1] + c[:, 2])
        det = a * cc - b * b
        hm = f(0.5) * (a - cc)
        lam = f(0.5) * (a + cc) + np.sqrt(hm * hm + b * b)
        r = np.ceil(f(3.0) * np.sqrt(lam))
        u, v = m[:, 0], m[:, 1]
        fmax = np.finfo(np.float32).max
        ok = (det > 0) & (det <= fmax) & (np.abs(u) <= fmax) & (np.abs(v) <= fmax) & (r <= fmax) & (o > 0) & ~np.isnan(d)
        x0 = np.maximum(np.ceil(u - r), f(0)); x1 = np.minimum(np.floor(u + r), f(width - 1))
        y0 = np.maximum(np.ceil(v - r), f(0)); y1 = np.minimum(np.floor(v + r), f(height - 1))
    ok &= (x0 <= x1) & (y0 <= y1)
    rect = np.zeros((m.shape[0], 4), np.int64)
    rect[ok] = np.stack([x0[ok].astype(np.int64) >> 4, y0[ok].astype(np.int64) >> 4,
                         x1[ok].astype(np.int64) >> 4, y1[ok].astype(np.int64) >> 4], 1)
    touched = np.where(ok, (rect[:, 2] - rect[:, 0] + 1) * (rect[:, 3] - rect[:, 1] + 1), 0)
    return {"tile_rect": rect, "tiles_touched": touched.astype(np.int64), "key": order_key(d)}


def lists2d(dec: dict, width: int, height: int) -> tuple:
    """Per-tile lists in the order (order key, index): (sorted_vals, ranges)."""
    tx, ty = (width + 15) // 16, (height + 15) // 16
    tiles, gids = [], []
    for gi in np.nonzero(dec["tiles_touched"] > 0)[0]:
        x0, y0, x1, y1 = dec["tile_rect"][gi]
        for yy in range(y0, y1 + 1):
            for xx in range(x0, x1 + 1):
                tiles.append(yy * tx + xx)
                gids.append(gi)
    tiles = np.asarray(tiles, np.int64)
    gids = np.asarray(gids, np.int64)
    order = np.lexsort((gids, dec["key"][gids].astype(np.int64), tiles)) if tiles.size else np.zeros(0, np.int64)
    tiles, gids = tiles[order], gids[order]
    starts = np.searchsorted(tiles, np.arange(tx * ty), "left")
    ends = np.searchsorted(tiles, np.arange(tx * ty), "right")
    return gids.astype(np.uint32), np.stack([starts, ends], 1).astype(np.uint32)


def pre2d_t(means, covs, colours, opacities) -> dict:
    """The per-Gaussian quantities the compositor reads, for 2D splats."""
    torch = _torch()
    a, c = covs[:, 0, 0], covs[:, 1, 1]
    b = 0.5 * (covs[:, 0, 1] + covs[:, 1, 0])
    det = a * c - b * b
    return {"mean2d": means, "conic": torch.stack([c / det, -b / det, a / det], 1), "opacity": opacities,
            "rgb": colours}


def render_grad_2d(means, covs, colours, opacities, depths, width: int, height: int, grad_image,
                   band: float = 2e-3, cutoffs: bool = True, dense: bool = False, exact: bool = False) -> dict:
    """Image and gradients of L = sum(grad_image * image) for 2D splats, in
    float64 torch ops. dense=True lists every Gaussian at every pixel (in depth
    order), as the pages' rasterise_2d does; otherwise each pixel gets its
    tile's list. Returns numpy ``image`` [H,W,3], ``final_T``, ``n_contrib``,
    ``events`` [H,W] and gradients ``means``, ``covs`` (full 2x2), ``colours``,
    ``opacities``. exact=True takes the continuous inputs as given (float64)
    instead of their float32 values (the decisions always use float32)."""
    torch = _torch()
    n = int(np.asarray(means).shape[0])
    py, px = np.mgrid[0:height, 0:width]
    px, py = px.ravel(), py.ravel()
    if dense:
        order = np.lexsort((np.arange(n), order_key(depths).astype(np.int64)))
        idx = np.broadcast_to(order[None, :], (px.size, n)).copy()
    else:
        dec = decide2d_f32(means, covs, opacities, depths, width, height)
        sv, rg = lists2d(dec, width, height)
        idx = pixel_lists(sv, rg, {"width": width}, px, py)
    cast = (lambda x: np.asarray(x, np.float64)) if exact else (lambda x: np.asarray(x, np.float32).astype(np.float64))
    leaves = [torch.tensor(cast(x), requires_grad=True) for x in (means, covs, colours, opacities)]
    pre = pre2d_t(*leaves)
    out, Tfin, ncon, ev = composite_t(pre, idx, px, py, np.zeros(3), band, cutoffs)
    g = torch.tensor(np.asarray(grad_image, np.float64).reshape(-1, 3))
    grads = torch.autograd.grad((g * out).sum(), leaves)
    return {"image": out.detach().numpy().reshape(height, width, 3),
            "final_T": Tfin.detach().numpy().reshape(height, width),
            "n_contrib": ncon.reshape(height, width), "events": ev.reshape(height, width),
            "means": grads[0].numpy(), "covs": grads[1].numpy(), "colours": grads[2].numpy(),
            "opacities": grads[3].numpy()}


def dense_rasterise_2d(means, covs, colours, opacities, depths, width: int, height: int) -> np.ndarray:
    """The pages' rasterise_2d written out in numpy float64: every Gaussian at
    every integer pixel, alpha = clamp(o exp(-0.5 d^T cov^-1 d), 0, 0.99), in
    increasing depth order, C += T alpha c, T *= 1 - alpha, no background."""
    m = np.asarray(means, np.float32).astype(np.float64)
    cv = np.asarray(covs, np.float32).astype(np.float64)
    col = np.asarray(colours, np.float32).astype(np.float64)
    o = np.asarray(opacities, np.float32).astype(np.float64)
    order = np.lexsort((np.arange(m.shape[0]), order_key(depths).astype(np.int64)))
    y, x = np.mgrid[0:height, 0:width].astype(np.float64)
    T = np.ones((height, width))
    out = np.zeros((height, width, 3))
    for gi in order:
        inv = np.linalg.inv(0.5 * (cv[gi] + cv[gi].T))
        dx, dy = x - m[gi, 0], y - m[gi, 1]
        q = inv[0, 0] * dx * dx + 2 * inv[0, 1] * dx * dy + inv[1, 1] * dy * dy
        a = np.clip(o[gi] * np.exp(-0.5 * q), 0.0, 0.99)
        out += (T * a)[..., None] * col[gi][None, None, :]
        T = T * (1.0 - a)
    return out


# --------------------------------------------------------------------------- densify / prune
# Section "Densation et taille": clone a Gaussian whose gradient magnitude is
# high but whose scale is small, split a large one with a high gradient into
# two smaller ones, prune those whose opacity fell below a threshold.

def densify(params: dict, accum, count, xi, grad_threshold: float, scale_threshold: float,
            prune_opacity: float) -> dict:
    """The densification step on host arrays. Decisions in float32 on the
    logit and the log-scales against thresholds mapped in float64 (o < t iff
    logit < log(t/(1-t)); max s > t iff max log s > log t), gradient g = accum /
    count (float32 division, 0 if count = 0). Split children at mu + R S xi_c,
    log-scales - log(1.6) (float64 arithmetic). Returns the new arrays
    (float64) and ``action`` (0 keep, 1 clone, 2 split, 3 prune)."""
    f = np.float32
    lg = np.asarray(params["opacity_logits"], f)
    ls = np.asarray(params["log_scales"], f)
    acc = np.asarray(accum, f)
    cnt = np.asarray(count, np.uint32)
    logit_thr = f(np.log(prune_opacity / (1.0 - prune_opacity)))
    ls_thr = f(np.log(scale_threshold))
    with np.errstate(divide="ignore", invalid="ignore"):
        avg = np.where(cnt > 0, acc / np.maximum(cnt, 1).astype(f), f(0))
    high = (cnt > 0) & (avg >= f(grad_threshold))
    big = ls.max(axis=1) > ls_thr
    action = np.where(lg < logit_thr, 3, np.where(high, np.where(big, 2, 1), 0)).astype(np.uint8)
    q = np.asarray(params["quats"], np.float64)
    q = q / np.linalg.norm(q, axis=1, keepdims=True)
    w, x, y, z = q.T
    R = np.stack([np.stack([1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y)], 1),
                  np.stack([2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x)], 1),
                  np.stack([2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)], 1)], 1)
    s = np.exp(ls.astype(np.float64))
    out = {k: [] for k in PARAMS}
    src = []
    for gi, act in enumerate(action):
        if act == 3:
            continue
        copies = 1 if act == 0 else 2
        for c in range(copies):
            src.append(gi)
            for k in PARAMS:
                out[k].append(np.asarray(params[k][gi], np.float64))
            if act == 2:
                out["means"][-1] = np.asarray(params["means"][gi], np.float64) + R[gi] @ (s[gi] * np.asarray(xi[gi, c], np.float64))
                out["log_scales"][-1] = ls[gi].astype(np.float64) - np.log(1.6)
    res = {k: np.asarray(v) for k, v in out.items()}
    res.update(action=action, source=np.asarray(src, np.int64))
    return res
