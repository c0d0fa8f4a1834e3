"""Pins of the gradient oracle (oracle/gs_grad.py) against things other than
itself: the C oracle's forward composite, the C oracle's SH basis, central
finite differences of the forward, and closed forms for one Gaussian seen
along the optical axis (CPU only)."""
import math

import numpy as np
import pytest

import oracle
from oracle import gs_grad
from gaussian_splatting_tile_02_b300 import scenes

torch = pytest.importorskip("torch")


def _tiny():
    s = scenes.make_scene("tiny")
    cam = scenes.make_cameras("tiny")[0]
    cam = dict(cam, bg=np.array([0.1, 0.2, 0.3], np.float32))
    return s, cam


def test_forward_equals_c_oracle_composite():
    s, cam = _tiny()
    ref = oracle.render(s, cam, band=2e-3, max_ev=16)
    g = np.ones((64, 64, 3))
    r = gs_grad.render_grad(s, cam, g, ref=ref)
    img = np.zeros((64, 64, 3))
    img[r["py"], r["px"]] = r["image"]
    np.testing.assert_allclose(img, ref["image"], rtol=0, atol=1e-12)
    T = np.zeros((64, 64))
    T[r["py"], r["px"]] = r["final_T"]
    np.testing.assert_allclose(T, ref["final_T"], rtol=0, atol=1e-12)
    nc = np.zeros((64, 64), np.int64)
    nc[r["py"], r["px"]] = r["n_contrib"]
    np.testing.assert_array_equal(nc, ref["n_contrib"].astype(np.int64))
    ev = np.zeros((64, 64), bool)
    ev[r["py"], r["px"]] = r["events"]
    # the C oracle flags skip/stop events; this oracle adds the 0.99 cap
    assert np.all(ev[ref["n_events"] > 0])


def test_sh_basis_equals_c_oracle():
    d = np.random.default_rng(3).standard_normal((200, 3))
    d /= np.linalg.norm(d, axis=1, keepdims=True)
    np.testing.assert_allclose(gs_grad.sh_basis_t(torch.tensor(d)).numpy(), oracle.sh_basis(d), rtol=0, atol=1e-14)


@pytest.mark.parametrize("config", ["tiny", "100k"])
def test_autograd_matches_central_differences(config):
    if config == "tiny":
        s, cam = _tiny()
    else:
        s = scenes.make_scene("100k", n=400)
        cam = dict(scenes.make_cameras("100k")[0], width=96, height=80, cx=np.float32(48), cy=np.float32(40))
    H, W = int(cam["height"]), int(cam["width"])
    ref = oracle.render(s, cam)
    rng = np.random.default_rng(7)
    g = rng.standard_normal((H, W, 3))
    # keep pixels whose decisions are far (1%) from every threshold, so that a
    # perturbation of 1e-6 cannot move them
    probe = gs_grad.render_grad(s, cam, np.ones((H, W, 3)), ref=ref, band=1e-2)
    ev = np.zeros((H, W), bool)
    ev[probe["py"], probe["px"]] = probe["events"]
    g[ev] = 0.0
    r = gs_grad.render_grad(s, cam, g, ref=ref)
    st = gs_grad.setup(s, cam, g, ref)
    p64 = gs_grad.params64(s)
    used = r["used"]
    checked = 0
    for k in gs_grad.PARAMS:
        arr = p64[k]
        for _ in range(8):
            gi = int(rng.choice(used))
            sub = np.unravel_index(int(rng.integers(arr[gi].size)), arr[gi].shape) if arr[gi].ndim else ()
            pos = (gi, *sub)
            h = 1e-6 * max(1.0, abs(arr[pos]))
            plus, minus = {kk: v.copy() for kk, v in p64.items()}, {kk: v.copy() for kk, v in p64.items()}
            plus[k][pos] += h
            minus[k][pos] -= h
            fd = (gs_grad.loss_value(st, cam, plus) - gs_grad.loss_value(st, cam, minus)) / (2 * h)
            ad = r[k][pos]
            assert abs(fd - ad) <= 2e-6 * (1.0 + abs(ad)), (k, pos, fd, ad)
            checked += 1
    assert checked == 40


def _single(pixel):
    """One isotropic Gaussian on the optical axis of the tiny camera, seen at
    integer pixel (32, 32); upstream gradient e_r at ``pixel`` only."""
    s_px = 0.05
    scene = {"means": np.zeros((1, 3), np.float32), "quats": np.array([[1, 0, 0, 0]], np.float32),
             "log_scales": np.full((1, 3), np.log(s_px), np.float32),
             "opacity_logits": np.array([0.3], np.float32),
             "sh": np.array([[[0.2, 0.7, 0.4]]], np.float32), "sh_degree": 0}
    cam = dict(scenes.make_cameras("tiny")[0], bg=np.array([0.1, 0.2, 0.3], np.float32))
    g = np.zeros((64, 64, 3))
    g[pixel[1], pixel[0], 0] = 1.0
    r = gs_grad.render_grad(scene, cam, g)
    p = gs_grad.params64(scene)
    o = 1.0 / (1.0 + math.exp(-p["opacity_logits"][0]))
    c_r = math.sqrt(1 / (4 * math.pi)) * p["sh"][0, 0, 0] + 0.5
    s = math.exp(p["log_scales"][0, 0])
    A = (4.0 / (64.0 * s)) ** 2                       # conic of Sigma' = (f s / z)^2 I
    return r, o, c_r, A, s


def test_closed_form_at_the_centre():
    r, o, c_r, A, s = _single((32, 32))
    bg_r = np.float64(np.float32(0.1))
    assert r["image"][0, 0] == pytest.approx(o * c_r + (1 - o) * bg_r, rel=1e-14)
    assert r["sh"][0, 0, 0] == pytest.approx(o * math.sqrt(1 / (4 * math.pi)), rel=1e-13)
    assert r["sh"][0, 0, 1] == 0.0 and r["sh"][0, 0, 2] == 0.0
    assert r["opacity_logits"][0] == pytest.approx((c_r - bg_r) * o * (1 - o), rel=1e-13)
    assert r["opacity"][0] == pytest.approx(c_r - bg_r, rel=1e-13)
    assert r["rgb"][0, 0] == pytest.approx(o, rel=1e-13)
    # at the centre the Gaussian's shape and position have zero first-order effect
    np.testing.assert_allclose(r["means"], 0.0, atol=1e-14)
    np.testing.assert_allclose(r["quats"], 0.0, atol=1e-14)
    np.testing.assert_allclose(r["log_scales"], 0.0, atol=1e-14)
    np.testing.assert_allclose(r["mean2d"], 0.0, atol=1e-14)


def test_closed_form_one_pixel_right_of_the_centre():
    r, o, c_r, A, s = _single((33, 32))
    bg_r = np.float64(np.float32(0.1))
    alpha = o * math.exp(-0.5 * A)                     # dx = 1, dy = 0
    dLda = c_r - bg_r
    z, f = 4.0, 64.0
    # d alpha / d u = alpha A dx; u = f x / z + cx
    assert r["mean2d"][0, 0] == pytest.approx(dLda * alpha * A, rel=1e-12)
    assert r["means"][0, 0] == pytest.approx(dLda * alpha * A * f / z, rel=1e-12)
    assert abs(r["means"][0, 1]) < 1e-13
    # depth enters through A = (z / (f s))^2: dA/dz = 2 A / z, d sigma / dA = dx^2 / 2
    assert r["means"][0, 2] == pytest.approx(-dLda * alpha * 0.5 * (2 * A / z), rel=1e-12)
    # scales: A = (z/f)^2 / s_x^2, so dA/dlog s_x = -2 A; s_y and s_z do not enter at dy = 0
    assert r["log_scales"][0, 0] == pytest.approx(dLda * alpha * A, rel=1e-12)
    assert abs(r["log_scales"][0, 1]) < 1e-13 and abs(r["log_scales"][0, 2]) < 1e-13
    assert r["conic"][0, 0] == pytest.approx(-dLda * alpha * 0.5, rel=1e-12)


def _splats2d(n=40, W=50, H=37, seed=0):
    rng = np.random.default_rng(seed)
    means = (rng.random((n, 2)) * [W, H]).astype(np.float32)
    th = rng.random(n) * np.pi
    s = np.exp(rng.normal(0.8, 0.5, (n, 2)))
    R = np.stack([np.stack([np.cos(th), -np.sin(th)], -1), np.stack([np.sin(th), np.cos(th)], -1)], -2)
    covs = (R @ (s[:, :, None] ** 2 * np.eye(2)[None]) @ R.transpose(0, 2, 1)).astype(np.float32)
    col = rng.random((n, 3)).astype(np.float32)
    op = (0.2 + 0.7 * rng.random(n)).astype(np.float32)
    dep = rng.normal(0, 1, n).astype(np.float32)
    return means, covs, col, op, dep, W, H


def test_2d_dense_mode_is_the_pages_formula():
    """With every Gaussian listed at every pixel and no cut-offs, the 2D oracle is
    the pages' rasterise_2d written out separately in numpy."""
    args = _splats2d()
    W, H = args[-2], args[-1]
    dense = gs_grad.dense_rasterise_2d(*args)
    r = gs_grad.render_grad_2d(*args, np.ones((H, W, 3)), cutoffs=False, dense=True)
    np.testing.assert_allclose(r["image"], dense, rtol=0, atol=1e-13)
    # the tile renderer's cut-offs (3-sigma tiles, 1/255 skip, 1e-4 stop) move
    # pixels by at most about 0.011 per truncated Gaussian
    t = gs_grad.render_grad_2d(*args, np.ones((H, W, 3)))
    assert 0.0 < np.abs(t["image"] - dense).max() < 0.02


def test_2d_order_key_and_rectangles():
    keys = gs_grad.order_key(np.float32([-2.0, -0.0, 0.0, 1e-30, 3.0, -1e30]))
    assert list(np.argsort(keys, kind="stable")) == [5, 0, 1, 2, 3, 4]
    # an isotropic Gaussian of variance 4 at (20.5, 9): r = ceil(3 * 2) = 6
    d = gs_grad.decide2d_f32(np.float32([[20.5, 9.0]]), np.float32([[[4, 0], [0, 4]]]), np.float32([0.5]),
                             np.float32([0.0]), 64, 64)
    # pixels x in [ceil(14.5), floor(26.5)] = [15, 26], y in [3, 15] -> tiles x 0..1, y 0..0
    assert list(d["tile_rect"][0]) == [0, 0, 1, 0] and d["tiles_touched"][0] == 2


def test_2d_gradients_match_central_differences():
    means, covs, col, op, dep, W, H = _splats2d(n=12, W=33, H=20, seed=3)
    g = np.random.default_rng(1).standard_normal((H, W, 3))
    probe = gs_grad.render_grad_2d(means, covs, col, op, dep, W, H, np.ones((H, W, 3)), band=1e-2)
    g[probe["events"]] = 0.0
    r = gs_grad.render_grad_2d(means, covs, col, op, dep, W, H, g)
    base = {"means": means, "covs": covs, "colours": col, "opacities": op}
    rng = np.random.default_rng(2)
    for k, arr in base.items():
        for _ in range(4):
            pos = tuple(int(rng.integers(sz)) for sz in arr.shape)
            h = 1e-6 * max(1.0, abs(float(arr[pos])))
            vals = []
            for sgn in (1, -1):
                a2 = {kk: v.astype(np.float64).copy() for kk, v in base.items()}
                a2[k][pos] += sgn * h
                if k == "covs":   # keep the matrix symmetric: perturb both off-diagonal entries
                    if pos[1] != pos[2]:
                        a2[k][(pos[0], pos[2], pos[1])] += sgn * h
                img = gs_grad.render_grad_2d(a2["means"], a2["covs"], a2["colours"], a2["opacities"], dep, W, H,
                                             g, exact=True)["image"]
                vals.append(float((g * img).sum()))
            fd = (vals[0] - vals[1]) / (2 * h)
            ad = r[k][pos] + (r[k][(pos[0], pos[2], pos[1])] if k == "covs" and pos[1] != pos[2] else 0.0)
            assert abs(fd - ad) <= 1e-6 * (1.0 + abs(ad)), (k, pos, fd, ad)


def test_densify_rules_on_hand_made_cases():
    """One Gaussian per rule: prune (o < 0.005), keep (low gradient), clone (high
    gradient, small), split (high gradient, large) with xi = 0 and xi = e_x;
    and the boundaries: gradient exactly at the threshold counts as high,
    opacity exactly at the threshold is kept."""
    logit = lambda o: np.float32(np.log(o / (1 - o)))
    t = np.log(np.float32(0.005) / (1 - np.float32(0.005)))
    p = {"means": np.float32([[0, 0, 0], [1, 0, 0], [2, 0, 0], [3, 0, 0], [4, 0, 0], [5, 0, 0]]),
         "quats": np.float32([[1, 0, 0, 0]] * 6),
         "log_scales": np.float32([[-5, -5, -5], [-5, -5, -5], [-5, -6, -7], [-1, -3, -3], [-5, -5, -5],
                                   [np.log(0.2), -3, -3]]),
         "opacity_logits": np.float32([logit(0.001), logit(0.5), logit(0.5), logit(0.5), np.float32(t) + 1e-3, 2.0]),
         "sh": np.zeros((6, 1, 3), np.float32)}
    accum = np.float32([1.0, 1e-5, 4e-4, 1.0, 0.0, 2e-4])
    count = np.uint32([1, 1, 2, 1, 0, 1])
    xi = np.zeros((6, 2, 3), np.float32)
    xi[5, 1] = [1, 0, 0]
    r = gs_grad.densify(p, accum, count, xi, 2e-4, 0.01, 0.005)
    assert list(r["action"]) == [3, 0, 1, 2, 0, 2]
    assert list(r["source"]) == [1, 2, 2, 3, 3, 4, 5, 5]
    # split with xi = 0: children at the parent's centre; xi = e_x: + s_x e_x
    np.testing.assert_allclose(r["means"][3], [3, 0, 0], atol=1e-12)
    np.testing.assert_allclose(r["means"][7], [5 + 0.2, 0, 0], rtol=1e-6)
    np.testing.assert_allclose(r["log_scales"][6], np.float32([np.log(0.2), -3, -3]) - np.log(1.6), rtol=1e-12)
    np.testing.assert_array_equal(r["means"][1], r["means"][2])   # clone = exact copy
