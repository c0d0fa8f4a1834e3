"""Backward pass on the GPU (through the C ABI) against the gradient oracle
(oracle/gs_grad.py: the forward restated in float64 PyTorch ops, differentiated
by autograd).

The loss is L = sum(grad_image * image) for a seeded random grad_image. Pixels
where the oracle saw a decision within 2e-3 (relative) of a threshold have
their upstream gradient set to zero: there the 1/255 skip, the 1e-4 stop or the
0.99 cap can go either way in float32, and the derivative differs between the
branches. Both sides then compute the same function.

Tolerance, per gradient array: |gpu - oracle| <= 1e-3 |oracle| + 5e-5 max|oracle|.
- The GPU path is float32. Its per-Gaussian values carry relative errors of
  1e-6 to 1e-5 (the conic of an elongated footprint more).
- A gradient is a sum over pixels with mixed signs, so an entry's own relative
  error is unbounded where its terms cancel. The absolute part is scaled by the
  array's largest entry.
- The sums use float atomics, so the GPU's rounding order varies between runs.
- Measured on all cases below: at most 4.6e-6 of the scale, a tenth of the
  bound.
"""
import numpy as np
import pytest

import gaussian_splatting_tile_02_b300 as gs
from gaussian_splatting_tile_02_b300 import native, scenes

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

RTOL = 1e-3
ATOL_FRAC = 5e-5


@pytest.fixture(scope="module", autouse=True)
def cuda_only():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    native.lib()


def gpu_backward(scene, cam, grad_image):
    g = gs.gaussians_to_device(scene)
    p = gs.preprocess(g, cam)
    cap = int(gs.bin_keys(p, cam, 0)["num_keys"].item())
    b = gs.bin_keys(p, cam, cap)
    srt = gs.sort_pairs(b["keys"], b["vals"], b["num_keys"], gs.key_bits(cam), cap)
    ranges = gs.tile_ranges(srt["keys"], b["num_keys"], cam, cap)
    fwd = gs.rasterize(p, srt["vals"], ranges, cam)
    gi = torch.tensor(np.asarray(grad_image, np.float32), device="cuda")
    pg = gs.rasterize_backward(p, srt["vals"], ranges, cam, fwd["final_T"], fwd["n_contrib"], gi)
    pr = gs.preprocess_backward(g, cam, p, pg)
    # the same frame through gs_render / gs_render_backward
    r = gs.Renderer(g, cam["width"], cam["height"], cap + 1024)
    r.render(cam)
    rg = r.render_backward(cam, gi)
    torch.cuda.synchronize()
    u = lambda d: {k: v.cpu().numpy().astype(np.float64) for k, v in d.items()}
    return u(pg), u(pr), u(rg), fwd


def quiet_grad_image(oracle_mod, scene, cam, ref, rng, window=None):
    """Seeded N(0,1) upstream gradient, zero outside ``window`` (x0, y0, x1, y1)
    and at pixels with a near-threshold decision."""
    from oracle import gs_grad
    H, W = int(cam["height"]), int(cam["width"])
    x0, y0, x1, y1 = window if window is not None else (0, 0, W, H)
    g = np.zeros((H, W, 3))
    g[y0:y1, x0:x1] = rng.standard_normal((y1 - y0, x1 - x0, 3))
    probe = gs_grad.render_grad(scene, cam, np.where(g != 0, 1.0, 0.0), ref=ref)
    ev = np.zeros((H, W), bool)
    ev[probe["py"], probe["px"]] = probe["events"]
    g[ev] = 0.0
    return g, int(ev.sum())


def compare(gpu: dict, ref: dict, keys) -> dict:
    stats = {}
    for k in keys:
        a, b = gpu[k].reshape(ref[k].shape), ref[k]
        scale = float(np.abs(b).max())
        err = np.abs(a - b)
        bound = RTOL * np.abs(b) + ATOL_FRAC * scale
        stats[k] = {"max_err_over_scale": float(err.max() / scale) if scale > 0 else float(err.max()),
                    "scale": scale, "n_bad": int((err > bound).sum())}
    return stats


def check(oracle_mod, scene, cam, window=None, seed=0):
    from oracle import gs_grad
    ref_f = oracle_mod.render(scene, cam)
    rng = np.random.default_rng(seed)
    g, n_ev = quiet_grad_image(oracle_mod, scene, cam, ref_f, rng, window)
    ref = gs_grad.render_grad(scene, cam, g, ref=ref_f)
    pg, pr, rg, fwd = gpu_backward(scene, cam, g)
    s1 = compare(pg, ref, ("mean2d", "conic", "opacity", "rgb"))
    s2 = compare(pr, ref, gs_grad.PARAMS)
    s3 = compare(rg, ref, gs_grad.PARAMS)
    print(scene.get("config"), "events zeroed", n_ev, s1, s2, s3)
    for s in (s1, s2, s3):
        for k, v in s.items():
            assert v["n_bad"] == 0, (k, v)
    # Gaussians outside every listed pixel's list have exactly zero gradient
    untouched = np.setdiff1d(np.arange(int(scene["means"].shape[0])), ref["used"])
    for k in gs_grad.PARAMS:
        assert np.all(pr[k].reshape(ref[k].shape)[untouched] == 0.0), k
    return s1, s2


def test_backward_tiny_all_pixels(oracle_mod):
    scene = scenes.make_scene("tiny")
    cam = dict(scenes.make_cameras("tiny")[0], bg=np.array([0.1, 0.2, 0.3], np.float32))
    check(oracle_mod, scene, cam)


@pytest.mark.parametrize("degree", [0, 1, 3])
def test_backward_ragged_image_sh_degrees(oracle_mod, degree):
    base = scenes.make_scene("100k", n=3000)
    k = (degree + 1) ** 2
    scene = dict(base, sh=np.ascontiguousarray(base["sh"][:, :k]), sh_degree=degree)
    cam = dict(scenes.make_cameras("100k")[0], width=150, height=109, cx=np.float32(75.0), cy=np.float32(54.5),
               fx=np.float32(160.0), fy=np.float32(160.0), bg=np.array([0.3, 0.1, 0.2], np.float32))
    check(oracle_mod, scene, cam, seed=degree)


@pytest.mark.parametrize("name,window", [("1M", (905, 503, 969, 551)), ("5M", (531, 3, 571, 43)),
                                         ("stress", (101, 701, 149, 745))])
def test_backward_full_size_window(oracle_mod, name, window):
    """Full-size workloads in the bench's launch configuration; the upstream
    gradient is non-zero on a window only, so the oracle needs only the lists
    of the pixels in it."""
    scene = scenes.make_scene(name)
    cam = scenes.make_cameras(name)[0]
    check(oracle_mod, scene, cam, window=window, seed=11)


def test_backward_empty_and_all_culled():
    scene = scenes.make_scene("tiny")
    cam = scenes.make_cameras("tiny")[0]
    behind = dict(scene, means=(scene["means"] - np.array([0, 0, 10], np.float32)).astype(np.float32))
    g = np.random.default_rng(0).standard_normal((64, 64, 3))
    pg, pr, rg, _ = gpu_backward(behind, cam, g)
    for d in (pg, pr, rg):
        for k, v in d.items():
            assert np.all(v == 0.0), k
