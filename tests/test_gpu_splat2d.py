"""2D splats on the tile pipeline (gs_rasterize_2d and its backward, through the
autograd Function) against the 2D mode of the gradient oracle, and the pages'
toy fit run on the GPU kernels.

Forward: pixels where the oracle saw no decision within 2e-3 of a threshold
match its fp64 composite within 1e-4 per channel, with the same n_contrib (the
same list order and stop). Backward: the upstream gradient is zero on the
other pixels; tolerance as for the 3D backward,
|gpu - oracle| <= 1e-3 |oracle| + 5e-5 max|oracle|.
"""
import numpy as np
import pytest

from gaussian_splatting_tile_02_b300 import native, splat2d

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_only():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    native.lib()


def random_splats(n, W, H, seed):
    rng = np.random.default_rng(seed)
    means = (rng.random((n, 2)) * [W + 20, H + 20] - 10).astype(np.float32)   # some off the image
    th = rng.random(n) * np.pi
    s = np.exp(rng.normal(0.6, 0.7, (n, 2)))                                   # elongated ones too
    R = np.stack([np.stack([np.cos(th), -np.sin(th)], -1), np.stack([np.sin(th), np.cos(th)], -1)], -2)
    covs = (R @ (s[:, :, None] ** 2 * np.eye(2)[None]) @ R.transpose(0, 2, 1)).astype(np.float32)
    col = rng.random((n, 3)).astype(np.float32)
    op = (0.05 + 0.9 * rng.random(n)).astype(np.float32)
    dep = rng.normal(0, 1, n).astype(np.float32)                               # negative depths too
    dep[:5] = dep[5]                                                           # ties: by index
    return means, covs, col, op, dep


@pytest.mark.parametrize("n,W,H,seed", [(300, 150, 109, 0), (64, 64, 64, 1), (2000, 333, 200, 2)])
def test_rasterise_2d_forward_and_backward(n, W, H, seed):
    from oracle import gs_grad
    means, covs, col, op, dep = random_splats(n, W, H, seed)
    g = np.random.default_rng(seed + 10).standard_normal((H, W, 3))
    ref = gs_grad.render_grad_2d(means, covs, col, op, dep, W, H, np.ones((H, W, 3)))
    quiet = ~ref["events"]
    g[~quiet] = 0.0
    ref_g = gs_grad.render_grad_2d(means, covs, col, op, dep, W, H, g)

    t = {k: torch.tensor(v, device="cuda", requires_grad=k != "dep")
         for k, v in (("means", means), ("covs", covs), ("col", col), ("op", op), ("dep", dep))}
    img = splat2d.rasterise_2d(t["means"], t["covs"], t["col"], t["op"], t["dep"], (H, W))
    img.backward(torch.tensor(g, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    out = img.detach().cpu().numpy().astype(np.float64)
    err = np.abs(out - ref["image"]).max(-1)
    assert err[quiet].max() <= 1e-4, err[quiet].max()
    print("2d", n, W, H, "max err quiet", err[quiet].max(), "event pixels", int((~quiet).sum()))
    for name, key in (("means", "means"), ("covs", "covs"), ("col", "colours"), ("op", "opacities")):
        a = t[name].grad.cpu().numpy().astype(np.float64)
        b = ref_g[key]
        if key == "covs":   # compare the symmetric part: both sides split the off-diagonal evenly
            a = 0.5 * (a + a.transpose(0, 2, 1))
            b = 0.5 * (b + b.transpose(0, 2, 1))
        scale = np.abs(b).max()
        bad = np.abs(a - b) > 1e-3 * np.abs(b) + 5e-5 * scale
        assert not bad.any(), (name, float(np.abs(a - b).max() / scale))
    assert t["dep"].grad is None


def test_rasterise_2d_matches_n_contrib_of_oracle():
    from oracle import gs_grad
    means, covs, col, op, dep = random_splats(500, 128, 96, 5)
    ref = gs_grad.render_grad_2d(means, covs, col, op, dep, 128, 96, np.ones((96, 128, 3)))
    image, final_T, n_contrib, ws, cap = splat2d._forward(*(torch.tensor(x, device="cuda")
                                                            for x in (means, covs, col, op, dep)), 96, 128)
    torch.cuda.synchronize()
    quiet = ~ref["events"]
    np.testing.assert_array_equal(n_contrib.cpu().numpy()[quiet], ref["n_contrib"][quiet])
    np.testing.assert_allclose(final_T.cpu().numpy()[quiet], ref["final_T"][quiet], rtol=0, atol=1e-4)


def test_toy_fit_settles_into_the_two_shapes():
    """The pages' worked example: 64 Gaussians, Adam at 0.05, 200 steps of mean
    squared error against the red disc and blue square target."""
    r = splat2d.fit(steps=200, num=64, size=64, lr=0.05, seed=0)
    losses = r["losses"]
    print("toy fit mse", losses[0], losses[-1], r["final_mse"])
    assert all(np.isfinite(losses))
    assert r["final_mse"] < 0.2 * losses[0]
    # the red disc and the blue square come out in their colours
    img = r["image"]
    assert img[20, 20, 0] > 0.6 and img[20, 20, 2] < 0.5
    assert img[40, 45, 2] > 0.6 and img[40, 45, 0] < 0.5
