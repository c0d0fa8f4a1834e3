"""Densification and pruning on the GPU (gs_densify_stats, gs_densify) against
the oracle's restatement of the rules (oracle/gs_grad.py densify).

Bit for bit: every action (keep, clone, split, prune), the new count, the
order of the survivors, and every copied parameter. Split children's centres
within 1e-5 of |mu| + max s, since R S xi is float32 on the GPU.
"""
import numpy as np
import pytest

import gaussian_splatting_tile_02_b300 as gs
from gaussian_splatting_tile_02_b300 import native, scenes

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_only():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    native.lib()


def synthetic_state(n, seed):
    rng = np.random.default_rng(seed)
    scene = scenes.make_scene("100k", n=n)
    scene["opacity_logits"] = rng.normal(0.0, 3.0, n).astype(np.float32)          # some below the prune threshold
    scene["log_scales"] = rng.normal(-4.0, 1.0, (n, 3)).astype(np.float32)        # both sides of log(0.01)
    accum = np.abs(rng.normal(0.0, 4e-4, n)).astype(np.float32)
    count = rng.integers(0, 4, n).astype(np.uint32)
    xi = rng.standard_normal((n, 2, 3)).astype(np.float32)
    return scene, accum, count, xi


def test_densify_matches_oracle():
    from oracle import gs_grad
    scene, accum, count, xi = synthetic_state(50_000, 0)
    g = gs.gaussians_to_device(scene)
    t = lambda a: torch.tensor(a, device="cuda")
    out = gs.densify(g, t(accum), t(count.view(np.int32)), t(xi), 2e-4, 0.01, 0.005)
    ref = gs_grad.densify(scene, accum, count, xi, 2e-4, 0.01, 0.005)
    act = out["action"].cpu().numpy()
    np.testing.assert_array_equal(act, ref["action"])
    assert all((act == a).any() for a in range(4)), np.bincount(act)
    assert out["n"] == ref["source"].shape[0]
    split = ref["action"][ref["source"]] == 2
    for k in gs_grad.PARAMS:
        a = out[k].cpu().numpy().astype(np.float64).reshape(ref[k].shape)
        if k == "means":
            scale = np.abs(ref[k]).max(1, keepdims=True) + np.exp(ref["log_scales"] + np.log(1.6)).max(1, keepdims=True)
            np.testing.assert_array_equal(a[~split], ref[k][~split])
            assert np.all(np.abs(a[split] - ref[k][split]) <= 1e-5 * scale[split])
        elif k == "log_scales":
            np.testing.assert_array_equal(a[~split], ref[k][~split])
            np.testing.assert_allclose(a[split], ref[k][split], rtol=0, atol=1e-6)
        else:
            np.testing.assert_array_equal(a, ref[k])


def test_densify_stats_accumulates_visible_gaussians():
    rng = np.random.default_rng(1)
    n = 10_000
    gm = rng.standard_normal((n, 2)).astype(np.float32)
    tt = (rng.random(n) < 0.7).astype(np.int32)
    acc = torch.zeros(n, device="cuda")
    cnt = torch.zeros(n, dtype=torch.int32, device="cuda")
    for _ in range(3):
        gs.densify_stats(torch.tensor(gm, device="cuda"), torch.tensor(tt, device="cuda"), acc, cnt)
    torch.cuda.synchronize()
    norm = np.sqrt((gm.astype(np.float64) ** 2).sum(1))
    np.testing.assert_array_equal(cnt.cpu().numpy(), 3 * tt)
    np.testing.assert_allclose(acc.cpu().numpy(), 3 * norm * tt, rtol=1e-6, atol=0)


def test_densify_capacity_overflow_is_reported():
    scene, accum, count, xi = synthetic_state(4_000, 2)
    accum[:] = 1.0
    count[:] = 1
    scene["opacity_logits"][:] = 3.0                   # nothing pruned, everything cloned or split
    g = gs.gaussians_to_device(scene)
    t = lambda a: torch.tensor(a, device="cuda")
    with pytest.raises(native.GsError):
        gs.densify(g, t(accum), t(count.view(np.int32)), t(xi), 2e-4, 0.01, 0.005, capacity=4_000 + 10)
    out = gs.densify(g, t(accum), t(count.view(np.int32)), t(xi), 2e-4, 0.01, 0.005, capacity=8_000)
    assert out["n"] == 8_000


def test_render_backward_densify_render():
    """A densification period on a real frame with a synthetic loss: render,
    backward, accumulate the statistics, densify, render the new set."""
    scene = scenes.make_scene("100k")
    cam = scenes.make_cameras("100k")[0]
    g = gs.gaussians_to_device(scene)
    p = gs.preprocess(g, cam)
    cap = int(gs.bin_keys(p, cam, 0)["num_keys"].item())
    b = gs.bin_keys(p, cam, cap)
    srt = gs.sort_pairs(b["keys"], b["vals"], b["num_keys"], gs.key_bits(cam), cap)
    ranges = gs.tile_ranges(srt["keys"], b["num_keys"], cam, cap)
    fwd = gs.rasterize(p, srt["vals"], ranges, cam)
    target = torch.zeros_like(fwd["image"])
    pg = gs.rasterize_backward(p, srt["vals"], ranges, cam, fwd["final_T"], fwd["n_contrib"],
                               2.0 * (fwd["image"] - target) / target.numel())
    n = int(g["n"])
    acc = torch.zeros(n, device="cuda")
    cnt = torch.zeros(n, dtype=torch.int32, device="cuda")
    gs.densify_stats(pg["mean2d"], p["tiles_touched"], acc, cnt)
    xi = torch.randn((n, 2, 3), device="cuda", generator=torch.Generator(device="cuda").manual_seed(0))
    thr = float(torch.quantile((acc / cnt.clamp(min=1))[cnt > 0], 0.9))
    new = gs.densify(g, acc, cnt, xi, thr, 0.01, 0.005)
    act = np.bincount(new["action"].cpu().numpy(), minlength=4)
    assert new["n"] == n + act[1] + act[2] - act[3] and act[1] + act[2] > 0
    r = gs.Renderer.for_scene(new, cam)
    r.render(cam)
    torch.cuda.synchronize()
    assert r.status()[0] == native.GS_OK
    assert np.isfinite(r.image.cpu().numpy()).all()
