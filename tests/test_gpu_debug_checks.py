"""The debug build (libgs_b300_debug.so, kernels' index checks on) on the GPU:
every path runs with zero failed checks and gives the release build's results
bit for bit; and the checks do fire, counted not trapped, on a list made
inconsistent on purpose in a way every kernel tolerates (an inverted tile
range, an index outside the scene -- both are read as empty / clamped)."""
import ctypes

import numpy as np
import pytest

import gaussian_splatting_tile_02_b300 as gs
from gaussian_splatting_tile_02_b300 import native, scenes, splat2d

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    D = native.debug_lib()
    counter = torch.zeros(1, dtype=torch.int64, device="cuda")
    native.check(D.gs_debug_set_check_counter(counter.data_ptr()), "set counter")
    yield D, counter
    native.check(D.gs_debug_set_check_counter(None), "clear counter")


def render_with(L, g, cam, cap):
    H, W = int(cam["height"]), int(cam["width"])
    wsb = int(L.gs_render_workspace_bytes(int(g["n"]), W, H, cap))
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    img = torch.empty((H, W, 3), device="cuda")
    fT = torch.empty((H, W), device="cuda")
    nc = torch.empty((H, W), dtype=torch.int32, device="cuda")
    native.check(L.gs_render(ctypes.byref(gs.gaussians_struct(g)), ctypes.byref(gs.camera_struct(cam)), cap,
                             ws.data_ptr(), wsb, img.data_ptr(), fT.data_ptr(), nc.data_ptr(), None), "render")
    gimg = torch.randn((H, W, 3), device="cuda", generator=torch.Generator(device="cuda").manual_seed(0))
    grads = gs.alloc_param_grads(g)
    native.check(L.gs_render_backward(ctypes.byref(gs.gaussians_struct(g)), ctypes.byref(gs.camera_struct(cam)), cap,
                                      ws.data_ptr(), wsb, fT.data_ptr(), nc.data_ptr(), gimg.data_ptr(),
                                      ctypes.byref(gs._ggrad_struct(grads)), None), "backward")
    torch.cuda.synchronize()
    return img.cpu().numpy(), nc.cpu().numpy(), {k: v.cpu().numpy() for k, v in grads.items()}


@pytest.mark.parametrize("name", ["tiny", "100k", "1M", "stress"])
def test_debug_build_zero_failures_and_same_results(dbg, name):
    D, counter = dbg
    scene = scenes.make_scene(name, n=300_000 if name == "stress" else None)
    cam = scenes.make_cameras(name)[0]
    g = gs.gaussians_to_device(scene)
    cap = int(gs.Renderer.count_keys(g, cam) * 1.1) + 1024
    counter.zero_()
    img_d, nc_d, gr_d = render_with(D, g, cam, cap)
    assert int(counter.item()) == 0
    img_r, nc_r, gr_r = render_with(native.lib(), g, cam, cap)
    np.testing.assert_array_equal(img_d, img_r)
    np.testing.assert_array_equal(nc_d, nc_r)
    # gradients: float atomics add each (warp, entry) partial sum in a run-dependent
    # order, and a Gaussian under thousands of pixels sums terms of both signs
    # far larger than the result, so two runs differ by more than the rounding
    # of the result; compare against the array's scale
    for k in gr_r:
        scale = max(np.abs(gr_r[k]).max(), 1e-30)
        rel = float(np.abs(gr_d[k] - gr_r[k]).max() / scale)
        print(name, k, "max |debug - release| / scale", rel)
        assert rel <= 1e-3, k


def test_debug_checks_fire_on_inconsistent_lists(dbg):
    """An inverted range and an out-of-scene index, given to step 5 directly:
    both are tolerated (empty tile, clamped index) and both are counted."""
    D, counter = dbg
    scene = scenes.make_scene("tiny")
    cam = scenes.make_cameras("tiny")[0]
    g = gs.gaussians_to_device(scene)
    p = gs.preprocess(g, cam)
    cap = int(gs.bin_keys(p, cam, 0)["num_keys"].item())
    b = gs.bin_keys(p, cam, cap)
    srt = gs.sort_pairs(b["keys"], b["vals"], b["num_keys"], gs.key_bits(cam), cap)
    ranges = gs.tile_ranges(srt["keys"], b["num_keys"], cam, cap)
    rg = ranges.clone()
    lens = (rg[:, 1] - rg[:, 0]).cpu().numpy()
    heavy = int(lens.argmax())
    assert lens[heavy] > 0
    rg[(heavy + 1) % rg.shape[0]] = torch.tensor([5, 2], dtype=torch.int32)   # end < start
    vals = srt["vals"].clone()
    vals[int(rg[heavy, 0])] = 1 << 30                       # not a Gaussian of the scene
    img = torch.empty((64, 64, 3), device="cuda")
    counter.zero_()
    native.check(D.gs_rasterize(ctypes.byref(gs.projected_struct(p)), int(g["n"]), vals.data_ptr(), rg.data_ptr(),
                                ctypes.byref(gs.camera_struct(cam)), img.data_ptr(), None, None, None, None),
                 "rasterize")
    torch.cuda.synchronize()
    assert int(counter.item()) >= 2


def test_debug_build_2d_and_densify(dbg):
    D, counter = dbg
    counter.zero_()
    # the 2D path through the debug library
    rng = np.random.default_rng(0)
    n, W, H = 500, 120, 90
    means = torch.tensor(rng.random((n, 2)) * [W, H], dtype=torch.float32, device="cuda")
    covs = torch.tensor(np.tile(np.eye(2) * 4.0, (n, 1, 1)), dtype=torch.float32, device="cuda")
    col = torch.rand((n, 3), device="cuda")
    op = torch.full((n,), 0.5, device="cuda")
    dep = torch.rand(n, device="cuda")
    cap = splat2d.key_capacity(n, W, H)
    wsb = int(D.gs_render_workspace_bytes(n, W, H, cap))
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    img = torch.empty((H, W, 3), device="cuda")
    native.check(D.gs_rasterize_2d(means.data_ptr(), covs.data_ptr(), col.data_ptr(), op.data_ptr(), dep.data_ptr(),
                                   n, W, H, cap, ws.data_ptr(), wsb, img.data_ptr(), None, None, None), "2d")
    torch.cuda.synchronize()
    assert int(counter.item()) == 0
    ref = splat2d.rasterise_2d(means, covs, col, op, dep, (H, W))
    np.testing.assert_array_equal(img.cpu().numpy(), ref.detach().cpu().numpy())
