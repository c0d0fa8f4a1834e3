"""gs_bin_static -- binning without any device allocation -- against gs_bin.

gs_bin_static exists for callers that cannot allocate device memory (plugins
whose host application owns all GPU memory, real-time loops that forbid
cudaMalloc after start-up). It keeps its scratch in a device array inside the
library, so its results must equal gs_bin's bit for bit, call after call,
whatever an earlier call left in that array. Calls go through the C ABI.
"""
import ctypes

import numpy as np
import pytest

import gaussian_splatting_tile_02_b300 as gs
from gaussian_splatting_tile_02_b300 import native, scenes

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _bin_both(g, cam, cap):
    L = native.lib()
    p = gs.preprocess(g, cam)
    n = int(g["n"])
    dev = g["means"].device
    ref = gs.bin_keys(p, cam, cap)
    off = torch.full((max(n, 1),), -1, dtype=torch.int32, device=dev)
    keys = torch.full((max(cap, 1),), -1, dtype=torch.int64, device=dev)
    vals = torch.full((max(cap, 1),), -1, dtype=torch.int32, device=dev)
    nk = torch.full((1,), -1, dtype=torch.int64, device=dev)
    st = L.gs_bin_static(ctypes.byref(gs.projected_struct(p)), n, ctypes.byref(gs.camera_struct(cam)),
                         off.data_ptr(), keys.data_ptr(), vals.data_ptr(), cap, nk.data_ptr(),
                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == native.GS_OK
    torch.cuda.synchronize()
    K = int(ref["num_keys"].item())
    assert int(nk.item()) == K
    m = min(K, cap)
    np.testing.assert_array_equal(off[:n].cpu().numpy(), ref["offsets"][:n].cpu().numpy())
    np.testing.assert_array_equal(keys[:m].cpu().numpy(), ref["keys"][:m].cpu().numpy())
    np.testing.assert_array_equal(vals[:m].cpu().numpy(), ref["vals"][:m].cpu().numpy())
    return K


def test_bin_static_matches_bin_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    big = gs.gaussians_to_device(scenes.make_scene("100k"))
    cam_big = scenes.make_cameras("100k")[0]
    small = gs.gaussians_to_device(scenes.make_scene("tiny"))
    cam_small = scenes.make_cameras("tiny")[0]
    # the larger problem first, so the second call runs over what it left behind
    k1 = _bin_both(big, cam_big, 400_000)
    k2 = _bin_both(small, cam_small, 2000)
    assert k1 > 100_000 and 0 < k2 < 2000
    # and once more with a capacity below the key count
    _bin_both(big, cam_big, k1 - 5000)


def test_bin_static_rejects_oversized_input():
    L = native.lib()
    p = native.GsProjected()
    cam = gs.camera_struct(scenes.axis_camera(4.0, 64.0, 64, 64))
    too_many = 16777216 + 1
    st = L.gs_bin_static(ctypes.byref(p), too_many, ctypes.byref(cam), 256, 256, 256, 16, 256, None)
    assert st == native.GS_ERR_INVALID_ARG
