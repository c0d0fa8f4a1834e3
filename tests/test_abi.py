"""CPU-side checks of the C-ABI library: it builds for sm_103a, loads, exports
every entry point include/gs.h declares, and rejects bad arguments on the host
before touching the GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import gaussian_splatting_tile_02_b300 as gs
from gaussian_splatting_tile_02_b300 import build, native, scenes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gs_[a-z0-9_]+)\s*\(", text)))


def test_library_builds_and_exports_every_declared_symbol():
    build.build()
    L = native.lib()
    names = declared_functions()
    assert len(names) >= 14
    for name in names:
        assert hasattr(L, name), name
    assert set(names) == set(native._SIGNATURES), "binding must cover exactly the declared entry points"
    assert L.gs_abi_version() == 2
    assert L.gs_debug_checks_enabled() == 0


def test_debug_build_exports_the_same_symbols():
    D = native.debug_lib()
    for name in declared_functions():
        assert hasattr(D, name), name
    assert D.gs_debug_checks_enabled() == 1 and D.gs_abi_version() == 2


def test_status_strings():
    L = native.lib()
    for s in range(6):
        assert L.gs_status_string(s)
    assert L.gs_status_string(99) == b"unknown status"


def test_workspace_sizes():
    L = native.lib()
    a = L.gs_render_workspace_bytes(1000, 64, 64, 5000)
    b = L.gs_render_workspace_bytes(2000, 64, 64, 5000)
    c = L.gs_render_workspace_bytes(1000, 64, 64, 50000)
    assert 0 < a < b and a < c
    assert L.gs_render_workspace_bytes(-1, 64, 64, 10) == 0
    assert L.gs_sort_workspace_bytes(0) > 0 and L.gs_bin_workspace_bytes(0) > 0
    # 256-byte status header + aligned scratch
    assert L.gs_sort_workspace_bytes(1 << 20) % 256 == 0
    # the boundary's name for the render workspace size
    for args in ((1000, 64, 64, 5000), (10**6, 1920, 1080, 3 * 10**6), (0, 1, 1, 0), (-1, 64, 64, 10)):
        assert L.gs_workspace_bytes(*args) == L.gs_render_workspace_bytes(*args)


def test_workspace_lists_lie_inside_the_workspace():
    """gs_render_workspace_lists is host arithmetic: the sorted list and the ranges sit inside
    the workspace, 256-byte aligned, apart from each other, with room for capacity and tiles."""
    L = native.lib()
    base = 1 << 30
    for n, w, h, cap in ((1000, 64, 64, 5000), (10**6, 1920, 1080, 3 * 10**6), (0, 1, 1, 0)):
        size = L.gs_render_workspace_bytes(n, w, h, cap)
        vp, rp = ctypes.c_void_p(), ctypes.c_void_p()
        assert L.gs_render_workspace_lists(base, n, w, h, cap, ctypes.byref(vp), ctypes.byref(rp)) == native.GS_OK
        tiles = ((w + 15) // 16) * ((h + 15) // 16)
        v, r = vp.value - base, rp.value - base
        assert v % 256 == 0 and r % 256 == 0
        assert 0 < v and v + 4 * cap <= size and 0 < r and r + 8 * tiles <= size
        assert v + 4 * cap <= r or r + 8 * tiles <= v
    vp, rp = ctypes.c_void_p(), ctypes.c_void_p()
    assert L.gs_render_workspace_lists(None, 10, 64, 64, 10, ctypes.byref(vp), ctypes.byref(rp)) == \
        native.GS_ERR_WORKSPACE
    assert L.gs_render_workspace_lists(base, -1, 64, 64, 10, ctypes.byref(vp), ctypes.byref(rp)) == \
        native.GS_ERR_INVALID_ARG


def test_render_order_of_the_steps():
    """Tile-first when the key capacity is at most 2^20 pairs, unless an order is pinned."""
    L = native.lib()
    assert L.gs_render_tile_first(10**6, 1920, 1080, 1 << 20) == 1
    assert L.gs_render_tile_first(10**6, 1920, 1080, (1 << 20) + 1) == 0
    assert L.gs_render_tile_first(10**6, 1920, 1080, 3 * 10**6) == 0
    assert L.gs_render_tile_first(10**5, 1920, 1080, 400_000) == 1
    assert L.gs_render_tile_first(256, 64, 64, 2000) == 1
    assert L.gs_render_tile_first(10, 0, 64, 10) == 0
    try:
        assert L.gs_set_steps_order(1) == native.GS_OK
        assert L.gs_render_tile_first(256, 64, 64, 2000) == 0
        assert L.gs_set_steps_order(2) == native.GS_OK
        assert L.gs_render_tile_first(10**6, 1920, 1080, 3 * 10**6) == 1
        assert L.gs_set_steps_order(3) == native.GS_ERR_INVALID_ARG
        assert L.gs_set_steps_order(-1) == native.GS_ERR_INVALID_ARG
        assert L.gs_render_tile_first(10**6, 1920, 1080, 3 * 10**6) == 1
    finally:
        assert L.gs_set_steps_order(0) == native.GS_OK
    assert L.gs_render_tile_first(10**6, 1920, 1080, 3 * 10**6) == 0


def test_fp32_peak_probe_rejects_bad_arguments():
    L = native.lib()
    n = ctypes.c_int64(0)
    assert L.gs_fp32_peak_probe(0, 10, 0, 256, ctypes.byref(n), None) == native.GS_ERR_INVALID_ARG
    assert L.gs_fp32_peak_probe(4, 0, 0, 256, ctypes.byref(n), None) == native.GS_ERR_INVALID_ARG
    assert L.gs_fp32_peak_probe(4, 10, 1, None, ctypes.byref(n), None) == native.GS_ERR_INVALID_ARG


def test_last_device_status_rejects_a_missing_or_misaligned_workspace():
    L = native.lib()
    assert L.gs_last_device_status(None) == native.GS_ERR_WORKSPACE
    assert L.gs_last_device_status(256 + 8) == native.GS_ERR_WORKSPACE


def _cam(**over):
    cam = scenes.axis_camera(4.0, 64.0, 64, 64)
    cam.update(over)
    return cam


def test_host_validation_rejects_bad_arguments():
    L = native.lib()
    cam = gs.camera_struct(_cam())
    g = native.GsGaussians()
    p = native.GsProjected()
    # n < 0, degree out of range, null arrays with n > 0, null camera
    g.n = -1
    assert L.gs_preprocess(ctypes.byref(g), ctypes.byref(cam), ctypes.byref(p), None) == native.GS_ERR_INVALID_ARG
    g.n, g.sh_degree = 0, 4
    assert L.gs_preprocess(ctypes.byref(g), ctypes.byref(cam), ctypes.byref(p), None) == native.GS_ERR_INVALID_ARG
    g.n, g.sh_degree = 10, 0
    assert L.gs_preprocess(ctypes.byref(g), ctypes.byref(cam), ctypes.byref(p), None) == native.GS_ERR_INVALID_ARG
    assert L.gs_preprocess(ctypes.byref(g), None, ctypes.byref(p), None) == native.GS_ERR_INVALID_ARG
    # misaligned quaternion pointer
    g.means = g.log_scales = g.opacity_logits = g.sh = 1 << 20
    g.quats = (1 << 20) + 4
    assert L.gs_preprocess(ctypes.byref(g), ctypes.byref(cam), ctypes.byref(p), None) == native.GS_ERR_INVALID_ARG
    # bad cameras: near <= 0, zero width, non-finite focal
    for bad in (dict(near=0.0), dict(width=0), dict(fx=float("nan")), dict(height=40000)):
        c = gs.camera_struct(_cam(**bad))
        g2 = native.GsGaussians()
        g2.n = 0
        assert L.gs_preprocess(ctypes.byref(g2), ctypes.byref(c), ctypes.byref(p), None) == \
            native.GS_ERR_INVALID_ARG, bad
    # sort: bad key_bits, capacity beyond the 30-bit status words, short workspace
    assert L.gs_sort(None, None, None, None, 8, 0, 0, None, 0, None) == native.GS_ERR_INVALID_ARG
    assert L.gs_sort(None, None, None, None, 8, 0, 65, None, 0, None) == native.GS_ERR_INVALID_ARG
    assert L.gs_sort(8, 8, 8, 8, 8, 1 << 30, 40, 256, 1 << 40, None) == native.GS_ERR_INVALID_ARG
    assert L.gs_sort(8, 8, 8, 8, 8, 100, 40, 256, 16, None) == native.GS_ERR_WORKSPACE
    assert L.gs_sort(8, 8, 8, 8, 8, 100, 40, 260, 1 << 20, None) == native.GS_ERR_WORKSPACE
    # render: short workspace
    g3 = native.GsGaussians()
    g3.n = 0
    assert L.gs_render(ctypes.byref(g3), ctypes.byref(cam), 10, 256, 8, 256, None, None, None) == \
        native.GS_ERR_WORKSPACE
    assert L.gs_read_status(None, None, None, None) == native.GS_ERR_WORKSPACE
    # render / batch / 2D: n beyond the depth sort's 30-bit counts (checked before any pointer use)
    g4 = native.GsGaussians()
    g4.n, g4.sh_degree = 1 << 30, 0
    g4.means = g4.log_scales = g4.opacity_logits = g4.sh = g4.quats = 1 << 20
    assert L.gs_render(ctypes.byref(g4), ctypes.byref(cam), 10, 1 << 20, 1 << 40, 256, None, None, None) == \
        native.GS_ERR_INVALID_ARG
    cams = (native.GsCamera * 1)(cam)
    streams = (ctypes.c_void_p * 1)(None)
    assert L.gs_render_batch(ctypes.byref(g4), cams, 1, 10, 1 << 20, 1 << 40, 256, None, None, streams, 1) == \
        native.GS_ERR_INVALID_ARG
    assert L.gs_rasterize_2d(256, 256, 256, 256, 256, 1 << 30, 64, 64, 10, 1 << 20, 1 << 40, 256, None, None,
                             None) == native.GS_ERR_INVALID_ARG
    # batch: views out of range, too many streams; backward / densify: null outputs
    g3.n = 0
    assert L.gs_render_batch(ctypes.byref(g3), cams, 0, 10, 1 << 20, 1 << 40, 256, None, None, streams, 1) == \
        native.GS_ERR_INVALID_ARG
    many = (ctypes.c_void_p * 9)(*([None] * 9))
    assert L.gs_render_batch(ctypes.byref(g3), cams, 1, 10, 1 << 20, 1 << 40, 256, None, None, many, 9) == \
        native.GS_ERR_INVALID_ARG
    assert L.gs_render_backward(ctypes.byref(g3), ctypes.byref(cam), 10, 1 << 20, 1 << 40, None, None, None,
                                None, None) == native.GS_ERR_INVALID_ARG
    assert L.gs_densify(ctypes.byref(g3), None, None, None, 2e-4, 0.01, 0.005, None, None, None, None, 0,
                        None) == native.GS_ERR_INVALID_ARG
    out = native.GsGaussiansOut()
    out.n, out.sh_degree = 0, 0
    assert L.gs_densify(ctypes.byref(g3), None, None, None, 2e-4, 0.01, 1.5, ctypes.byref(out), 256, None, 256,
                        1 << 20, None) == native.GS_ERR_INVALID_ARG


def test_key_bits():
    assert gs.key_bits(scenes.make_cameras("1M")[0]) == 45        # 8160 tiles
    assert gs.key_bits(scenes.make_cameras("100k")[0]) == 43      # 1200 tiles
    assert gs.key_bits(scenes.make_cameras("tiny")[0]) == 36      # 16 tiles
    assert gs.key_bits(scenes.axis_camera(1, 1, 16, 16)) == 32    # one tile


@pytest.mark.parametrize("tiles_x,tiles_y", [(1, 1), (4, 4), (40, 30), (63, 65), (64, 64), (120, 68),
                                             (121, 67), (240, 135), (9, 500), (512, 270)])
def test_tile_keys_are_a_bijection_that_keeps_8x4_blocks_together(tiles_x, tiles_y):
    """The tile-sort keys: one per tile, all distinct and below 2^bits, inverted by
    gs_debug_tile_of_key; below 4096 tiles the key is the tile id, from 4096 up the tiles of
    one block of 8 x 4 share the key's low bits and differ only in the five above them."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    L = native.lib()
    tiles = tiles_x * tiles_y
    bits = L.gs_debug_tile_key_bits(tiles_x, tiles_y)
    assert bits == bench.tile_key_bits(tiles_x, tiles_y)
    assert 1 <= bits <= 32
    keys = {}
    for ty in range(tiles_y):
        for tx in range(tiles_x):
            k = L.gs_debug_tile_key(tiles_x, tiles_y, tx, ty)
            assert 0 <= k < (1 << bits)
            assert k not in keys
            keys[k] = (tx, ty)
            assert L.gs_debug_tile_of_key(tiles_x, tiles_y, k) == ty * tiles_x + tx
            if tiles < 4096:
                assert k == ty * tiles_x + tx
            else:
                low = k & ((1 << (bits - 5)) - 1)
                assert low == (ty // 4) * -(-tiles_x // 8) + tx // 8
                assert k >> (bits - 5) == (ty % 4) * 8 + tx % 8
    # every other key below 2^bits belongs to no tile
    valid = sum(L.gs_debug_tile_of_key(tiles_x, tiles_y, k) >= 0 for k in range(1 << bits))
    assert valid == tiles
    assert L.gs_debug_tile_of_key(tiles_x, tiles_y, 1 << bits) == -1
    assert L.gs_debug_tile_key(tiles_x, tiles_y, tiles_x, 0) == -1
    assert L.gs_debug_tile_key(tiles_x, tiles_y, 0, tiles_y) == -1
    assert L.gs_debug_tile_key_bits(0, 5) == -1
