"""Pins for the oracle's threshold-flip helper, composite_pixel_flipped (CPU).

The GPU image check accepts a pixel that is off by more than the tolerance
only if the oracle's composite of that pixel, with one or two of its
near-threshold decisions inverted, reproduces it ("several results are
correct"). These tests pin the helper that re-composites a pixel with chosen
decisions inverted, on hand-made pixels whose results have closed forms:

- the skip below 1/255 inverted for a Gaussian whose alpha sits just below
  (or just above) it;
- the stop once T < 1e-4 inverted at the layer where T crosses it (so the next
  layer is taken), and at a layer before it (so the walk ends early);
- both at once;
- flips at positions the walk never reaches, or of a decision that is never
  taken there, change nothing;
- with no flips the helper equals the whole-image composite, on a non-square
  image.

Compositing rule: lesson page "3D Gaussian Splatting à partir de zéro",
section "La règle de composition alpha" (C = sum alpha_i T_i c_i,
T_{i+1} = T_i (1 - alpha_i), front to back), with the tile renderer's
cut-offs (skip alpha < 1/255, stop once T < 1e-4). At a Gaussian's projected
centre alpha equals its opacity exactly (exp(0) = 1).
"""
import math

import numpy as np
import pytest

from gaussian_splatting_tile_02_b300 import scenes

C0 = math.sqrt(1.0 / (4.0 * math.pi))
CX = CY = 32          # principal point of the 64x64 camera: every on-axis Gaussian projects here


def _scene(means, logits, dcs):
    n = len(means)
    sh = np.zeros((n, 1, 3), np.float32)
    sh[:, 0, :] = np.asarray(dcs, np.float32)
    return {"means": np.asarray(means, np.float32).reshape(n, 3),
            "quats": np.tile(np.float32([1, 0, 0, 0]), (n, 1)),
            "log_scales": np.full((n, 3), math.log(0.05), np.float32),
            "opacity_logits": np.asarray(logits, np.float32).reshape(n),
            "sh": sh, "sh_degree": 0, "n": n}


def _logit(o):
    return math.log(o / (1.0 - o))


def _opacity(o):
    """The opacity the path sees for target o: sigmoid of the float32 logit."""
    return 1.0 / (1.0 + math.exp(-float(np.float32(_logit(o)))))


def _colour(dc):
    return C0 * np.asarray(dc, np.float32).astype(np.float64) + 0.5


def _cam(bg):
    return scenes.axis_camera(4.0, 64.0, 64, 64, 0.2, bg)


BG = (0.25, 0.5, 0.75)
N_STACK = 10
A_STACK = 0.95            # (1 - 0.95)^3 = 1.25e-4 >= 1e-4 > (1 - 0.95)^4: four layers taken


def _stack_dcs():
    # a different colour per layer, so that which layers are taken shows in the pixel
    return [[0.1 * k - 0.4, 0.5 - 0.07 * k, 0.03 * k * k - 0.2] for k in range(N_STACK)]


def _stack_scene(front_o=None):
    """Ten on-axis layers with opacity 0.95 at depths 2.0, 2.3, ...; optionally one more
    on-axis Gaussian in front of them (depth 1.5) with opacity front_o."""
    means = [[0.0, 0.0, -2.0 + 0.3 * k] for k in range(N_STACK)]
    logits = [_logit(A_STACK)] * N_STACK
    dcs = _stack_dcs()
    if front_o is not None:
        means = [[0.0, 0.0, -2.5]] + means
        logits = [_logit(front_o)] + logits
        dcs = [[0.6, -0.1, 0.3]] + dcs
    return _scene(means, logits, dcs)


def _flipped(oracle_mod, r, cam, flips, x=CX, y=CY):
    return oracle_mod.composite_pixel_flipped(r["proj"], r["sorted_vals"], r["ranges"], cam, x, y, flips)


def _stack_expect(n_taken, t0=1.0, c_front=None, a_front=None, skip_layer=None):
    """Closed form of the stack pixel when the walk takes layers [0, n_taken) (minus skip_layer),
    starting from transmittance t0 after an optional front Gaussian."""
    a = _opacity(A_STACK)
    cs = [_colour(d) for d in _stack_dcs()]
    C = np.zeros(3)
    T = 1.0
    if a_front is not None:
        C += a_front * c_front
        T = 1.0 - a_front
    T *= t0
    for k in range(n_taken):
        if k == skip_layer:
            continue
        C += a * T * cs[k]
        T *= 1.0 - a
    return C + T * np.float32(BG).astype(np.float64), T


def test_no_flip_equals_the_composite(oracle_mod):
    """With an empty flip list the helper is the composite of that pixel, bit for bit, on a
    640x480 image (tile index y/16 * tiles_x + x/16: a transposed index lands elsewhere)."""
    s = scenes.make_scene("100k", n=3000)
    cam = scenes.make_cameras("100k")[0]
    r = oracle_mod.render(s, cam)
    rng = np.random.default_rng(11)
    pix = [(int(x), int(y)) for x, y in zip(rng.integers(0, 640, 40), rng.integers(0, 480, 40))]
    pix += [(639, 5), (3, 479), (639, 479), (400, 100), (100, 400)]
    nonbg = 0
    for x, y in pix:
        rgb, T = _flipped(oracle_mod, r, cam, [], x, y)
        np.testing.assert_array_equal(rgb, r["image"][y, x])
        assert T == r["final_T"][y, x]
        nonbg += T < 1.0
    assert nonbg >= 10     # the sample covers pixels with contributions


@pytest.mark.parametrize("o", [0.999 / 255, 0.9999 / 255])
def test_skip_flip_below_threshold_takes_the_gaussian(oracle_mod, o):
    """alpha just below 1/255: skipped, so the pixel is the background; inverting the skip
    gives alpha c + (1 - alpha) bg."""
    cam = _cam(BG)
    dc = [0.7, -0.3, 0.2]
    r = oracle_mod.render(_scene([[0, 0, 0]], [_logit(o)], [dc]), cam)
    bg = np.float32(BG).astype(np.float64)
    a = _opacity(o)
    assert a < 1.0 / 255
    rgb0, T0 = _flipped(oracle_mod, r, cam, [])
    np.testing.assert_array_equal(rgb0, bg)
    assert T0 == 1.0
    rgb, T = _flipped(oracle_mod, r, cam, [(0, oracle_mod.EV_SKIP)])
    np.testing.assert_allclose(rgb, a * _colour(dc) + (1 - a) * bg, rtol=1e-14)
    np.testing.assert_allclose(T, 1 - a, rtol=1e-15)


def test_skip_flip_above_threshold_drops_the_gaussian(oracle_mod):
    """alpha just above 1/255: taken; inverting the skip leaves the background, T = 1."""
    cam = _cam(BG)
    o = 1.001 / 255
    r = oracle_mod.render(_scene([[0, 0, 0]], [_logit(o)], [[0.7, -0.3, 0.2]]), cam)
    a = _opacity(o)
    rgb0, T0 = _flipped(oracle_mod, r, cam, [])
    np.testing.assert_allclose(T0, 1 - a, rtol=1e-15)
    rgb, T = _flipped(oracle_mod, r, cam, [(0, oracle_mod.EV_SKIP)])
    np.testing.assert_array_equal(rgb, np.float32(BG).astype(np.float64))
    assert T == 1.0


def test_stop_flip_at_the_crossing_takes_the_next_layer(oracle_mod):
    """T crosses 1e-4 at layer 3 (0-based): the walk stops there. Inverting that stop takes
    layer 4, whose own stop then ends the walk: T = (1 - a)^5."""
    cam = _cam(BG)
    r = oracle_mod.render(_stack_scene(), cam)
    assert r["n_contrib"][CY, CX] == 4
    rgb0, T0 = _flipped(oracle_mod, r, cam, [])
    e0, eT0 = _stack_expect(4)
    np.testing.assert_allclose(rgb0, e0, rtol=1e-13)
    np.testing.assert_allclose(T0, eT0, rtol=1e-12)
    rgb, T = _flipped(oracle_mod, r, cam, [(3, oracle_mod.EV_STOP)])
    e, eT = _stack_expect(5)
    np.testing.assert_allclose(rgb, e, rtol=1e-13)
    np.testing.assert_allclose(T, eT, rtol=1e-12)
    # a stop flip moves the pixel by about T times a colour difference (here ~1e-6), far
    # below the image tolerance but far above the closed forms' rounding
    assert abs(rgb - rgb0).max() > 1e-7 and T < T0


def test_stop_flip_before_the_crossing_ends_the_walk(oracle_mod):
    """Inverting the (not taken) stop at layer 2, where T = 1.25e-4, ends the walk there."""
    cam = _cam(BG)
    r = oracle_mod.render(_stack_scene(), cam)
    rgb, T = _flipped(oracle_mod, r, cam, [(2, oracle_mod.EV_STOP)])
    e, eT = _stack_expect(3)
    np.testing.assert_allclose(rgb, e, rtol=1e-13)
    np.testing.assert_allclose(T, eT, rtol=1e-12)


def test_skip_flip_inside_the_stack(oracle_mod):
    """Inverting the skip of layer 1 (alpha = 0.95, far above 1/255) drops it: layers 0, 2, 3, 4
    are taken and the stop comes at layer 4."""
    cam = _cam(BG)
    r = oracle_mod.render(_stack_scene(), cam)
    rgb, T = _flipped(oracle_mod, r, cam, [(1, oracle_mod.EV_SKIP)])
    e, eT = _stack_expect(5, skip_layer=1)
    np.testing.assert_allclose(rgb, e, rtol=1e-13)
    np.testing.assert_allclose(T, eT, rtol=1e-12)


def test_two_flips_closed_form(oracle_mod):
    """A front Gaussian with alpha just below 1/255 (list position 0) before the stack
    (positions 1..10). Inverting its skip and the stop at position 4 (stack layer 3) gives
    a0 c0 + (1 - a0) sum_{k<5} a (1-a)^k c_k + (1 - a0)(1 - a)^5 bg; the order of the flips
    in the list does not matter, and each flip alone gives its own closed form."""
    cam = _cam(BG)
    o0 = 0.999 / 255
    r = oracle_mod.render(_stack_scene(front_o=o0), cam)
    a0 = _opacity(o0)
    c0 = _colour([0.6, -0.1, 0.3])
    S, P = oracle_mod.EV_SKIP, oracle_mod.EV_STOP
    cases = {
        (): _stack_expect(4),
        ((0, S),): _stack_expect(4, c_front=c0, a_front=a0),
        ((4, P),): _stack_expect(5),
        ((0, S), (4, P)): _stack_expect(5, c_front=c0, a_front=a0),
        ((4, P), (0, S)): _stack_expect(5, c_front=c0, a_front=a0),
    }
    for flips, (e, eT) in cases.items():
        rgb, T = _flipped(oracle_mod, r, cam, list(flips))
        np.testing.assert_allclose(rgb, e, rtol=1e-13, err_msg=str(flips))
        np.testing.assert_allclose(T, eT, rtol=1e-12, err_msg=str(flips))


def test_flips_the_walk_never_takes_change_nothing(oracle_mod):
    """A stop flip at a skipped entry (its stop is never evaluated), flips past the stop and
    flips past the end of the list leave the pixel as it is."""
    cam = _cam(BG)
    S, P = oracle_mod.EV_SKIP, oracle_mod.EV_STOP
    r1 = oracle_mod.render(_scene([[0, 0, 0]], [_logit(0.999 / 255)], [[0.7, -0.3, 0.2]]), cam)
    base1 = _flipped(oracle_mod, r1, cam, [])
    for flips in ([(0, P)], [(1, S)], [(5, P), (9, S)]):
        rgb, T = _flipped(oracle_mod, r1, cam, flips)
        np.testing.assert_array_equal(rgb, base1[0])
        assert T == base1[1]
    r2 = oracle_mod.render(_stack_scene(), cam)
    base2 = _flipped(oracle_mod, r2, cam, [])
    for flips in ([(5, S)], [(7, P)], [(4, P), (8, S)], [(50, S)], [(12, P), (60, S)]):
        rgb, T = _flipped(oracle_mod, r2, cam, flips)
        np.testing.assert_array_equal(rgb, base2[0], err_msg=str(flips))
        assert T == base2[1]
