"""Comparison helpers for the GPU-vs-oracle parity tests.

Image rule (pixel tolerance 1e-4 per channel, fp32 GPU against the fp64
oracle): a pixel passes if it is within tolerance of the oracle's composite,
or -- where the oracle saw an alpha within a relative band of 1/255 or a
transmittance within the band of 1e-4 -- within tolerance of the oracle's
composite with one or two of those decisions inverted. Both decisions are
correct results of the method in finite precision; such pixels are counted
and reported.
"""
from __future__ import annotations

import itertools

import numpy as np

TOL = 1e-4
BAND = 2e-3      # relative band around the 1/255 and 1e-4 thresholds
MAX_EV = 16


def oracle_render(oracle, scene, cam):
    return oracle.render(scene, cam, band=BAND, max_ev=MAX_EV)


def check_image(oracle, ref, cam, image, final_T=None, n_contrib=None, tol=TOL, max_report=5):
    """Returns a stats dict; stats['unexplained'] lists pixels that fail."""
    image = np.asarray(image, np.float64)
    err = np.abs(image - ref["image"]).max(-1)
    bad = np.argwhere(err > tol)
    flipped = np.zeros(err.shape, bool)
    unexplained = []
    proj, sv, rg = ref["proj"], ref["sorted_vals"], ref["ranges"]
    for (y, x) in bad:
        nev = int(min(ref["n_events"][y, x], MAX_EV))
        evs = [(int(ref["ev_pos"][y, x, i]), int(ref["ev_type"][y, x, i])) for i in range(nev)]
        ok = False
        for k in (1, 2):
            for comb in itertools.combinations(evs, k):
                rgb, _ = oracle.composite_pixel_flipped(proj, sv, rg, cam, int(x), int(y), list(comb))
                if np.abs(rgb - image[y, x]).max() <= tol:
                    ok = True
                    break
            if ok:
                break
        if ok:
            flipped[y, x] = True
        else:
            unexplained.append((int(y), int(x), float(err[y, x]), nev))
    quiet = ref["n_events"] == 0     # pixels with no decision near a threshold
    stats = {"max_err": float(err.max()) if err.size else 0.0,
             "max_err_no_events": float(err[quiet].max()) if quiet.any() else 0.0,
             "max_err_unflipped": float(err[~flipped].max()) if (~flipped).any() else 0.0,
             "n_pixels": int(err.size), "n_flipped": int(flipped.sum()),
             "unexplained": unexplained[:max_report], "n_unexplained": len(unexplained)}
    if final_T is not None:
        dT = np.abs(np.asarray(final_T, np.float64) - ref["final_T"])
        stats["max_dT_unflipped"] = float(dT[~flipped].max()) if (~flipped).any() else 0.0
    if n_contrib is not None:
        nc = np.asarray(n_contrib).astype(np.int64)
        mism = (nc != ref["n_contrib"].astype(np.int64)) & ~flipped
        # a decision inside the band that did not change the colour beyond tol can still move n_contrib
        near = ref["n_events"] > 0
        stats["n_contrib_mismatch"] = int((mism & ~near).sum())
        stats["n_contrib_mismatch_near"] = int((mism & near).sum())
    return stats


def tile_lists_in_tile_order(vals, ranges):
    """The per-tile lists of a sorted array (vals[ranges[t, 0]:ranges[t, 1]] for tile t),
    concatenated in tile-id order, with their lengths. Checks that the lists tile [0, K)."""
    vals = np.asarray(vals).view(np.uint32)
    r = np.asarray(ranges).view(np.uint32).reshape(-1, 2).astype(np.int64)
    lens = np.maximum(r[:, 1] - r[:, 0], 0)
    nz = np.nonzero(lens)[0]
    by_start = nz[np.argsort(r[nz, 0], kind="stable")]
    ends = r[by_start, 0] + lens[by_start]
    assert len(by_start) == 0 or (r[by_start[0], 0] == 0 and np.array_equal(r[by_start[1:], 0], ends[:-1])), \
        "tile lists overlap or leave gaps"
    K = int(lens.sum())
    idx = np.repeat(r[:, 0] - np.concatenate(([0], np.cumsum(lens)[:-1])), lens) + np.arange(K)
    return vals[idx], lens


def assert_same_tile_lists(vals, ranges, ref_vals, ref_ranges):
    """Every tile's list equal (same Gaussians, same order), whatever the order of the lists
    in the array."""
    a, la = tile_lists_in_tile_order(vals, ranges)
    b, lb = tile_lists_in_tile_order(ref_vals, ref_ranges)
    np.testing.assert_array_equal(la, lb)
    np.testing.assert_array_equal(a, b)


def assert_image_parity(stats):
    assert stats["n_unexplained"] == 0, stats
    assert stats["max_err_unflipped"] <= TOL, stats
    if "n_contrib_mismatch" in stats:
        assert stats["n_contrib_mismatch"] == 0, stats
