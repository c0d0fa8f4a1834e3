"""Mutation check of the oracle pins (CPU): a plausible mistake planted in a
copy of the oracle -- a flipped sign, a transposed operand, a dropped factor,
a reversed tie-break, a wrong threshold -- must make at least one pin fail.

Each C mutation rewrites one source fragment of oracle/gs_oracle.c in a
temporary copy, builds it with the oracle's own flags and swaps it in for the
named pins only. The Python mutations rewrite one fragment of a function of
oracle/gs_grad.py the same way. Nothing here touches the CUDA path.
"""
import ctypes
import inspect
import os
import subprocess
import textwrap

import numpy as np
import pytest

import oracle
from oracle import gs_grad

import test_oracle_flip_pins as fpins
import test_oracle_grad_pins as gpins
import test_oracle_pins as pins

C_MUTATIONS = [
    ("band-1 SH sign", "Y[1] = -c1 * y;", "Y[1] = c1 * y;",
     [(pins.test_sh_printed_constants_signs_and_monomials, {})]),
    ("rotation entry sign (fp64)", "G[1] = 2 * (x * y - w * z);", "G[1] = 2 * (x * y + w * z);",
     [(pins.test_rotation_about_z_closed_form, {})]),
    ("camera rotation transposed in the EWA product", "mat_mul(WT, JT, WTJT, 3, 3, 2);",
     "mat_mul(Wm, JT, WTJT, 3, 3, 2);", [(pins.test_ewa_matches_finite_difference_jacobian, {})]),
    ("Jacobian sign", "double J[6] = {fx / z, 0.0, -fx * xc[0] / (z * z),",
     "double J[6] = {fx / z, 0.0, fx * xc[0] / (z * z),", [(pins.test_ewa_matches_finite_difference_jacobian, {})]),
    ("conic off-diagonal sign", "conic[3 * g + 1] = -b / det;", "conic[3 * g + 1] = b / det;",
     [(pins.test_conic_is_inverse_of_cov2d, {})]),
    ("transmittance update", "T = T * (1.0 - alpha);\n        used++;", "T = T * alpha;\n        used++;",
     [(pins.test_two_gaussians_front_to_back_closed_form, {})]),
    ("half dropped from the exponent", "double alpha = opacity[g] * exp(-0.5 * q);\n        if (alpha > OR_ALPHA_MAX)",
     "double alpha = opacity[g] * exp(-q);\n        if (alpha > OR_ALPHA_MAX)",
     [(pins.test_tiled_equals_untiled_brute_force, {})]),
    ("tie-break reversed", "if (a->val != b->val) return a->val < b->val ? -1 : 1;",
     "if (a->val != b->val) return a->val < b->val ? 1 : -1;", [(pins.test_sort_matches_stable_library_sort, {})]),
    ("rotation entry sign (decision program)", "G[1] = 2.0f * (xy - wz);", "G[1] = 2.0f * (xy + wz);",
     [(pins.test_decision_program_second_build, {"name": "100k", "n": 30000})]),
    ("no skip below 1/255", "int skip = alpha < OR_ALPHA_MIN;", "int skip = alpha < 0.0;",
     [(pins.test_skip_below_one_over_255, {})]),
    # the threshold-flip helper behind the GPU image check's "several results are correct" rule
    ("flip type ignored by the skip decision", "if (flip_pos[f] == j && flip_type[f] == OR_EV_SKIP) skip = !skip;",
     "if (flip_pos[f] == j) skip = !skip;",
     [(fpins.test_flips_the_walk_never_takes_change_nothing, {}),
      (fpins.test_stop_flip_at_the_crossing_takes_the_next_layer, {})]),
    ("stop flip one list position late", "if (flip_pos[f] == j && flip_type[f] == OR_EV_STOP) stop = !stop;",
     "if (flip_pos[f] == j + 1 && flip_type[f] == OR_EV_STOP) stop = !stop;",
     [(fpins.test_stop_flip_at_the_crossing_takes_the_next_layer, {}), (fpins.test_two_flips_closed_form, {})]),
    # (the wrong column stays inside the 640x480 tile grid: y / 16 < 30 < 40 tiles per row)
    ("flipped pixel's tile column taken from y", "const int64_t tile = (int64_t)(y / 16) * TX + (x / 16);",
     "const int64_t tile = (int64_t)(y / 16) * TX + (y / 16);", [(fpins.test_no_flip_equals_the_composite, {})]),
]


def _build_mutant(tmp_path, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gs_oracle.c")).read()
    assert src.count(old) >= 1, old
    path_c = tmp_path / "mutant.c"
    path_c.write_text(src.replace(old, new, 1))
    path_so = tmp_path / "mutant.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, str(path_c), "-o", str(path_so), "-lm"])
    lib = ctypes.CDLL(str(path_so))
    lib.or_scan.restype = ctypes.c_uint64
    lib.or_get_threads.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("label,old,new,catchers", C_MUTATIONS, ids=[m[0] for m in C_MUTATIONS])
def test_c_oracle_mutation_is_caught(tmp_path, monkeypatch, label, old, new, catchers):
    oracle.build()
    monkeypatch.setattr(oracle, "_lib", _build_mutant(tmp_path, old, new))
    for fn, kwargs in catchers:
        with pytest.raises(AssertionError):
            fn(oracle, **kwargs)


PY_MUTATIONS = [
    ("band-2 SH sign (gradient oracle)", "sh_basis_t", "k2 * x * y, k2 * y * z", "-k2 * x * y, k2 * y * z",
     gpins.test_sh_basis_equals_c_oracle),
    ("Jacobian sign (gradient oracle)", "preprocess_t", '-f["fx"] * x / (z * z)', 'f["fx"] * x / (z * z)',
     gpins.test_forward_equals_c_oracle_composite),
    ("inclusive transmittance (gradient oracle)", "composite_t",
     "Texcl = torch.cat([torch.ones((P, 1), dtype=torch.float64), Tincl[:, :-1]], dim=1)", "Texcl = Tincl",
     gpins.test_forward_equals_c_oracle_composite),
    ("off-diagonal not halved (2D)", "pre2d_t", "b = 0.5 * (covs[:, 0, 1] + covs[:, 1, 0])",
     "b = covs[:, 0, 1] + covs[:, 1, 0]", gpins.test_2d_dense_mode_is_the_pages_formula),
]


@pytest.mark.parametrize("label,func,old,new,catcher", PY_MUTATIONS, ids=[m[0] for m in PY_MUTATIONS])
def test_gradient_oracle_mutation_is_caught(monkeypatch, label, func, old, new, catcher):
    pytest.importorskip("torch")
    src = textwrap.dedent(inspect.getsource(getattr(gs_grad, func)))
    assert src.count(old) == 1, old
    ns = dict(vars(gs_grad))
    exec(compile(src.replace(old, new), f"<mutant {func}>", "exec"), ns)
    monkeypatch.setattr(gs_grad, func, ns[func])
    with pytest.raises(AssertionError):
        catcher()
