"""Gaussian footprint (PULSAR_FLAG_GAUSSIAN; the splat variant of the NuRec
pages): CUDA path vs the oracle through the C ABI.  Decisions and tile lists
bit-exact (the footprint changes none); image, buffers and gradients within
the plain path's tolerances."""
from __future__ import annotations

from dataclasses import replace

import pytest

import gpu_helpers as gh
from splat_rendering_gb300 import scenes
from test_gpu_parity import _check_lists, _oracle_all

pytestmark = pytest.mark.gpu

CASES = {
    "pinhole": dict(seed=111, n=3000, width=96, height=80, rot_deg=14, shift=(0.1, 0.2, -0.1),
                    rrange=(0.005, 0.4)),
    "orthographic": dict(seed=112, n=2500, width=80, height=70, f=28.0, orthographic=True,
                         rot_deg=9, rrange=(0.005, 0.3)),
    "sixteen_channels": dict(seed=113, n=2000, width=72, height=64, channels=16, n_track=8,
                             rrange=(0.01, 0.3)),
    "floor_no_cutoff": dict(seed=114, n=2000, width=64, height=64, geom_cutoff=False,
                            rrange=(0.001, 0.02)),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_gaussian_footprint(oracle_lib, case):
    sc = scenes.random_scene(**CASES[case])
    sc = replace(sc, params=replace(sc.params, gaussian=True))
    o, d, offs, ids = _oracle_all(oracle_lib, sc)
    g = gh.run_gpu(sc, max_pairs=len(ids) + 64)
    assert g["code"] == 0 and g["hits"] == o["hits"]
    gh.assert_decisions_equal(g, d)
    _check_lists(g, offs, ids)
    gh.compare_frame(g, o, f"gaussian {case}")


def test_gaussian_headline_full_frame(oracle_lib):
    sc = scenes.make("headline")
    sc = replace(sc, params=replace(sc.params, gaussian=True))
    o, d, offs, ids = _oracle_all(oracle_lib, sc)
    g = gh.run_gpu(sc, max_pairs=len(ids) + 1024)
    assert g["code"] == 0 and g["n_pairs"] == len(ids) and g["hits"] == o["hits"]
    _check_lists(g, offs, ids)
    gh.compare_frame(g, o, "gaussian headline")
