"""Orthographic camera (Pulsar Sec. B.1.1): CUDA path vs the CPU oracle
through the C ABI, on seeded inputs.

Bit-exact: per-sphere fp32 decisions, tile lists, tracked ids, hit counts.
Within tolerance: image, stabiliser and normaliser, gradients (the same
bars as the pinhole parity tests).
"""
from __future__ import annotations

import numpy as np
import pytest

import gpu_helpers as gh
from splat_rendering_gb300 import scenes
from test_gpu_parity import _check_lists, _oracle_all

pytestmark = pytest.mark.gpu

ORTHO = {
    # f in pixels per world unit; spheres fill the image's box
    "ortho_tiny": dict(seed=81, n=1000, width=64, height=64, f=28.0, rrange=(0.01, 0.1)),
    # ragged image, rotated and translated camera, fx != fy, off-centre principal point
    "ortho_ragged": dict(seed=82, n=3000, width=77, height=45, f=30.0, fy=36.0, cx=35.3,
                         cy=20.1, rot_deg=25, shift=(0.2, -0.1, 0.3), rrange=(0.005, 0.4)),
    # radii below the kappa floor (0.75 / f_min): the 1/f_min branch everywhere
    "ortho_floor": dict(seed=83, n=2000, width=60, height=52, f=20.0, fy=23.0,
                        rrange=(0.001, 0.03), geom_cutoff=False),
    # big spheres: tile lists longer than one warp's and one block's sort
    "ortho_long_lists": dict(seed=84, n=12000, width=64, height=64, f=24.0,
                             rrange=(0.4, 1.3), zrange=(2.5, 6.5), spread=1.4),
    "ortho_wide_payload": dict(seed=85, n=600, width=40, height=33, f=14.0, channels=19,
                               n_track=11, rrange=(0.05, 0.5)),
}


@pytest.mark.parametrize("case", sorted(ORTHO))
def test_ortho_cases(oracle_lib, case):
    sc = scenes.random_scene(orthographic=True, **ORTHO[case])
    o, d, offs, ids = _oracle_all(oracle_lib, sc)
    g = gh.run_gpu(sc, max_pairs=len(ids) + 64)
    assert g["code"] == 0
    assert g["n_pairs"] == len(ids)
    assert g["hits"] == o["hits"]
    gh.assert_decisions_equal(g, d)
    _check_lists(g, offs, ids)
    gh.compare_frame(g, o, case)
    if case == "ortho_long_lists":
        assert np.diff(offs).max() > 2048
    if case == "ortho_floor":
        assert (d["floor"][d["keep"] == 1] == 1).mean() > 0.5


def test_ortho_medium_frame(oracle_lib):
    """100,000 spheres on a 512 x 512 orthographic frame, rotated camera."""
    sc = scenes.random_scene(86, 100_000, 512, 512, f=100.0, rot_deg=8, zrange=(2.0, 10.0),
                             znear=1.0, zfar=11.0, rrange=(0.002, 0.05), orange=(0.05, 1.0),
                             orthographic=True)
    o, d, offs, ids = _oracle_all(oracle_lib, sc)
    g = gh.run_gpu(sc, max_pairs=len(ids) + 1024)
    assert g["code"] == 0 and g["n_pairs"] == len(ids) and g["hits"] == o["hits"]
    gh.assert_decisions_equal(g, d)
    _check_lists(g, offs, ids)
    gh.compare_frame(g, o, "ortho medium")


def test_ortho_and_pinhole_share_a_context(oracle_lib):
    """One context renders an orthographic frame, then a pinhole frame, then
    the orthographic one again; each matches the oracle."""
    ortho = scenes.random_scene(87, 900, 48, 40, f=18.0, orthographic=True, rrange=(0.02, 0.3))
    pin = scenes.random_scene(87, 900, 48, 40, rrange=(0.02, 0.3))
    from splat_rendering_gb300 import pulsar as pl
    r = pl.Renderer(max_spheres=900, max_pairs=1 << 16, max_width=48, max_height=40,
                    max_channels=3, max_track=5)
    for sc in (ortho, pin, ortho):
        o, d, offs, ids = _oracle_all(oracle_lib, sc)
        g = gh.run_gpu(sc, renderer=r)
        assert g["code"] == 0
        gh.assert_decisions_equal(g, d)
        _check_lists(g, offs, ids)
        gh.compare_frame(g, o, f"shared context {sc.cameras[0].orthographic}")
    r.close()


def test_ortho_headline_full_frame(oracle_lib):
    """The headline sizes with an orthographic camera (1M spheres, 1024 x 1024,
    the workload `bench.py --scene headline_ortho` times): decisions, tile
    lists, image and gradients over the full frame."""
    sc = scenes.make("headline_ortho")
    o, d, offs, ids = _oracle_all(oracle_lib, sc)
    g = gh.run_gpu(sc, max_pairs=len(ids) + 1024)
    assert g["code"] == 0 and g["n_pairs"] == len(ids) and g["hits"] == o["hits"]
    gh.assert_decisions_equal(g, d)
    _check_lists(g, offs, ids)
    gh.compare_frame(g, o, "headline ortho")
