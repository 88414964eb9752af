"""Pins of the oracle's Gaussian footprint (the splat variant of the NuRec
pages; reading: sigma = r_eff / 3 over the sphere's support, shifted to 0 at
the rim) against an independent restatement and finite differences.  No GPU.
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np

import closed_form as cf
from splat_rendering_gb300 import scenes
from test_oracle_pins import _check_fd, _fd_scene, _render


def _gauss(sc):
    return replace(sc, params=replace(sc.params, gaussian=True))


def test_gaussian_matches_independent_restatement(oracle_lib):
    """Image and hit lists against the cross-product brute force with the
    Gaussian weight written from sigma = r/3 (fp64 decisions)."""
    for seed, rot in ((6, 0.0), (7, 15.0)):
        sc = _gauss(scenes.random_scene(seed, 80, 36, 30, rot_deg=rot, rrange=(0.05, 0.5),
                                        shift=(0.1, 0.0, 0.2)))
        out = _render(oracle_lib, sc, fp64=True)
        ref, hits = cf.render(sc.pos, sc.radius, sc.opacity, sc.features, sc.cameras[0],
                              sc.params, sc.bg, gaussian=True)
        assert np.abs(out["image"] - ref).max() < 1e-12
        assert (out["nhits"] == np.array([[len(h) for h in row] for row in hits])).all()


def test_gaussian_keeps_the_decisions(oracle_lib):
    """Only the distance factor changes: hit lists, tracked ids and tile
    lists are the linear footprint's; the image is not."""
    sc = scenes.random_scene(8, 300, 48, 40, rot_deg=7, rrange=(0.02, 0.4))
    a = _render(oracle_lib, sc)
    b = _render(oracle_lib, _gauss(sc))
    assert np.array_equal(a["ids"], b["ids"]) and np.array_equal(a["nhits"], b["nhits"])
    assert np.abs(a["image"] - b["image"]).max() > 1e-3


def test_gaussian_gradients_match_central_differences(oracle_lib):
    """Analytic gradients of the Gaussian footprint for every parameter family,
    including the kappa floor branch, against central finite differences."""
    sc = _gauss(_fd_scene(seed=9))
    out = _render(oracle_lib, sc, fp64=True, grad_image=sc.grad_images[0])
    assert out["nhits"].max() < sc.params.n_track
    rng = np.random.default_rng(1)
    sph = rng.choice(sc.n, 10, replace=False).tolist() + [0, 1]
    bad = []
    bad += _check_fd(oracle_lib, sc, out["grad_pos"], "pos",
                     [(i, k) for i in sph for k in range(3)], 1e-6)
    bad += _check_fd(oracle_lib, sc, out["grad_radius"], "radius", [(i,) for i in sph], 1e-6)
    bad += _check_fd(oracle_lib, sc, out["grad_opacity"], "opacity", [(i,) for i in sph], 1e-6)
    bad += _check_fd(oracle_lib, sc, out["grad_features"], "features",
                     [(i, k) for i in sph for k in range(2)], 1e-5)
    gc = out["grad_cam"]
    bad += _check_fd(oracle_lib, sc, gc[:9], "R", list(range(9)), 1e-7)
    bad += _check_fd(oracle_lib, sc, gc[9:12], "t", list(range(3)), 1e-7)
    for j, name in enumerate(("fx", "fy", "cx", "cy")):
        bad += _check_fd(oracle_lib, sc, float(gc[12 + j]), name, [0], 1e-5)
    assert not bad, bad
    assert np.abs(out["grad_pos"][:4]).max() > 0
