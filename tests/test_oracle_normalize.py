"""The oracle's normalised gradients (Pulsar Sec. B.2: sphere gradients
averaged over the contributing pixels, camera gradients normalised by the
projected sphere area and 1e-3).

PARITY UNPINNED: the normalised quantities are not derivatives of anything,
so no finite difference or closed form outside the oracle fixes them.  These
tests only hold the oracle to its own stated reading -- the scale factors
relative to its (pinned) plain gradients -- so that the CUDA path has a
definite target.  No GPU.
"""
from __future__ import annotations

import math
from dataclasses import replace

import numpy as np

from splat_rendering_gb300 import scenes
from test_oracle_pins import _render


def _norm(sc):
    return replace(sc, params=replace(sc.params, normalize_grads=True))


def test_sphere_gradients_are_averaged_over_tracking_pixels(oracle_lib):
    sc = scenes.random_scene(41, 300, 60, 44, rot_deg=12, rrange=(0.02, 0.4))
    G = sc.grad_images[0]
    a = _render(oracle_lib, sc, grad_image=G)
    b = _render(oracle_lib, _norm(sc), grad_image=G)
    assert np.array_equal(a["image"], b["image"]) and np.array_equal(a["ids"], b["ids"])
    nj = np.bincount(a["ids"][a["ids"] >= 0].reshape(-1), minlength=sc.n).astype(np.float64)
    assert (nj > 1).sum() > 20 and (nj == 0).sum() > 0
    s = np.where(nj > 0, 1.0 / np.maximum(nj, 1), 1.0)
    np.testing.assert_allclose(b["grad_pos"], a["grad_pos"] * s[:, None], rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(b["grad_radius"], a["grad_radius"] * s, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(b["grad_opacity"], a["grad_opacity"] * s, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(b["grad_features"], a["grad_features"] * s[:, None], rtol=1e-12,
                               atol=1e-300)


def test_camera_share_scaled_by_area_and_1e3(oracle_lib):
    """One sphere at a time: the camera gradient is the plain one times
    1e-3 / (pi (f_min r_eff / c.z)^2), pinhole and orthographic."""
    for ortho, seed in ((False, 42), (True, 43)):
        base = scenes.random_scene(seed, 6, 40, 30, rrange=(0.05, 0.3), orthographic=ortho,
                                   f=(14.0 if ortho else None), rot_deg=10)
        cam = base.cameras[0]
        for j in range(base.n):
            sc = replace(base, pos=base.pos[j:j + 1], radius=base.radius[j:j + 1],
                         opacity=base.opacity[j:j + 1], features=base.features[j:j + 1])
            a = _render(oracle_lib, sc, grad_image=sc.grad_images[0])
            if not (a["ids"] >= 0).any():
                continue
            b = _render(oracle_lib, _norm(sc), grad_image=sc.grad_images[0])
            R = cam.R.astype(np.float64).reshape(3, 3)
            c = R @ sc.pos[0].astype(np.float64) + cam.t.astype(np.float64)
            fmin = min(cam.fx, cam.fy)
            r = float(sc.radius[0])
            reff = max(r, sc.params.kappa / fmin * (1.0 if ortho else c[2]))
            rz = reff if ortho else reff / c[2]
            A = math.pi * (fmin * rz) ** 2
            np.testing.assert_allclose(b["grad_cam"], a["grad_cam"] * 1e-3 / A, rtol=1e-6,
                                       atol=1e-300)
