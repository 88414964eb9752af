"""Pins of the oracle's orthographic camera (Pulsar Sec. B.1.1: sphere
projections are bounded for orthogonal as well as pinhole cameras) against
facts fixed outside it: an independent world-space restatement of the
blend, finite differences, rigid-motion identities and the one-pixel floor.
No GPU.
"""
from __future__ import annotations

import math
from dataclasses import replace

import numpy as np
import pytest

import closed_form as cf
from splat_rendering_gb300 import scenes
from test_oracle_pins import _check_fd, _render


def _ortho_scene(seed, n=60, W=40, H=34, f=14.0, **kw):
    kw.setdefault("zrange", (2.0, 6.0))
    kw.setdefault("rrange", (0.03, 0.4))
    return scenes.random_scene(seed, n, W, H, f=f, orthographic=True, **kw)


@pytest.mark.parametrize("fp64", [True, False])
def test_ortho_matches_world_space_restatement(oracle_lib, fp64):
    """Image and hit lists equal the world-space brute force (distance to
    a ray along the viewing axis, un-shifted exponentials)."""
    for seed, rot in ((3, 0.0), (4, 17.0), (5, 40.0)):
        sc = _ortho_scene(seed, rot_deg=rot, shift=(0.2, -0.1, 0.3), fy=11.0, cx=18.3, cy=15.9)
        cam = sc.cameras[0]
        out = _render(oracle_lib, sc, fp64=fp64)
        ref, hits = cf.render_ortho(sc.pos, sc.radius, sc.opacity, sc.features, cam,
                                    sc.params, sc.bg)
        nref = np.array([[len(h) for h in row] for row in hits])
        if fp64:
            assert np.abs(out["image"] - ref).max() < 1e-12
            assert (out["nhits"] == nref).all()
            for y in range(cam.height):
                for x in range(cam.width):
                    assert [i for i in out["ids"][y, x] if i >= 0] == hits[y][x][:sc.params.n_track]
        else:
            # fp32 decisions: only pixels in a silhouette's rounding band may differ
            assert (out["nhits"] != nref).sum() <= 3
            same = out["nhits"] == nref
            assert np.abs(out["image"][same] - ref[same]).max() < 1e-5


def test_ortho_single_sphere_values(oracle_lib):
    """One sphere seen orthographically: rho at each pixel is the plain 2-D
    distance in world units, so F is known in closed form."""
    cam = scenes._camera(np.eye(3), np.zeros(3), 10.0, 32, 32, 1.0, 9.0, orthographic=True)
    p = scenes.Params(gamma=0.1, n_track=4, channels=1)
    c, r, o = (0.13, -0.21, 4.0), 0.9, 0.7
    sc = scenes.Scene("one", np.array([c], np.float32), np.array([r], np.float32),
                      np.array([o], np.float32), np.array([[2.0]], np.float32), [cam], p,
                      np.zeros(1, np.float32), [np.ones((32, 32, 1), np.float32)])
    out = _render(oracle_lib, sc, fp64=True)
    c32 = np.array(c, np.float32).astype(np.float64)
    zt = (9.0 - c32[2]) / 8.0
    o32 = float(np.float32(o))
    wbg = math.exp(1e-5 / 0.1)   # fp64 decisions: the parameters as given
    for y in range(32):
        for x in range(32):
            X = (x + 0.5 - 16.0) / 10.0
            Y = (y + 0.5 - 16.0) / 10.0
            rho = math.hypot(c32[0] - X, c32[1] - Y)
            r32 = float(np.float32(r))
            if rho < r32:
                w = o32 * (1 - rho / r32) * math.exp(o32 * zt / 0.1)
                want = w * 2.0 / (w + wbg)
            else:
                want = 0.0
            assert abs(out["image"][y, x, 0] - want) < 1e-12


def test_ortho_rectangle_and_one_pixel_floor(oracle_lib):
    """Every hit pixel lies in the sphere's pixel rectangle, the rectangle is
    [ceil(u - f r - 1/2), floor(u + f r - 1/2)], and with kappa = 0.75 px
    every kept sphere whose centre projects into the image hits a pixel
    (Sec. B.1.1)."""
    sc = _ortho_scene(21, n=400, W=48, H=40, f=16.0, rrange=(0.001, 0.2), rot_deg=9.0)
    cam = sc.cameras[0]
    d = oracle_lib.project(sc.pos, sc.radius, sc.opacity, cam, sc.params, fp64=True)
    out = _render(oracle_lib, sc, fp64=True, brute=True)
    c = cf.camera_space(sc.pos, cam)
    reff = np.maximum(sc.radius.astype(np.float64), sc.params.kappa / min(cam.fx, cam.fy))
    u = cam.cx + cam.fx * c[:, 0]
    v = cam.cy + cam.fy * c[:, 1]
    kept = d["keep"] == 1
    for i in np.nonzero(kept)[0]:
        lo = max(0, math.ceil(u[i] - cam.fx * reff[i] - 0.5))
        hi = min(cam.width - 1, math.floor(u[i] + cam.fx * reff[i] - 0.5))
        assert (d["rect"][i, 0], d["rect"][i, 1]) == (lo, hi)
    assert d["floor"][kept].sum() > 20
    for i in np.nonzero(kept)[0]:
        ys, xs = np.nonzero((out["ids"] == i).any(-1))
        x0, x1, y0, y1 = d["rect"][i]
        assert ((xs >= x0) & (xs <= x1) & (ys >= y0) & (ys <= y1)).all()
    # one-pixel floor: centres inside the image always hit (n_track large enough)
    sc2 = replace(sc, params=replace(sc.params, n_track=64))
    out2 = _render(oracle_lib, sc2, fp64=True)
    inside = kept & (u >= 0) & (u < cam.width) & (v >= 0) & (v < cam.height)
    for i in np.nonzero(inside)[0]:
        assert (out2["ids"] == i).any(), i


@pytest.mark.parametrize("fp64", [True, False])
def test_ortho_brute_equals_culled(oracle_lib, fp64):
    """Tile culling is exact for the orthographic camera too."""
    sc = _ortho_scene(31, n=300, W=70, H=45, f=20.0, rot_deg=9.0, rrange=(0.01, 0.5))
    a = _render(oracle_lib, sc, fp64=fp64, grad_image=sc.grad_images[0])
    b = _render(oracle_lib, sc, fp64=fp64, brute=True, grad_image=sc.grad_images[0])
    for k in ("image", "mg", "wsum", "ids", "nhits", "grad_pos", "grad_cam"):
        assert np.array_equal(a[k], b[k]), k


def test_ortho_gradients_match_central_differences(oracle_lib):
    """Analytic orthographic gradients (position, radius, opacity, features,
    R, t and fx, fy, cx, cy, including the kappa floor's 1/f_min branch)
    agree with central finite differences of the fp64-decision oracle."""
    sc = _ortho_scene(5, n=24, W=30, H=26, f=9.0, fy=10.5, cx=14.3, cy=12.8, rot_deg=11.0,
                      shift=(0.15, -0.1, 0.2), zrange=(2.0, 5.0), rrange=(0.25, 0.9),
                      channels=2, n_track=64, geom_cutoff=False)
    sc.radius[:4] = 0.01
    out = _render(oracle_lib, sc, fp64=True, grad_image=sc.grad_images[0])
    assert out["nhits"].max() < sc.params.n_track
    rng = np.random.default_rng(0)
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
    d = oracle_lib.project(sc.pos, sc.radius, sc.opacity, sc.cameras[0], sc.params)
    assert d["floor"][:4].all()
    # the depth of a floor sphere moves nothing but z~: its position gradient has a z part
    assert np.abs(out["grad_pos"][:4]).max() > 0


@pytest.mark.parametrize("cutoff", [True, False])
def test_ortho_rigid_motion_identities(oracle_lib, cutoff):
    """Moving every sphere and the camera together leaves the image unchanged:
    sum_j dL/dp_j = R^T dL/dt and the rotation identity hold orthographically."""
    sc = _ortho_scene(14, n=120, W=48, H=36, f=15.0, rot_deg=20, shift=(0.3, -0.2, 0.4),
                      rrange=(0.01, 0.3), geom_cutoff=cutoff)
    out = _render(oracle_lib, sc, grad_image=sc.grad_images[0])
    R = sc.cameras[0].R.astype(np.float64).reshape(3, 3)
    gR = out["grad_cam"][:9].reshape(3, 3)
    gt = out["grad_cam"][9:12]
    gp = out["grad_pos"]
    assert np.allclose(gp.sum(0), R.T @ gt, rtol=1e-10, atol=1e-9)
    p = sc.pos.astype(np.float64)
    for ax in range(3):
        Om = np.zeros((3, 3))
        i, j = [(1, 2), (2, 0), (0, 1)][ax]
        Om[i, j], Om[j, i] = -1.0, 1.0
        lhs = float((gp * (p @ Om.T)).sum())
        rhs = float((gR * (R @ Om)).sum())
        assert abs(lhs - rhs) < 1e-9 * (abs(lhs) + abs(rhs) + 1)
    assert np.abs(gp).max() > 0


def test_ortho_geometry_cutoff_area(oracle_lib):
    """The cutoff area of an orthographic sphere is pi (f_min r)^2 px^2: no
    1/c.z, so it does not change with depth."""
    sc = _ortho_scene(12, n=80, W=48, H=40, f=12.0, rrange=(0.02, 0.4))
    d = oracle_lib.project(sc.pos, sc.radius, sc.opacity, sc.cameras[0], sc.params)
    cam = sc.cameras[0]
    area = math.pi * (min(cam.fx, cam.fy) * sc.radius.astype(np.float64)) ** 2
    kept = d["keep"] == 1
    assert (d["cut"][kept] == (area[kept] <= 3.0)).all()
    assert d["cut"][kept].sum() > 5 and (d["cut"][kept] == 0).sum() > 5
