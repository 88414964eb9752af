"""Pins of the CPU oracle against facts fixed outside it (no GPU).

Each test names the passage of "Pulsar: Efficient Sphere-based Neural
Rendering" (paperlayer.ai summary of arXiv 2004.07484) or the mathematical
fact it checks.  A plausible slip in the oracle (a dropped term, a sign, a
swapped index, a wrong axis) fails at least one of them.
"""
from __future__ import annotations

import math
from dataclasses import replace

import numpy as np
import pytest

import closed_form as cf
from splat_rendering_gb300 import scenes


def _render(oracle_lib, sc, **kw):
    return oracle_lib.render(sc.pos, sc.radius, sc.opacity, sc.features, sc.cameras[0],
                             sc.params, sc.bg, **kw)


def _one_sphere(c, r, o, f, W=32, H=32, fx=40.0, fy=None, cx=None, cy=None, gamma=0.1,
                bg=None, C=None):
    C = len(f) if C is None else C
    cam = scenes._camera(np.eye(3), np.zeros(3), fx, W, H, 1.0, 9.0, fy=fy, cx=cx, cy=cy)
    p = scenes.Params(gamma=gamma, n_track=4, channels=C)
    return scenes.Scene("one", np.array([c], np.float32), np.array([r], np.float32),
                        np.array([o], np.float32), np.array([f], np.float32), [cam], p,
                        np.zeros(C, np.float32) if bg is None else np.asarray(bg, np.float32),
                        [np.ones((H, W, C), np.float32)])


# --------------------------------------------------------------- forward --
@pytest.mark.parametrize("fp64", [True, False])
def test_single_sphere_closed_form(oracle_lib, fp64):
    """One sphere: F = (w f + w_bg f_bg)/(w + w_bg), w = o d exp(o z~/gamma),
    d = 1 - rho/r, rho the ray-to-centre distance (Sec. 3.2, App. A)."""
    rng = np.random.default_rng(11)
    for _ in range(12):
        c = [rng.uniform(-1, 1), rng.uniform(-1, 1), rng.uniform(2, 8)]
        r = rng.uniform(0.05, 0.6)
        o = rng.uniform(0.05, 1.0)
        f = rng.uniform(-1, 1, 3)
        bg = rng.uniform(-1, 1, 3)
        gamma = rng.choice([0.05, 0.1, 1.0])
        sc = _one_sphere(c, r, o, f, fx=rng.uniform(20, 60), fy=rng.uniform(20, 60),
                         cx=rng.uniform(10, 22), cy=rng.uniform(10, 22), gamma=gamma, bg=bg)
        out = _render(oracle_lib, sc, fp64=fp64)
        ref, hits = cf.render(sc.pos, sc.radius, sc.opacity, sc.features, sc.cameras[0],
                              sc.params, sc.bg)
        tol = 1e-12 if fp64 else 5e-6   # fp32 decisions may differ at the silhouette only
        assert np.abs(out["image"] - ref).max() < tol
        nref = np.array([[len(h) for h in row] for row in hits])
        if fp64:
            assert (out["nhits"] == nref).all()
        else:
            assert (out["nhits"] != nref).sum() <= 2


def test_on_axis_sphere_values(oracle_lib):
    """Sphere on the optical axis, pixel rays symmetric about it: the four
    central pixels see rho = z sin(theta), theta the ray's angle to the axis."""
    z, r, o, gamma = 4.0, 0.5, 0.75, 0.5     # all exact in float32
    sc = _one_sphere([0, 0, z], r, o, [1.0], W=16, H=16, fx=16.0, gamma=gamma, C=1)
    out = _render(oracle_lib, sc, fp64=True)
    theta = math.atan(math.hypot(0.5, 0.5) / 16.0)
    rho = z * math.sin(theta)
    d = 1 - rho / r
    zt = (9.0 - z) / 8.0
    w = o * d * math.exp(o * zt / gamma)
    wbg = math.exp(1e-5 / gamma)
    F = w / (w + wbg)
    for (y, x) in [(7, 7), (7, 8), (8, 7), (8, 8)]:
        assert abs(out["image"][y, x, 0] - F) < 1e-14
    # stored normaliser in the shifted frame: W = (w + w_bg) exp(-m/gamma)
    m = max(1e-5, o * zt)
    assert abs(out["mg"][8, 8] - m / gamma) < 1e-14
    assert abs(out["wsum"][8, 8] - (w + wbg) * math.exp(-m / gamma)) < 1e-13


def test_partition_of_unity(oracle_lib):
    """Normalised blend (App. A): with one indicator channel per sphere plus a
    background channel, the channels of every pixel sum to one, each is a
    normalised weight in [0, 1]."""
    rng = np.random.default_rng(3)
    n = 7
    sc = scenes.random_scene(5, n, 24, 20, channels=n + 1, zrange=(2, 4), rrange=(0.2, 0.6))
    sc.features[:] = np.eye(n + 1, dtype=np.float32)[:n]
    sc.bg[:] = np.eye(n + 1, dtype=np.float32)[n]
    for fp64 in (True, False):
        out = _render(oracle_lib, sc, fp64=fp64)
        img = out["image"]
        assert np.abs(img.sum(-1) - 1.0).max() < 1e-13
        assert img.min() > -1e-6 and img.max() <= 1.0 + 1e-13
        # empty pixels are pure background
        empty = out["nhits"] == 0
        assert empty.any() and np.abs(img[empty][:, n] - 1.0).max() == 0.0


def test_opacity_zero_removes_sphere(oracle_lib):
    """Opacity scales the weight (Sec. 3.2): o = 0 gives the image of the
    scene without that sphere."""
    sc = scenes.random_scene(7, 30, 32, 32, zrange=(2, 5), rrange=(0.05, 0.3))
    base = _render(oracle_lib, sc)
    for j in (0, 5, 17):
        s2 = replace(sc, opacity=sc.opacity.copy())
        s2.opacity[j] = 0.0
        keep = np.arange(sc.n) != j
        s3 = replace(sc, pos=sc.pos[keep], radius=sc.radius[keep], opacity=sc.opacity[keep],
                     features=sc.features[keep])
        a, b = _render(oracle_lib, s2), _render(oracle_lib, s3)
        assert np.abs(a["image"] - b["image"]).max() < 1e-14
    assert base["hits"] > 0


def test_empty_and_background(oracle_lib):
    """No sphere, or every sphere culled: every pixel is the background."""
    sc = scenes.random_scene(1, 0, 17, 9)
    sc.bg[:] = [0.25, -1.0, 3.0]
    out = _render(oracle_lib, sc, grad_image=sc.grad_images[0])
    assert np.array_equal(out["image"], np.broadcast_to(sc.bg.astype(np.float64), (9, 17, 3)))
    assert (out["ids"] == -1).all() and out["hits"] == 0
    assert np.array_equal(out["grad_cam"], np.zeros(16))
    behind = scenes.random_scene(2, 20, 16, 16)
    behind.pos[:, 2] = -behind.pos[:, 2]           # all behind the camera
    out = _render(oracle_lib, behind)
    assert out["hits"] == 0


def test_permutation_invariance(oracle_lib):
    """The blend is commutative in sphere order (App. A): permuting the input
    leaves the image unchanged and maps tracked ids through the permutation."""
    sc = scenes.random_scene(9, 60, 40, 30, zrange=(2, 6), rrange=(0.05, 0.4), rot_deg=7,
                             shift=(0.1, -0.2, 0.3))
    perm = np.random.default_rng(0).permutation(sc.n)
    sp = replace(sc, pos=sc.pos[perm], radius=sc.radius[perm], opacity=sc.opacity[perm],
                 features=sc.features[perm])
    a = _render(oracle_lib, sc, grad_image=sc.grad_images[0])
    b = _render(oracle_lib, sp, grad_image=sc.grad_images[0])
    assert np.abs(a["image"] - b["image"]).max() < 1e-13
    ids_b = np.where(b["ids"] >= 0, perm[np.maximum(b["ids"], 0)], -1)
    assert np.array_equal(ids_b, a["ids"])
    for k in ("grad_pos", "grad_radius", "grad_opacity", "grad_features"):
        assert np.allclose(b[k], a[k][perm], rtol=1e-12, atol=1e-12)
    assert np.allclose(b["grad_cam"], a["grad_cam"], rtol=1e-11, atol=1e-11)


def test_gamma_limits(oracle_lib):
    """gamma -> infinity: the opacity*distance weighted mean with unit
    background weight; gamma -> 0: the hit with the largest o*z~ wins (a soft
    z-buffer), the textbook limits of the exp(o z~/gamma) depth factor."""
    sc = scenes.random_scene(4, 40, 32, 24, zrange=(2, 6), rrange=(0.1, 0.5))
    cam = sc.cameras[0]
    big = replace(sc, params=replace(sc.params, gamma=1e7))
    out = _render(oracle_lib, big, fp64=True)
    c = cf.camera_space(sc.pos, cam)
    r = cf.reff(sc.radius, c, cam, sc.params.kappa)
    q = cf.pixel_rays(cam)
    num = np.zeros((cam.height, cam.width, 3))
    den = np.ones((cam.height, cam.width))
    for i in range(sc.n):
        rho = cf.ray_distance(c[i], q)
        wgt = np.where(rho < r[i], sc.opacity[i] * (1 - rho / r[i]), 0.0)
        num += wgt[..., None] * sc.features[i]
        den += wgt
    assert np.abs(out["image"] - num / den[..., None]).max() < 1e-6
    small = replace(sc, params=replace(sc.params, gamma=1e-3, n_track=64))
    out = _render(oracle_lib, small, fp64=True)
    zt = (cam.zfar - c[:, 2]) / (cam.zfar - cam.znear)
    oz = sc.opacity.astype(np.float64) * zt
    checked = 0
    for y in range(cam.height):
        for x in range(cam.width):
            ids = [i for i in out["ids"][y, x] if i >= 0]
            if len(ids) < 2:
                continue
            v = sorted(oz[ids])
            best = ids[int(np.argmax(oz[ids]))]
            dbest = 1 - cf.ray_distance(c[best], q[y:y + 1, x:x + 1])[0, 0] / r[best]
            if v[-1] - v[-2] > 0.03 and dbest > 0.2:
                assert np.abs(out["image"][y, x] - sc.features[best]).max() < 1e-5
                checked += 1
    assert checked > 10


@pytest.mark.parametrize("seed,rot,fy", [(21, 0.0, None), (22, 12.0, 47.0), (23, 25.0, 70.0)])
def test_fp64_decisions_match_independent_brute_force(oracle_lib, seed, rot, fy):
    """fp64-decision oracle == independent cross-product brute force: same
    hit sets in (key, id) order, same image."""
    sc = scenes.random_scene(seed, 50, 36, 28, rot_deg=rot, fy=fy, shift=(0.2, 0.1, -0.3),
                             zrange=(2, 6), rrange=(0.03, 0.4))
    sc.params.n_track = 64
    out = _render(oracle_lib, sc, fp64=True, brute=True)
    ref, hits = cf.render(sc.pos, sc.radius, sc.opacity, sc.features, sc.cameras[0],
                          sc.params, sc.bg)
    assert np.abs(out["image"] - ref).max() < 1e-12
    for y in range(sc.cameras[0].height):
        for x in range(sc.cameras[0].width):
            got = [i for i in out["ids"][y, x] if i >= 0]
            assert got == hits[y][x]


@pytest.mark.parametrize("fp64", [True, False])
def test_brute_equals_culled(oracle_lib, fp64):
    """Tile culling (Sec. B.1.2) is exact: brute force over all spheres and the
    16x16-tile candidate lists give identical hit lists and values."""
    sc = scenes.random_scene(31, 300, 70, 45, rot_deg=9, zrange=(2, 6), rrange=(0.01, 0.3),
                             spread=1.3)
    a = _render(oracle_lib, sc, fp64=fp64, grad_image=sc.grad_images[0])
    b = _render(oracle_lib, sc, fp64=fp64, brute=True, grad_image=sc.grad_images[0])
    for k in ("image", "mg", "wsum", "ids", "nhits", "grad_pos", "grad_cam"):
        assert np.array_equal(a[k], b[k]), k


def test_fp32_decisions_track_fp64(oracle_lib):
    """The fp32 decision sequence is a faithful rounding of the definition:
    projected centre within 1e-9 relative, r_eff and key within one ulp,
    rectangle within one pixel, hit sets equal except in the rounding band."""
    sc = scenes.medium()
    cam = sc.cameras[0]
    sub = slice(0, 20000)
    d32 = oracle_lib.project(sc.pos[sub], sc.radius[sub], sc.opacity[sub], cam, sc.params)
    c = cf.camera_space(sc.pos[sub], cam)
    u = cam.cx + cam.fx * c[:, 0] / c[:, 2]
    v = cam.cy + cam.fy * c[:, 1] / c[:, 2]
    k = d32["keep"] == 1
    uv = d32["uv"].astype(np.float64)
    assert np.abs((uv[k, 0] + uv[k, 1]) - u[k]).max() < 1e-9 * np.abs(u[k]).max()
    assert np.abs((uv[k, 2] + uv[k, 3]) - v[k]).max() < 1e-9 * np.abs(v[k]).max()
    r = cf.reff(sc.radius[sub], c, cam, sc.params.kappa)
    assert (np.abs(d32["reff"][k] - r[k]) <= 2 * np.spacing(d32["reff"][k])).all()
    key = c[:, 2] - r
    assert (np.abs(d32["key"][k] - key[k]) <= 4 * np.spacing(d32["key"][k]) + 1e-6).all()
    # rectangle vs trigonometric tangent bounds
    bad = 0
    for i in np.nonzero(k)[0][:3000]:
        umin, umax = cf.tangent_bounds(c[i, 0], c[i, 2], r[i], cam.fx, cam.cx)
        lo = max(0, math.ceil(umin - 0.5))
        hi = min(cam.width - 1, math.floor(umax - 0.5))
        bad += abs(d32["rect"][i, 0] - lo) > 1 or abs(d32["rect"][i, 1] - hi) > 1
    assert bad == 0
    # hit sets: fp32 vs fp64 decisions on a 96x96 window
    win = (200, 200, 296, 296)
    a = oracle_lib.render(sc.pos, sc.radius, sc.opacity, sc.features, cam, sc.params, sc.bg,
                          window=win)
    b = oracle_lib.render(sc.pos, sc.radius, sc.opacity, sc.features, cam, sc.params, sc.bg,
                          window=win, fp64=True)
    assert (a["nhits"] != b["nhits"]).mean() < 1e-3
    assert np.abs(a["image"] - b["image"]).max() < 1e-5


def test_every_sphere_gets_a_pixel(oracle_lib):
    """Sec. B.1.1: every sphere is rendered on at least one pixel.  With the
    kappa = 0.75 px radius floor, every kept sphere whose projected centre
    lies inside the pixel-centre hull hits at least one pixel."""
    for sc, sub in ((scenes.tiny(), slice(None)), (scenes.medium(), slice(0, 30000))):
        cam = sc.cameras[0]
        d = oracle_lib.project(sc.pos[sub], sc.radius[sub], sc.opacity[sub], cam, sc.params)
        p = replace(sc.params, n_track=96)
        out = oracle_lib.render(sc.pos[sub], sc.radius[sub], sc.opacity[sub],
                                sc.features[sub], cam, p, sc.bg)
        assert out["nhits"].max() < 96
        seen = np.zeros(len(d["keep"]), bool)
        ids = out["ids"].reshape(-1)
        seen[ids[ids >= 0]] = True
        uv = d["uv"].astype(np.float64)
        u, v = uv[:, 0] + uv[:, 1], uv[:, 2] + uv[:, 3]
        inside = (d["keep"] == 1) & (u > 0.5) & (u < cam.width - 0.5) & (v > 0.5) & \
                 (v < cam.height - 0.5)
        assert inside.sum() > 0.5 * len(u[sub] if isinstance(sub, slice) else u)
        assert seen[inside].all()


def test_tile_lists_consistent_with_pixel_hits(oracle_lib):
    """Candidates are sorted by earliest possible intersection (Sec. 3.2,
    B.1.1): each pixel's hits appear in its tile's list in the same order,
    and the list holds exactly the spheres whose rectangle meets the tile."""
    sc = scenes.random_scene(41, 400, 80, 50, rot_deg=5, zrange=(2, 6), rrange=(0.01, 0.3))
    cam = sc.cameras[0]
    offs, ids = oracle_lib.tile_lists(sc.pos, sc.radius, sc.opacity, cam, sc.params)
    d = oracle_lib.project(sc.pos, sc.radius, sc.opacity, cam, sc.params)
    assert offs[-1] == d["ntiles"].sum()
    p = replace(sc.params, n_track=64)
    out = oracle_lib.render(sc.pos, sc.radius, sc.opacity, sc.features, cam, p, sc.bg)
    tx = (cam.width + 15) // 16
    for t in range(len(offs) - 1):
        lst = ids[offs[t]:offs[t + 1]]
        keys = d["key"][lst]
        assert (np.diff(keys) >= 0).all()
        ty_, tx_ = divmod(t, tx)
        rect = d["rect"]
        exp = np.nonzero((d["keep"] == 1) & (rect[:, 0] // 16 <= tx_) & (rect[:, 1] // 16 >= tx_) &
                         (rect[:, 2] // 16 <= ty_) & (rect[:, 3] // 16 >= ty_))[0]
        assert sorted(lst.tolist()) == exp.tolist()
        pos_in = {int(s): k for k, s in enumerate(lst)}
        for y in range(ty_ * 16, min(cam.height, ty_ * 16 + 16)):
            for x in range(tx_ * 16, min(cam.width, tx_ * 16 + 16)):
                h = [int(i) for i in out["ids"][y, x] if i >= 0]
                order = [pos_in[i] for i in h]
                assert order == sorted(order)


# -------------------------------------------------------------- backward --
def _fd_scene(seed=5, cutoff=False):
    sc = scenes.random_scene(seed, 24, 30, 26, channels=2, n_track=64, f=34.0, fy=38.0,
                             cx=14.3, cy=12.8, rot_deg=11.0, shift=(0.15, -0.1, 0.2),
                             zrange=(2.0, 5.0), rrange=(0.08, 0.5), geom_cutoff=cutoff)
    # a few spheres on the kappa floor so its branch is exercised too
    sc.radius[:4] = 0.01
    return sc


def _loss(oracle_lib, sc, pos, rad, opa, feat, cam):
    out = oracle_lib.render(pos, rad, opa, feat, cam, sc.params, sc.bg, fp64=True)
    return float((out["image"] * sc.grad_images[0].astype(np.float64)).sum())


def _fd(oracle_lib, sc, which, idx, h):
    cam = sc.cameras[0]
    vals = []
    for sgn in (1, -1):
        pos = sc.pos.astype(np.float64)
        rad = sc.radius.astype(np.float64)
        opa = sc.opacity.astype(np.float64)
        feat = sc.features.astype(np.float64)
        cm = replace(cam, R=cam.R.astype(np.float64), t=cam.t.astype(np.float64))
        if which == "pos":
            pos[idx] += sgn * h
        elif which == "radius":
            rad[idx] += sgn * h
        elif which == "opacity":
            opa[idx] += sgn * h
        elif which == "features":
            feat[idx] += sgn * h
        elif which == "R":
            cm.R[idx] += sgn * h
        elif which == "t":
            cm.t[idx] += sgn * h
        else:
            setattr(cm, which, getattr(cm, which) + sgn * h)
        vals.append(_loss(oracle_lib, sc, pos, rad, opa, feat, cm))
    return (vals[0] - vals[1]) / (2 * h)


def _check_fd(oracle_lib, sc, g, which, idxs, h):
    bad = []
    for idx in idxs:
        a = g[idx] if not isinstance(g, float) else g
        f1 = _fd(oracle_lib, sc, which, idx, h)
        f2 = _fd(oracle_lib, sc, which, idx, h / 4)
        if abs(f1 - f2) > 1e-4 * (abs(f1) + 1):     # a kink within the step: skip
            continue
        if abs(a - f2) > 2e-5 * (abs(f2) + 1):
            bad.append((which, idx, a, f2))
    return bad


def test_gradients_match_central_differences(oracle_lib):
    """Analytic gradients (Sec. B.2) of L = sum <G, F> agree with central finite
    differences of the fp64-decision oracle for every parameter family, with
    n_track above the depth complexity and the geometry cutoff off."""
    sc = _fd_scene()
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
    # the floor branch really is exercised and carries a position gradient
    d = oracle_lib.project(sc.pos, sc.radius, sc.opacity, sc.cameras[0], sc.params)
    assert d["floor"][:4].all() and np.abs(out["grad_pos"][:4]).max() > 0


def test_truncation_to_first_n_track(oracle_lib):
    """Only the first n_track hits of a pixel receive gradients (Sec. 2,
    B.1.3): with n_track = 1 a sphere's gradient comes only from pixels where
    it is the front-most hit; the image does not depend on n_track."""
    sc = _fd_scene(seed=8)
    G = sc.grad_images[0]
    full = _render(oracle_lib, sc, fp64=True, grad_image=G)
    one = _render(oracle_lib, replace(sc, params=replace(sc.params, n_track=1)), fp64=True,
                  grad_image=G)
    assert np.array_equal(full["image"], one["image"])
    front = set(int(i) for i in one["ids"][..., 0].reshape(-1) if i >= 0)
    for i in range(sc.n):
        if i not in front:
            assert one["grad_opacity"][i] == 0 and not one["grad_pos"][i].any()
    # pixels whose only hit is tracked agree between the two runs: isolate one sphere
    only = [i for i in front if np.count_nonzero(full["ids"] == i) ==
            np.count_nonzero(one["ids"][..., 0] == i) and
            all((full["ids"][full["ids"][..., 0] == i][:, 1:] == -1).all() for _ in [0])]
    for i in only:
        assert np.isclose(full["grad_opacity"][i], one["grad_opacity"][i], rtol=1e-12, atol=1e-14)


def test_geometry_cutoff(oracle_lib):
    """Sec. 6 / App. A: spheres projecting to at most ~3 px get no position or
    radius gradient (and no share of the camera gradient); opacity and feature
    gradients are unaffected."""
    sc = scenes.random_scene(12, 80, 48, 40, zrange=(2, 6), rrange=(0.005, 0.2))
    on = _render(oracle_lib, sc, grad_image=sc.grad_images[0])
    off = _render(oracle_lib, replace(sc, params=replace(sc.params, geom_cutoff=False)),
                  grad_image=sc.grad_images[0])
    d = oracle_lib.project(sc.pos, sc.radius, sc.opacity, sc.cameras[0], sc.params)
    cut = d["cut"] == 1
    cam = sc.cameras[0]
    c = cf.camera_space(sc.pos, cam)
    area = math.pi * (min(cam.fx, cam.fy) * sc.radius.astype(np.float64) / c[:, 2]) ** 2
    kept = d["keep"] == 1
    assert (cut[kept] == (area[kept] <= 3.0)).all()
    assert cut.sum() > 5 and (~cut & kept).sum() > 5
    assert not on["grad_pos"][cut].any() and not on["grad_radius"][cut].any()
    touched = cut & (np.abs(off["grad_pos"]).sum(1) > 0)
    assert touched.sum() > 0
    assert np.array_equal(on["grad_opacity"], off["grad_opacity"])
    assert np.array_equal(on["grad_features"], off["grad_features"])
    assert np.allclose(on["grad_pos"][~cut], off["grad_pos"][~cut], rtol=0, atol=0)


@pytest.mark.parametrize("cutoff", [True, False])
def test_rigid_motion_identities(oracle_lib, cutoff):
    """Moving every sphere and the camera together leaves the image unchanged,
    so the gradients satisfy  sum_j dL/dp_j = R^T dL/dt  (translation) and
    sum_j dL/dp_j x p_j = vee(R^T dL/dR - dL/dR^T R) (rotation) -- with the
    geometry cutoff on as well, since it drops a sphere's share everywhere."""
    sc = scenes.random_scene(14, 120, 48, 36, rot_deg=20, shift=(0.3, -0.2, 0.4),
                             zrange=(2, 6), rrange=(0.01, 0.3), geom_cutoff=cutoff)
    out = _render(oracle_lib, sc, grad_image=sc.grad_images[0])
    R = sc.cameras[0].R.astype(np.float64).reshape(3, 3)
    gR = out["grad_cam"][:9].reshape(3, 3)
    gt = out["grad_cam"][9:12]
    gp = out["grad_pos"]
    assert np.allclose(gp.sum(0), R.T @ gt, rtol=1e-10, atol=1e-9)
    # rotation: p -> p + Om p, R -> R - R Om for skew Om  =>  sum gp.(Om p) = <gR, R Om>
    p = sc.pos.astype(np.float64)
    for ax in range(3):
        Om = np.zeros((3, 3))
        i, j = [(1, 2), (2, 0), (0, 1)][ax]
        Om[i, j], Om[j, i] = -1.0, 1.0
        lhs = float((gp * (p @ Om.T)).sum())
        rhs = float((gR * (R @ Om)).sum())
        assert abs(lhs - rhs) < 1e-9 * (abs(lhs) + abs(rhs) + 1)
    assert np.abs(gp).max() > 0
