"""Pins of the oracle's per-entry error scales (no GPU).

Besides the gradients themselves the oracle reports, for every gradient
entry, two sums over the pixels that contribute to it (Pulsar Sec. B.2: a
sphere's gradient is a sum of per-pixel contributions through its tracked
hits):

* ``abs_*``  A = sum_p |c_p|, c_p = <G_p, dF_p/d theta> the pixel's
  contribution;
* ``sens_*`` S = sum_p sum_ch |d c_p / d F_p,ch|, how strongly the
  contribution depends on the image F that the backward takes as input.  For
  every parameter but the features c_p = s_p u_p with s_p = <G_p, f - F_p> / W_p
  and u_p = dw_p/d theta independent of F, so S = sum_p |c_p| ||G_p||_1 /
  |<G_p, f - F_p>|; the feature entries do not depend on F (S = 0).

The GPU parity tests widen the gradient tolerance with A and S, so a slip in
either would loosen every gradient check.  Here both are computed
independently: each pixel's contribution by central finite differences of the
closed-form single-sphere renderer (cross-product distance, un-shifted
exponentials), F from the same closed form.
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest

import closed_form as cf
from splat_rendering_gb300 import scenes


def _scene(c, r, o, f, W, H, fx, cx, cy, G, fy=None):
    # fy != fx by default: at fx == fy the kappa floor's f_min has a kink in fx
    fy = 1.1 * fx if fy is None else fy
    cam = scenes._camera(np.eye(3), np.zeros(3), fx, W, H, 1.0, 9.0, fy=fy, cx=cx, cy=cy)
    p = scenes.Params(n_track=4, channels=len(f), geom_cutoff=False)
    return scenes.Scene("one", np.array([c], np.float32), np.array([r], np.float32),
                        np.array([o], np.float32), np.array([f], np.float32), [cam], p,
                        np.zeros(len(f), np.float32), [np.asarray(G, np.float32)])


def _cf_image(sc, pos=None, radius=None, opacity=None, features=None, cam=None):
    img, _ = cf.render(sc.pos.astype(np.float64) if pos is None else pos,
                       sc.radius.astype(np.float64) if radius is None else radius,
                       sc.opacity.astype(np.float64) if opacity is None else opacity,
                       sc.features.astype(np.float64) if features is None else features,
                       sc.cameras[0] if cam is None else cam, sc.params, sc.bg)
    return img


def _cam64(cam):
    """The camera with float64 R and t, so perturbations are not rounded."""
    return replace(cam, R=np.asarray(cam.R, np.float64).copy(),
                   t=np.asarray(cam.t, np.float64).copy())


# (name, oracle key, index into the entry, perturbation of the closed-form inputs)
def _perturbers(sc):
    p0 = sc.pos.astype(np.float64)
    f0 = sc.features.astype(np.float64)
    cam = _cam64(sc.cameras[0])

    def pos(k):
        def g(h):
            p = p0.copy()
            p[0, k] += h
            return dict(pos=p)
        return g

    def feat(k):
        def g(h):
            f = f0.copy()
            f[0, k] += h
            return dict(features=f)
        return g

    def cam_field(name):
        def g(h):
            return dict(cam=replace(cam, **{name: getattr(cam, name) + h}))
        return g

    def cam_R(k):
        def g(h):
            R = cam.R.copy()
            R[k] += h
            return dict(cam=replace(cam, R=R))
        return g

    def cam_t(k):
        def g(h):
            t = cam.t.copy()
            t[k] += h
            return dict(cam=replace(cam, t=t))
        return g

    out = [("pos x", "grad_pos", (0, 0), pos(0)), ("pos y", "grad_pos", (0, 1), pos(1)),
           ("pos z", "grad_pos", (0, 2), pos(2)),
           ("radius", "grad_radius", (0,),
            lambda h: dict(radius=sc.radius.astype(np.float64) + h)),
           ("opacity", "grad_opacity", (0,),
            lambda h: dict(opacity=sc.opacity.astype(np.float64) + h))]
    out += [(f"feature {k}", "grad_features", (0, k), feat(k)) for k in range(sc.params.channels)]
    out += [(f"R{k}", "grad_cam", (k,), cam_R(k)) for k in (0, 2, 4, 5, 7)]
    out += [(f"t{k}", "grad_cam", (9 + k,), cam_t(k)) for k in range(3)]
    out += [(n, "grad_cam", (12 + k,), cam_field(n)) for k, n in enumerate(("fx", "fy", "cx", "cy"))]
    return out


def _independent_terms(sc, perturb, feature):
    """Per-pixel contributions by central differences and the two sums."""
    G = sc.grad_images[0].astype(np.float64)
    h = 1e-6
    dF = (_cf_image(sc, **perturb(h)) - _cf_image(sc, **perturb(-h))) / (2 * h)
    contrib = (G * dF).sum(-1)                              # [H,W]
    A = np.abs(contrib).sum()
    if feature:
        return contrib, A, 0.0, 0.0
    F = _cf_image(sc)
    f = sc.features[0].astype(np.float64)
    sdot = (G * (f - F)).sum(-1)
    mask = np.abs(contrib) > 0
    ratio = np.abs(G[mask]).sum(-1) / np.abs(sdot[mask])
    S = (np.abs(contrib[mask]) * ratio).sum()
    # the differences' noise (~1e-10 absolute per contribution) scaled like S
    return contrib, A, S, 1e-9 * ratio.sum()


def _check(oracle_lib, sc, expect_cancel=()):
    o = oracle_lib.render(sc.pos, sc.radius, sc.opacity, sc.features, sc.cameras[0], sc.params,
                          sc.bg, grad_image=sc.grad_images[0], fp64=True)
    assert o["nhits"].sum() > 0
    for name, key, idx, perturb in _perturbers(sc):
        feature = key == "grad_features"
        contrib, A, S, s_noise = _independent_terms(sc, perturb, feature)
        v, a, s = o[key][idx], o["abs_" + key][idx], o["sens_" + key][idx]
        # central differences (h = 1e-6) of values ~1: ~1e-10 absolute noise
        assert abs(v - contrib.sum()) <= 1e-6 * A + 1e-9, (name, v, contrib.sum())
        assert abs(a - A) <= 1e-6 * A + 1e-9, (name, a, A)
        assert abs(s - S) <= 1e-6 * S + s_noise, (name, s, S)
        if name in expect_cancel:
            # the contributions cancel: the value vanishes, A does not
            assert abs(v) <= 1e-9 * A and A > 1e-3, (name, v, A)
    return o


def test_one_pixel_abs_sum_is_the_magnitude(oracle_lib):
    """A single pixel and a single sphere: every entry is one contribution, so
    A = |value| exactly and S = |value| ||G||_1 / |<G, f - F>|."""
    rng = np.random.default_rng(5)
    for trial in range(4):
        c = [rng.uniform(-0.03, 0.03), rng.uniform(-0.03, 0.03), rng.uniform(2.5, 5.0)]
        G = rng.standard_normal((1, 1, 3))
        sc = _scene(c, rng.uniform(0.15, 0.3), rng.uniform(0.2, 1.0), rng.uniform(-1, 1, 3),
                    W=1, H=1, fx=rng.uniform(8, 12), cx=rng.uniform(0.3, 0.7),
                    cy=rng.uniform(0.3, 0.7), G=G)
        o = _check(oracle_lib, sc)
        F = o["image"][0, 0]
        f = sc.features[0].astype(np.float64)
        g = sc.grad_images[0][0, 0].astype(np.float64)   # as the oracle received it
        ratio = np.abs(g).sum() / abs(float(g @ (f - F)))
        for key in ("grad_pos", "grad_radius", "grad_opacity", "grad_cam"):
            v = np.abs(np.asarray(o[key], np.float64)).ravel()
            a = np.asarray(o["abs_" + key]).ravel()
            s = np.asarray(o["sens_" + key]).ravel()
            assert np.allclose(a, v, rtol=1e-13, atol=0), key
            assert np.allclose(s, v * ratio, rtol=1e-12, atol=0), key
        assert np.allclose(o["abs_grad_features"], np.abs(o["grad_features"]), rtol=1e-13)
        assert not o["sens_grad_features"].any()


def test_mirrored_pixels_cancel_in_value_not_in_abs_sum(oracle_lib):
    """Two pixels mirrored about a sphere on the plane c.x = 0.  With equal
    upstream gradients their contributions to dL/dc.x (= dL/dt_x) and dL/dcx
    are equal and opposite: the value is 0 while A is twice one contribution.
    With opposite upstream gradients the feature and opacity entries cancel
    instead."""
    base = dict(c=[0.0, 0.04, 4.0], r=0.5, o=0.7, f=[0.3, -0.8, 0.5], W=2, H=1, fx=20.0, cx=1.0,
                cy=0.5, fy=20.0)
    g = np.array([0.9, -0.4, 1.3])
    sym = _scene(G=np.stack([g, g])[None], **base)
    _check(oracle_lib, sym, expect_cancel=("pos x", "t0", "cx"))
    anti = _scene(G=np.stack([g, -g])[None], **base)
    _check(oracle_lib, anti, expect_cancel=("opacity", "feature 0", "feature 1", "feature 2"))


def test_many_pixels_terms(oracle_lib):
    """A sphere covering a few dozen pixels, fx != fy, an off-centre principal
    point: A and S summed over all of them."""
    rng = np.random.default_rng(9)
    W, H = 9, 7
    G = rng.standard_normal((H, W, 2))
    sc = _scene([0.05, -0.03, 3.0], 0.7, 0.6, [0.4, -0.2], W=W, H=H, fx=14.0, cx=4.3, cy=3.6,
                G=G, fy=11.0)
    o = _check(oracle_lib, sc)
    assert o["nhits"].sum() >= 20


@pytest.mark.parametrize("slip", ["abs x10", "sens wrong axis"])
def test_planted_slips_are_caught(oracle_lib, slip):
    """The checks above reject an abs sum ten times too large and a
    sensitivity summed over the pixels instead of the channels."""
    sc = _scene([0.0, 0.04, 4.0], 0.5, 0.7, [0.3, -0.8, 0.5], W=2, H=1, fx=20.0, cx=1.0,
                cy=0.5, fy=20.0, G=np.array([[[0.9, -0.4, 1.3], [0.9, -0.4, 1.3]]]))
    o = oracle_lib.render(sc.pos, sc.radius, sc.opacity, sc.features, sc.cameras[0], sc.params,
                          sc.bg, grad_image=sc.grad_images[0], fp64=True)
    name, key, idx, perturb = _perturbers(sc)[1]          # pos y
    contrib, A, S, _ = _independent_terms(sc, perturb, False)
    a, s = o["abs_" + key][idx], o["sens_" + key][idx]
    if slip == "abs x10":
        a = 10 * a
        assert abs(a - A) > 1e-6 * A
    else:
        # ||G||_1 taken per channel over the pixels instead of per pixel over channels
        G = sc.grad_images[0].astype(np.float64)
        F = o["image"]
        f = sc.features[0].astype(np.float64)
        sdot = (G * (f - F)).sum(-1)
        wrong = (np.abs(contrib) * np.abs(G).sum(1)[:, :1] / np.abs(sdot)).sum()
        assert abs(wrong - S) > 1e-6 * S
        assert abs(s - S) <= 1e-6 * S
