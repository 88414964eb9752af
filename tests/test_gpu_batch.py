"""Batched multi-camera launch (pulsar_project_cams): one project, bin,
forward and backward over all cameras of a rig, against the oracle run
camera by camera.

Bit-exact per camera: fp32 decisions, tile lists, tracked ids, hit counts.
Within tolerance: images and buffers per camera; sphere gradients against
the sum of the per-camera oracle gradients (L sums over cameras); camera
gradients per camera.  And the batch renders every camera exactly as the
single-camera path does.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import gpu_helpers as gh
from splat_rendering_gb300 import scenes

pytestmark = pytest.mark.gpu

LN2 = math.log(2.0)


def run_batch(sc, cams, grads, max_pairs, p=None):
    """Render cameras `cams` of one sphere set as one batch; per-camera views."""
    import torch
    from splat_rendering_gb300 import pulsar as pl
    p = sc.params if p is None else p
    K, n = len(cams), sc.n
    H, W = cams[0].height, cams[0].width
    r = pl.Renderer(max_spheres=max(n, 1), max_pairs=max_pairs, max_width=W, max_height=H,
                    max_channels=p.channels, max_track=p.n_track, max_cams=K)
    t = gh._t
    img = r.render(t(sc.pos), t(sc.radius), t(sc.opacity), t(sc.features.reshape(n, -1)),
                   [pl.camera(c) for c in cams], pl.params(p, count_hits=True), t(sc.bg))
    g = r.backward(t(np.stack(grads)))
    code, m, h = r.status(raise_on_error=False)
    torch.cuda.synchronize()
    out = {"code": code, "n_pairs": m, "hits": h, "image": img.cpu().numpy()}
    out.update({f"grad_{k}": v.cpu().numpy() for k, v in g.items()})
    out["records"] = r.debug("records").view(np.uint32).reshape(K, n, 16)
    out["tile_offsets"] = r.debug("tile_offsets").view(np.uint32).astype(np.int64)
    out["tile_ids"] = r.debug("tile_ids").view(np.uint32)[:m].astype(np.int64)
    out["mg"] = r.debug("mg").view(np.float32).reshape(K, H, W).astype(np.float64) * LN2
    out["wsum"] = r.debug("wsum").view(np.float32).reshape(K, H, W)
    out["ids"] = np.moveaxis(r.debug("ids").view(np.int32).reshape(p.n_track, K, H, W), 0, -1)
    out["nhits"] = r.debug("nhits").view(np.int32).reshape(K, H, W)
    r.close()
    return out


def check_batch(oracle_lib, sc, cams, grads, window=None, p=None):
    p = sc.params if p is None else p
    K = len(cams)
    per = []
    for k, cam in enumerate(cams):
        o = oracle_lib.render(sc.pos, sc.radius, sc.opacity, sc.features, cam, p, sc.bg,
                              grad_image=grads[k], window=window)
        d = oracle_lib.project(sc.pos, sc.radius, sc.opacity, cam, p)
        offs, ids = oracle_lib.tile_lists(sc.pos, sc.radius, sc.opacity, cam, p)
        per.append((o, d, offs, ids))
    total = sum(len(x[3]) for x in per)
    g = run_batch(sc, cams, grads, max_pairs=total + 1024, p=p)
    assert g["code"] == 0 and g["n_pairs"] == total
    if window is None:   # (the oracle counts the window's hits only)
        assert g["hits"] == sum(x[0]["hits"] for x in per)
    B = (len(g["tile_offsets"]) - 1) // K
    for k, (o, d, offs, ids) in enumerate(per):
        what = f"camera {k}"
        gk = {key: g[key][k] for key in ("image", "mg", "wsum", "ids", "nhits", "records")}
        gh.assert_decisions_equal(gk, d)
        lo, hi = g["tile_offsets"][k * B], g["tile_offsets"][(k + 1) * B]
        assert np.array_equal(g["tile_offsets"][k * B:(k + 1) * B + 1] - lo, offs), what
        assert np.array_equal(g["tile_ids"][lo:hi], ids.astype(np.int64)), what
        gh.compare_frame(gk, o, what, window=window, grads=False)
        sl = (slice(None), slice(None)) if window is None else \
            (slice(window[1], window[3]), slice(window[0], window[2]))
        dF = gh.image_err(gk["image"][sl], o["image"])
        dF_all = max(dF_all, dF) if k else dF
        gh.assert_close(g["grad_cam"][k], o["grad_cam"], gh.GRAD_RTOL, gh.GRAD_ATOL,
                        f"{what} grad_cam", o["abs_grad_cam"], o["sens_grad_cam"], dF)
    for key in ("grad_pos", "grad_radius", "grad_opacity", "grad_features"):
        ref = sum(x[0][key] for x in per)
        a = sum(x[0]["abs_" + key] for x in per)
        s = sum(x[0]["sens_" + key] for x in per)
        gh.assert_close(g[key], ref, gh.GRAD_RTOL, gh.GRAD_ATOL, f"batch {key}", a, s, dF_all)
    return g


def _rig(seed, K, W, H, ortho_at=()):
    """K cameras looking at the sphere cloud from different poses."""
    rng = np.random.default_rng(seed)
    cams = []
    for k in range(K):
        axis = rng.standard_normal(3)
        axis /= np.linalg.norm(axis)
        R = scenes._rotation(axis, math.radians(rng.uniform(0, 20)))
        t = rng.uniform(-0.3, 0.3, 3)
        if k in ortho_at:
            cams.append(scenes._camera(R, t, 16.0, W, H, 1.0, 7.0, orthographic=True))
        else:
            cams.append(scenes._camera(R, t, rng.uniform(40, 70), W, H, 1.0, 7.0,
                                       fy=rng.uniform(40, 70), cx=W / 2 + 1.3, cy=H / 2 - 0.7))
    return cams


def test_small_mixed_rig(oracle_lib):
    """Four cameras (one orthographic), full frames, gradients of all kinds."""
    sc = scenes.random_scene(101, 2500, 64, 48, rrange=(0.01, 0.3), zrange=(2.0, 6.0))
    cams = _rig(101, 4, 64, 48, ortho_at=(2,))
    rng = np.random.default_rng(7)
    grads = [rng.standard_normal((48, 64, 3)).astype(np.float32) for _ in cams]
    check_batch(oracle_lib, sc, cams, grads)


def test_driving_rig_batched(oracle_lib):
    """The six driving cameras in one batch: decisions and tile lists of every
    camera, images and gradients on a 320 x 192 window of each."""
    sc = scenes.driving()
    win = (800, 560, 1120, 752)
    grads = [gh.windowed_grad(sc, k, win) for k in range(6)]
    check_batch(oracle_lib, sc, sc.cameras, grads, window=win)


def test_batch_renders_each_camera_as_the_single_path():
    """Every camera's image, stabiliser and tracked ids are bit-identical to
    those of the single-camera path (the same arithmetic per tile)."""
    sc = scenes.random_scene(102, 3000, 80, 60, rrange=(0.01, 0.3))
    cams = _rig(102, 3, 80, 60, ortho_at=(1,))
    grads = [sc.grad_images[0]] * 3
    g = run_batch(sc, cams, grads, max_pairs=1 << 18)
    for k, cam in enumerate(cams):
        one = scenes.Scene(sc.name, sc.pos, sc.radius, sc.opacity, sc.features, [cam], sc.params,
                           sc.bg, [grads[k]])
        s = gh.run_gpu(one, max_pairs=1 << 18)
        assert np.array_equal(g["image"][k], s["image"]), k
        assert np.array_equal(g["ids"][k], s["ids"]), k
        assert np.array_equal(g["mg"][k], s["mg"]), k


def test_sixteen_channel_rig(oracle_lib):
    """Three cameras (one orthographic) with 16 channels and n_track 8: the
    batched instantiations of the wide-feature forward and backward, and the
    finalize that sums feature and opacity gradients over the cameras."""
    sc = scenes.random_scene(103, 1500, 48, 40, channels=16, n_track=8, rrange=(0.02, 0.3))
    cams = _rig(103, 3, 48, 40, ortho_at=(1,))
    rng = np.random.default_rng(9)
    grads = [rng.standard_normal((40, 48, 16)).astype(np.float32) for _ in cams]
    check_batch(oracle_lib, sc, cams, grads)
