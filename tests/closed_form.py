"""Independent fp64 restatement of the blend for tiny inputs (test helper).

Written from the Pulsar paper's description (Sec. 3.2, App. A) with
formulations deliberately different from the oracle's, so that a slip in
either shows up as a disagreement:

* ray-to-centre distance from the cross product |c x q| / |q| (the oracle
  uses the Lagrange-identity form in pixel offsets);
* tangent-cone pixel bounds from tan(alpha +- beta) with atan2/asin (the
  oracle uses the trigonometry-free identity);
* un-shifted exponentials exp(o z / gamma) (the oracle shifts by the max).

Pure numpy, brute force over every pixel and sphere: only for small scenes.
"""
from __future__ import annotations

import math

import numpy as np


def camera_space(pos, cam):
    R = np.asarray(cam.R, np.float64).reshape(3, 3)
    t = np.asarray(cam.t, np.float64)
    return np.asarray(pos, np.float64) @ R.T + t


def reff(radius, c, cam, kappa):
    fmin = min(cam.fx, cam.fy)
    return np.maximum(np.asarray(radius, np.float64), kappa * c[:, 2] / fmin)


def pixel_rays(cam):
    xs = (np.arange(cam.width) + 0.5 - cam.cx) / cam.fx
    ys = (np.arange(cam.height) + 0.5 - cam.cy) / cam.fy
    a, b = np.meshgrid(xs, ys)                       # [H,W]
    return np.stack([a, b, np.ones_like(a)], -1)     # [H,W,3]


def ray_distance(c, q):
    """|c x q| / |q| for every pixel ray q [H,W,3] and centre c [3]."""
    cr = np.cross(np.broadcast_to(c, q.shape), q)
    return np.linalg.norm(cr, axis=-1) / np.linalg.norm(q, axis=-1)


def tangent_bounds(X, Z, Rr, f, c0):
    """Projected extent of a sphere along one axis via angles."""
    alpha = math.atan2(X, Z)
    beta = math.asin(min(1.0, Rr / math.hypot(X, Z)))
    lo = alpha - beta
    hi = alpha + beta
    umin = c0 + f * math.tan(lo) if lo > -math.pi / 2 else -math.inf
    umax = c0 + f * math.tan(hi) if hi < math.pi / 2 else math.inf
    return umin, umax


def render(pos, radius, opacity, features, cam, params, bg, gaussian=False):
    """Returns image [H,W,C], per-pixel sorted hit ids (list of lists), weights.
    gaussian: the distance factor is a Gaussian of standard deviation r/3 over
    the same support, shifted and scaled to run from 1 at the centre to 0 at
    the rim."""
    c = camera_space(pos, cam)
    r = reff(radius, c, cam, params.kappa)
    q = pixel_rays(cam)
    H, W = cam.height, cam.width
    C = features.shape[1]
    zt = (cam.zfar - c[:, 2]) / (cam.zfar - cam.znear)
    o = np.asarray(opacity, np.float64)
    num = np.zeros((H, W, C)) + math.exp(params.bg_eps / params.gamma) * np.asarray(bg, np.float64)
    den = np.zeros((H, W)) + math.exp(params.bg_eps / params.gamma)
    hits = [[[] for _ in range(W)] for _ in range(H)]
    keyv = c[:, 2] - r
    order = np.lexsort((np.arange(len(keyv)), keyv))
    for i in order:
        z = c[i, 2]
        if not (cam.znear < z < cam.zfar and r[i] < z):
            continue
        rho = ray_distance(c[i], q)
        m = rho < r[i]
        if not m.any():
            continue
        if gaussian:
            sigma = r[i] / 3.0
            tail = math.exp(-0.5 * 9.0)
            d = (np.exp(-0.5 * (rho / sigma) ** 2) - tail) / (1.0 - tail)
        else:
            d = 1.0 - rho / r[i]
        w = np.where(m, o[i] * d * math.exp(o[i] * zt[i] / params.gamma), 0.0)
        num += w[..., None] * np.asarray(features[i], np.float64)
        den += w
        for y, x in zip(*np.nonzero(m)):
            hits[y][x].append(int(i))
    return num / den[..., None], hits


def render_ortho(pos, radius, opacity, features, cam, params, bg):
    """Orthographic counterpart of render(): pixel (x, y) is the camera-space
    ray o + s e_z from o = (X, Y, 0), X = (x + 0.5 - cx)/fx, Y = (y + 0.5 -
    cy)/fy; the ray-to-centre distance is taken as the 3-D distance from the
    centre c to its closest point on the ray, o + ((c - o).e_z) e_z, instead
    of from pixel offsets to the projected centre.  Returns image [H,W,C] and
    per-pixel hit ids in (key, id) order."""
    c = camera_space(pos, cam)
    r = np.maximum(np.asarray(radius, np.float64), params.kappa / min(cam.fx, cam.fy))
    H, W = cam.height, cam.width
    X = (np.arange(W) + 0.5 - cam.cx) / cam.fx
    Y = (np.arange(H) + 0.5 - cam.cy) / cam.fy
    Xg, Yg = np.meshgrid(X, Y)
    org = np.stack([Xg, Yg, np.zeros_like(Xg)], -1)            # [H,W,3]
    ez = np.array([0.0, 0.0, 1.0])
    C = features.shape[1]
    zt = (cam.zfar - c[:, 2]) / (cam.zfar - cam.znear)
    o = np.asarray(opacity, np.float64)
    num = np.zeros((H, W, C)) + math.exp(params.bg_eps / params.gamma) * np.asarray(bg, np.float64)
    den = np.zeros((H, W)) + math.exp(params.bg_eps / params.gamma)
    hits = [[[] for _ in range(W)] for _ in range(H)]
    keyv = c[:, 2] - r
    order = np.lexsort((np.arange(len(keyv)), keyv))
    for i in order:
        z = c[i, 2]
        if not (cam.znear < z < cam.zfar and r[i] < z):
            continue
        dvec = c[i] - org
        closest = org + (dvec @ ez)[..., None] * ez
        rho = np.linalg.norm(c[i] - closest, axis=-1)
        m = rho < r[i]
        if not m.any():
            continue
        d = 1.0 - rho / r[i]
        w = np.where(m, o[i] * d * math.exp(o[i] * zt[i] / params.gamma), 0.0)
        num += w[..., None] * np.asarray(features[i], np.float64)
        den += w
        for y, x in zip(*np.nonzero(m)):
            hits[y][x].append(int(i))
    return num / den[..., None], hits
