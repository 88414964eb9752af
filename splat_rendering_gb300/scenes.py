"""Seeded synthetic scenes for the sphere renderer.

This module only draws inputs: sphere positions, radii, opacities, feature
payloads, pinhole cameras and upstream image gradients.  It holds none of the
renderer's arithmetic, so both the CUDA path and the CPU oracle can be fed
from it.  All arrays are float32 (the renderer's input type); every draw uses
``numpy.random.default_rng(seed)`` (PCG64) in the fixed order
positions, radii, opacities, features, camera, upstream gradient.

The five named workloads stand in for the scenes the Pulsar paper and the
NuRec profiling article measure on (NeRF captures, head scans, driving logs),
none of which is available here:

* ``tiny``      1,000 spheres, 64x64, focal 64 px (Pulsar-style toy scene)
* ``medium``    100,000 spheres, 512x512, focal 512 px, camera rotated <=10 deg
* ``headline``  1,000,000 spheres, 1024x1024, focal 1024 px -- the scale of the
                Pulsar paper's 1M-sphere timing (Sec. 1 and Table 2)
* ``neural``    the headline scene with 16-channel N(0,1) feature vectors
* ``driving``   2,000,000 spheres on a ground plane plus Gaussian clusters,
                six 1920x1080 cameras at 60 deg yaw spacing (NuRec-like rig)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# Blending and pruning constants shared by every workload (readings of the
# Pulsar paper, which prints no values for them).
GAMMA = 0.1          # blending temperature
BG_EPS = 1e-5        # background "depth" in the blend
STOP_TAU = 1e-8      # early-stop tolerance of the forward pass
KAPPA = 0.75         # minimum projected radius in pixels
GEOM_MIN_AREA = 3.0  # projected area (px^2) at or below which geometry grads are dropped


@dataclass
class Camera:
    R: np.ndarray            # [9] float32, world->camera rotation, row-major
    t: np.ndarray            # [3] float32
    fx: float
    fy: float
    cx: float
    cy: float
    width: int
    height: int
    znear: float
    zfar: float
    orthographic: bool = False   # rays along +z from (X, Y, 0); fx, fy in pixels per unit

    def packed(self) -> np.ndarray:
        """[R(9), t(3), fx, fy, cx, cy, znear, zfar] as float32."""
        return np.concatenate([
            self.R.astype(np.float32), self.t.astype(np.float32),
            np.array([self.fx, self.fy, self.cx, self.cy, self.znear, self.zfar],
                     dtype=np.float32)])


@dataclass
class Params:
    gamma: float = GAMMA
    bg_eps: float = BG_EPS
    stop_tau: float = STOP_TAU
    kappa: float = KAPPA
    geom_min_area: float = GEOM_MIN_AREA
    n_track: int = 5
    channels: int = 3
    geom_cutoff: bool = True
    normalize_grads: bool = False   # averaged sphere / area-normalised camera gradients
    gaussian: bool = False          # Gaussian footprint (sigma = r_eff / 3) instead of linear


@dataclass
class Scene:
    name: str
    pos: np.ndarray          # [N,3] float32
    radius: np.ndarray       # [N]   float32
    opacity: np.ndarray      # [N]   float32
    features: np.ndarray     # [N,C] float32
    cameras: list            # list[Camera]
    params: Params
    bg: np.ndarray           # [C] float32
    grad_images: list = field(default_factory=list)   # per camera [H,W,C] float32

    @property
    def n(self) -> int:
        return int(self.pos.shape[0])


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _log_uniform(rng, lo, hi, n):
    return np.exp(rng.uniform(math.log(lo), math.log(hi), n))


def _rotation(axis, angle) -> np.ndarray:
    """Rodrigues rotation matrix (float64) about a unit axis."""
    x, y, z = axis
    c, s = math.cos(angle), math.sin(angle)
    C = 1.0 - c
    return np.array([[c + x * x * C, x * y * C - z * s, x * z * C + y * s],
                     [y * x * C + z * s, c + y * y * C, y * z * C - x * s],
                     [z * x * C - y * s, z * y * C + x * s, c + z * z * C]])


def _camera(R, t, f, width, height, znear, zfar, fy=None, cx=None, cy=None,
            orthographic=False) -> Camera:
    return Camera(R=_f32(np.asarray(R).reshape(9)), t=_f32(np.asarray(t).reshape(3)),
                  fx=float(np.float32(f)), fy=float(np.float32(f if fy is None else fy)),
                  cx=float(np.float32(width / 2 if cx is None else cx)),
                  cy=float(np.float32(height / 2 if cy is None else cy)),
                  width=int(width), height=int(height),
                  znear=float(np.float32(znear)), zfar=float(np.float32(zfar)),
                  orthographic=bool(orthographic))


def _grads(rng, cams, C):
    return [_f32(rng.standard_normal((c.height, c.width, C))) for c in cams]


def tiny(seed: int = 0) -> Scene:
    rng = np.random.default_rng(seed)
    n = 1000
    pos = np.stack([rng.uniform(-1, 1, n), rng.uniform(-1, 1, n), rng.uniform(2, 6, n)], 1)
    rad = _log_uniform(rng, 0.01, 0.1, n)
    opa = rng.uniform(0.1, 1.0, n)
    feat = rng.uniform(0.0, 1.0, (n, 3))
    cams = [_camera(np.eye(3), np.zeros(3), 64, 64, 64, 1.0, 7.0)]
    return Scene("tiny", _f32(pos), _f32(rad), _f32(opa), _f32(feat), cams,
                 Params(n_track=5, channels=3), _f32(np.zeros(3)), _grads(rng, cams, 3))


def medium(seed: int = 1) -> Scene:
    rng = np.random.default_rng(seed)
    n = 100_000
    pos = np.stack([rng.uniform(-2, 2, n), rng.uniform(-2, 2, n), rng.uniform(2, 10, n)], 1)
    rad = _log_uniform(rng, 0.002, 0.05, n)
    opa = rng.uniform(0.05, 1.0, n)
    feat = rng.uniform(0.0, 1.0, (n, 3))
    axis = rng.standard_normal(3)
    axis /= np.linalg.norm(axis)
    angle = math.radians(rng.uniform(0.0, 10.0))
    cams = [_camera(_rotation(axis, angle), np.zeros(3), 512, 512, 512, 1.0, 11.0)]
    return Scene("medium", _f32(pos), _f32(rad), _f32(opa), _f32(feat), cams,
                 Params(n_track=5, channels=3), _f32(np.zeros(3)), _grads(rng, cams, 3))


def _frustum_volume(rng, n, z0, z1, half_tan):
    """Uniform in the volume of a square frustum |x|,|y| <= half_tan*z, z in [z0,z1]."""
    u = rng.uniform(0.0, 1.0, n)
    z = np.cbrt(z0 ** 3 + u * (z1 ** 3 - z0 ** 3))
    x = rng.uniform(-1.0, 1.0, n) * half_tan * z
    y = rng.uniform(-1.0, 1.0, n) * half_tan * z
    return np.stack([x, y, z], 1)


def headline(seed: int = 2, n: int = 1_000_000) -> Scene:
    rng = np.random.default_rng(seed)
    pos = _frustum_volume(rng, n, 1.0, 20.0, 0.5)
    rad = _log_uniform(rng, 0.001, 0.03, n)
    opa = rng.uniform(0.05, 1.0, n)
    feat = rng.uniform(0.0, 1.0, (n, 3))
    cams = [_camera(np.eye(3), np.zeros(3), 1024, 1024, 1024, 0.5, 21.0)]
    return Scene("headline", _f32(pos), _f32(rad), _f32(opa), _f32(feat), cams,
                 Params(n_track=5, channels=3), _f32(np.zeros(3)), _grads(rng, cams, 3))


def headline_ortho(seed: int = 2, n: int = 1_000_000) -> Scene:
    """The headline scene's sizes seen by an orthographic camera: 1M spheres
    uniform in the box |x|, |y| <= 7, z in [1, 20], 1024 x 1024 pixels at
    1024/14 px per unit (so projected radii match the headline's median
    depth), same radius, opacity and feature distributions."""
    rng = np.random.default_rng(seed)
    pos = np.stack([rng.uniform(-7.0, 7.0, n), rng.uniform(-7.0, 7.0, n),
                    rng.uniform(1.0, 20.0, n)], 1)
    rad = _log_uniform(rng, 0.001, 0.03, n)
    opa = rng.uniform(0.05, 1.0, n)
    feat = rng.uniform(0.0, 1.0, (n, 3))
    cams = [_camera(np.eye(3), np.zeros(3), 1024 / 14, 1024, 1024, 0.5, 21.0, orthographic=True)]
    return Scene("headline_ortho", _f32(pos), _f32(rad), _f32(opa), _f32(feat), cams,
                 Params(n_track=5, channels=3), _f32(np.zeros(3)), _grads(rng, cams, 3))


def neural(seed: int = 3, n: int = 1_000_000) -> Scene:
    rng = np.random.default_rng(seed)
    pos = _frustum_volume(rng, n, 1.0, 20.0, 0.5)
    rad = _log_uniform(rng, 0.001, 0.03, n)
    opa = rng.uniform(0.05, 1.0, n)
    feat = rng.standard_normal((n, 16))
    cams = [_camera(np.eye(3), np.zeros(3), 1024, 1024, 1024, 0.5, 21.0)]
    return Scene("neural", _f32(pos), _f32(rad), _f32(opa), _f32(feat), cams,
                 Params(n_track=8, channels=16), _f32(np.zeros(16)), _grads(rng, cams, 16))


def driving_cameras(width=1920, height=1080, hfov_deg=60.0):
    f = (width / 2) / math.tan(math.radians(hfov_deg / 2))
    centre = np.array([0.0, -1.5, 0.0])
    cams = []
    for k in range(6):
        th = math.radians(60.0 * k)
        R = np.array([[math.cos(th), 0.0, -math.sin(th)],
                      [0.0, 1.0, 0.0],
                      [math.sin(th), 0.0, math.cos(th)]])
        cams.append(_camera(R, -R @ centre, f, width, height, 0.5, 100.0))
    return cams


def driving(seed: int = 4, n: int = 2_000_000) -> Scene:
    rng = np.random.default_rng(seed)
    n_plane = int(round(0.7 * n))
    n_clu = n - n_plane
    plane = np.stack([rng.uniform(-30, 30, n_plane), np.zeros(n_plane),
                      rng.uniform(2, 80, n_plane)], 1)
    centres = np.stack([rng.uniform(-30, 30, 50), rng.uniform(-3, 0, 50),
                        rng.uniform(2, 80, 50)], 1)
    which = rng.integers(0, 50, n_clu)
    clusters = centres[which] + rng.standard_normal((n_clu, 3))
    pos = np.concatenate([plane, clusters], 0)
    rad = _log_uniform(rng, 0.01, 0.3, n)
    opa = rng.uniform(0.05, 1.0, n)
    feat = rng.uniform(0.0, 1.0, (n, 3))
    cams = driving_cameras()
    return Scene("driving", _f32(pos), _f32(rad), _f32(opa), _f32(feat), cams,
                 Params(n_track=5, channels=3), _f32(np.zeros(3)), _grads(rng, cams, 3))


def random_scene(seed: int, n: int, width: int, height: int, *, channels: int = 3,
                 n_track: int = 5, f: float | None = None, fy: float | None = None,
                 zrange=(2.0, 6.0), rrange=(0.01, 0.1), orange=(0.1, 1.0),
                 spread: float = 1.0, rot_deg: float = 0.0, shift=(0.0, 0.0, 0.0),
                 cx: float | None = None, cy: float | None = None,
                 znear: float = 1.0, zfar: float = 7.0, gamma: float = GAMMA,
                 geom_cutoff: bool = True, orthographic: bool = False) -> Scene:
    """A small scene for edge-case and property tests (same draw order).  With
    an orthographic camera, f is in pixels per world unit and the spheres fill
    the image's box instead of its frustum."""
    rng = np.random.default_rng(seed)
    f = float(max(width, height)) if f is None else f
    z = rng.uniform(zrange[0], zrange[1], n)
    hx = spread * (width / 2) / f
    hy = spread * (height / 2) / (f if fy is None else fy)
    sz = np.ones_like(z) if orthographic else z
    pos = np.stack([rng.uniform(-1, 1, n) * hx * sz, rng.uniform(-1, 1, n) * hy * sz, z], 1)
    rad = _log_uniform(rng, rrange[0], rrange[1], n) if n else np.zeros(0)
    opa = rng.uniform(orange[0], orange[1], n)
    feat = rng.uniform(0.0, 1.0, (n, channels))
    if rot_deg:
        axis = rng.standard_normal(3)
        axis /= np.linalg.norm(axis)
        R = _rotation(axis, math.radians(rot_deg))
    else:
        R = np.eye(3)
    # a camera transform that keeps the sampled camera-space positions: p_world = R^T (p_cam - t)
    t = np.asarray(shift, dtype=np.float64)
    pos_w = (pos - t) @ R
    cams = [_camera(R, t, f, width, height, znear, zfar, fy=fy, cx=cx, cy=cy,
                    orthographic=orthographic)]
    p = Params(n_track=n_track, channels=channels, gamma=gamma, geom_cutoff=geom_cutoff)
    return Scene(f"random{seed}", _f32(pos_w), _f32(rad), _f32(opa), _f32(feat), cams, p,
                 _f32(np.zeros(channels)), _grads(rng, cams, channels))


def shading_mlp(seed: int = 5) -> np.ndarray:
    """Seeded weights of the per-pixel shading MLP (16 features + 3 view
    direction -> 64 -> 64 -> 3), flat float32 in the order W1 [64,19], b1,
    W2 [64,64], b2, W3 [3,64], b3; He-normal weights, small biases."""
    rng = np.random.default_rng(seed)
    parts = [rng.standard_normal((64, 19)) * math.sqrt(2.0 / 19), rng.uniform(-0.1, 0.1, 64),
             rng.standard_normal((64, 64)) * math.sqrt(2.0 / 64), rng.uniform(-0.1, 0.1, 64),
             rng.standard_normal((3, 64)) * math.sqrt(1.0 / 64), rng.uniform(-0.1, 0.1, 3)]
    return _f32(np.concatenate([np.asarray(q).reshape(-1) for q in parts]))


def shading_grad(seed: int, height: int, width: int) -> np.ndarray:
    """Seeded dL/d rgb [H, W, 3] (N(0,1)) for the shading MLP's backward."""
    return _f32(np.random.default_rng(seed).standard_normal((height, width, 3)))


CONFIGS = {
    "tiny": tiny,
    "medium": medium,
    "headline": headline,
    "headline_ortho": headline_ortho,
    "neural": neural,
    "driving": driving,
}


def make(name: str, **kw) -> Scene:
    return CONFIGS[name](**kw)
