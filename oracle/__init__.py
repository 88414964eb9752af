"""CPU oracle for the Pulsar-style sphere renderer -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does: it has no
CPU fallback.  The numerics live in ``pulsar_oracle.cpp`` (plain fp64 C++,
OpenMP over pixel rows / spheres); this module only builds and calls it.

Every function follows a passage of "Pulsar: Efficient Sphere-based Neural
Rendering" (paperlayer.ai summary of arXiv 2004.07484); the readings of what
the pages leave open are listed in the C++ file's header.

Parity pins: all oracle functions are pinned by tests/test_oracle_*.py
(closed forms, partition of unity, opacity-zero removal, permutation
invariance, gamma limits, brute == culled, fp32 == fp64 decisions away from
ties, translation identity, central finite differences).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pulsar_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the oracle with g++ (OpenMP if available, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-fno-finite-math-only", _SRC, "-o", _LIB + ".tmp"]
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(_LIB + ".tmp", _LIB)
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            return _LIB
    raise RuntimeError("oracle build failed:\n" + r.stderr)


class _Cam(ctypes.Structure):
    _fields_ = [("R", ctypes.c_double * 9), ("t", ctypes.c_double * 3),
                ("fx", ctypes.c_double), ("fy", ctypes.c_double), ("cx", ctypes.c_double),
                ("cy", ctypes.c_double), ("znear", ctypes.c_double), ("zfar", ctypes.c_double),
                ("width", ctypes.c_int32), ("height", ctypes.c_int32),
                ("orthographic", ctypes.c_int32)]


class _Params(ctypes.Structure):
    _fields_ = [("gamma", ctypes.c_double), ("bg_eps", ctypes.c_double),
                ("kappa", ctypes.c_double), ("geom_min_area", ctypes.c_double),
                ("n_track", ctypes.c_int32), ("channels", ctypes.c_int32),
                ("geom_cutoff", ctypes.c_int32), ("fp64_decisions", ctypes.c_int32),
                ("normalize", ctypes.c_int32), ("gaussian", ctypes.c_int32)]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_project.restype = ctypes.c_int
        lib.oracle_project.argtypes = [P, P, P, ctypes.c_int64, P, P] + [P] * 9
        lib.oracle_tile_lists.restype = ctypes.c_int64
        lib.oracle_tile_lists.argtypes = [P, P, P, ctypes.c_int64, P, P, P, P, ctypes.c_int64]
        lib.oracle_render.restype = ctypes.c_int64
        lib.oracle_render.argtypes = ([P, P, P, P, ctypes.c_int64, P, P, P] +
                                      [ctypes.c_int32] * 5 + [P] * 12)
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_threads(n: int) -> None:
    """Threads of the following oracle calls (n <= 0: all host cores)."""
    _load().oracle_set_threads(int(n))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _cam(cam) -> _Cam:
    """Camera fields as fp64 (float32 inputs convert exactly)."""
    c = _Cam()
    c.R[:] = [float(v) for v in np.asarray(cam.R, np.float64).reshape(9)]
    c.t[:] = [float(v) for v in np.asarray(cam.t, np.float64).reshape(3)]
    for k in ("fx", "fy", "cx", "cy", "znear", "zfar"):
        setattr(c, k, float(getattr(cam, k)))
    c.width, c.height = int(cam.width), int(cam.height)
    c.orthographic = 1 if getattr(cam, "orthographic", False) else 0
    return c


def _params(p, fp64: bool) -> _Params:
    """Blend parameters as the float32 values the renderer's interface carries
    (fp64 decisions: as given)."""
    q = _Params()
    r = (lambda v: float(v)) if fp64 else (lambda v: float(np.float32(v)))
    q.gamma, q.bg_eps = r(p.gamma), r(p.bg_eps)
    q.kappa, q.geom_min_area = r(p.kappa), r(p.geom_min_area)
    q.n_track, q.channels = int(p.n_track), int(p.channels)
    q.geom_cutoff = 1 if p.geom_cutoff else 0
    q.fp64_decisions = 1 if fp64 else 0
    q.normalize = 1 if getattr(p, "normalize_grads", False) else 0
    q.gaussian = 1 if getattr(p, "gaussian", False) else 0
    return q


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def project(pos, radius, opacity, cam, params, fp64: bool = False) -> dict:
    """Per-sphere decision quantities (fp32 sequence unless fp64=True)."""
    lib = _load()
    pos, radius, opacity = _f64(pos).reshape(-1, 3), _f64(radius), _f64(opacity)
    n = pos.shape[0]
    out = dict(keep=np.zeros(n, np.int32), uv=np.zeros((n, 4), np.float32),
               reff=np.zeros(n, np.float32), key=np.zeros(n, np.float32),
               s2=np.zeros(n, np.float32), rect=np.zeros((n, 4), np.int32),
               floor=np.zeros(n, np.int32), cut=np.zeros(n, np.int32),
               ntiles=np.zeros(n, np.int32))
    c, q = _cam(cam), _params(params, fp64)
    rc = lib.oracle_project(_ptr(pos), _ptr(radius), _ptr(opacity), n, ctypes.byref(c),
                            ctypes.byref(q), _ptr(out["keep"]), _ptr(out["uv"]), _ptr(out["reff"]),
                            _ptr(out["key"]), _ptr(out["s2"]), _ptr(out["rect"]),
                            _ptr(out["floor"]), _ptr(out["cut"]), _ptr(out["ntiles"]))
    if rc != 0:
        raise RuntimeError(f"oracle_project failed: {rc}")
    return out


def tile_lists(pos, radius, opacity, cam, params, fp64: bool = False):
    """(offsets [B+1] int64, ids [M] int32) of the 16x16 tile lists."""
    lib = _load()
    pos, radius, opacity = _f64(pos).reshape(-1, 3), _f64(radius), _f64(opacity)
    n = pos.shape[0]
    B = ((cam.width + 15) // 16) * ((cam.height + 15) // 16)
    offsets = np.zeros(B + 1, np.int64)
    c, q = _cam(cam), _params(params, fp64)
    cap = 0
    while True:
        ids = np.zeros(max(cap, 1), np.int32)
        m = lib.oracle_tile_lists(_ptr(pos), _ptr(radius), _ptr(opacity), n, ctypes.byref(c),
                                  ctypes.byref(q), _ptr(offsets), _ptr(ids), cap)
        if m >= 0:
            return offsets, ids[:m]
        cap = -m - 1


def render(pos, radius, opacity, features, cam, params, bg, grad_image=None, window=None,
           brute: bool = False, fp64: bool = False) -> dict:
    """Render a pixel window (default: whole image) and optionally the gradients
    of sum(<grad_image, F>) over that window.  All values are fp64."""
    lib = _load()
    pos, radius, opacity = _f64(pos).reshape(-1, 3), _f64(radius), _f64(opacity)
    n = pos.shape[0]
    C, T = int(params.channels), int(params.n_track)
    features = _f64(features).reshape(n, C)
    bg = _f64(bg).reshape(C)
    if window is None:
        window = (0, 0, cam.width, cam.height)
    x0, y0, x1, y1 = (int(v) for v in window)
    h, w = y1 - y0, x1 - x0
    out = dict(image=np.zeros((h, w, C)), mg=np.zeros((h, w)), wsum=np.zeros((h, w)),
               ids=np.zeros((h, w, T), np.int32), nhits=np.zeros((h, w), np.int32))
    G = None
    gabs = None
    if grad_image is not None:
        G = _f64(grad_image).reshape(cam.height, cam.width, C)
        out.update(grad_pos=np.zeros((n, 3)), grad_radius=np.zeros(n),
                   grad_opacity=np.zeros(n), grad_features=np.zeros((n, C)),
                   grad_cam=np.zeros(16))
        gabs = np.zeros(2 * ((5 + C) * n + 16))
    c, q = _cam(cam), _params(params, fp64)
    H = lib.oracle_render(_ptr(pos), _ptr(radius), _ptr(opacity), _ptr(features), n,
                          ctypes.byref(c), ctypes.byref(q), _ptr(bg), x0, y0, x1, y1,
                          1 if brute else 0, _ptr(G), _ptr(out["image"]), _ptr(out["mg"]),
                          _ptr(out["wsum"]), _ptr(out["ids"]), _ptr(out["nhits"]),
                          _ptr(out.get("grad_pos")), _ptr(out.get("grad_radius")),
                          _ptr(out.get("grad_opacity")), _ptr(out.get("grad_features")),
                          _ptr(out.get("grad_cam")), _ptr(gabs))
    if H < 0:
        raise RuntimeError(f"oracle_render failed: {H}")
    if gabs is not None:
        # per gradient entry: sum over pixels of |per-pixel contribution| (abs_*)
        # and of its L1 sensitivity to the input image F (sens_*)
        L = (5 + C) * n + 16
        for pre, buf in (("abs_", gabs[:L]), ("sens_", gabs[L:])):
            out[pre + "grad_pos"] = buf[:3 * n].reshape(n, 3)
            out[pre + "grad_radius"] = buf[3 * n:4 * n]
            out[pre + "grad_opacity"] = buf[4 * n:5 * n]
            out[pre + "grad_features"] = buf[5 * n:(5 + C) * n].reshape(n, C)
            out[pre + "grad_cam"] = buf[(5 + C) * n:]
    out["hits"] = int(H)
    return out


def render_scene(scene, cam_index: int = 0, with_grads: bool = True, **kw) -> dict:
    """Convenience wrapper over a scene object (duck-typed: pos, radius,
    opacity, features, cameras, params, bg, grad_images)."""
    cam = scene.cameras[cam_index]
    G = scene.grad_images[cam_index] if with_grads else None
    return render(scene.pos, scene.radius, scene.opacity, scene.features, cam, scene.params,
                  scene.bg, grad_image=G, **kw)
