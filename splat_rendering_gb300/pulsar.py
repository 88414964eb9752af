"""Python binding of the C ABI in include/pulsar.h (argument marshalling only).

Every step of the rendering path runs in the CUDA kernels of libpulsar.so.
There is no CPU fallback: if the library is missing, loading raises.
PyTorch is used only for device memory and streams.

Functions mirror the C entry points:
    create, destroy, project, bin, forward, backward, status, strerror,
    debug_copy
Tensor arguments are CUDA torch tensors (float32, contiguous) or raw device
pointers (int); streams are torch.cuda.Stream objects, raw handles (int) or
None for the current torch stream.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpulsar.so")

OK, ERR_ARG, ERR_CUDA, ERR_CAPACITY, ERR_STATE, ERR_NOMEM, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5, -6
ERR_INTERNAL = -7   # debug build: a device index check failed
FLAG_GEOM_CUTOFF = 0x1
FLAG_COUNT_HITS = 0x2
FLAG_NORMALIZE_GRADS = 0x4
FLAG_GAUSSIAN = 0x8
DBG = dict(records=1, tile_offsets=5, tile_ids=6, mg=7, wsum=8, ids=9, nhits=10)

_lib = None


class PulsarError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


class Camera(ctypes.Structure):
    _fields_ = [("R", ctypes.c_float * 9), ("t", ctypes.c_float * 3),
                ("fx", ctypes.c_float), ("fy", ctypes.c_float), ("cx", ctypes.c_float),
                ("cy", ctypes.c_float), ("width", ctypes.c_int32), ("height", ctypes.c_int32),
                ("znear", ctypes.c_float), ("zfar", ctypes.c_float),
                ("orthographic", ctypes.c_int32)]


class Params(ctypes.Structure):
    _fields_ = [("gamma", ctypes.c_float), ("bg_eps", ctypes.c_float),
                ("stop_tau", ctypes.c_float), ("kappa", ctypes.c_float),
                ("geom_min_area", ctypes.c_float), ("n_track", ctypes.c_int32),
                ("channels", ctypes.c_int32), ("flags", ctypes.c_uint32)]


EXPORTS = ("pulsar_create", "pulsar_create_cams", "pulsar_destroy", "pulsar_project",
           "pulsar_project_cams", "pulsar_bin", "pulsar_shade_forward", "pulsar_shade_backward",
           "pulsar_forward", "pulsar_backward", "pulsar_status", "pulsar_strerror",
           "pulsar_debug_copy", "pulsar_debug_inject", "pulsar_render_noalloc")


def load(path: str = LIB_PATH):
    """Load libpulsar.so and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m splat_rendering_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.pulsar_create.argtypes = [ctypes.POINTER(P), ctypes.c_int, I64, I64, I32, I32, I32, I32]
    lib.pulsar_create_cams.argtypes = [ctypes.POINTER(P), ctypes.c_int, I64, I64, I32, I32, I32,
                                       I32, I32]
    lib.pulsar_destroy.argtypes = [P]
    lib.pulsar_project.argtypes = [P, P, P, P, I64, ctypes.POINTER(Camera),
                                   ctypes.POINTER(Params), P]
    lib.pulsar_project_cams.argtypes = [P, P, P, P, I64, ctypes.POINTER(Camera), I32,
                                        ctypes.POINTER(Params), P]
    lib.pulsar_bin.argtypes = [P, P]
    lib.pulsar_shade_forward.argtypes = [P, P, P, P, P]
    lib.pulsar_shade_backward.argtypes = [P] * 7
    lib.pulsar_forward.argtypes = [P, P, P, P, P]
    lib.pulsar_backward.argtypes = [P] + [P] * 9 + [P]
    lib.pulsar_status.argtypes = [P, P, ctypes.POINTER(I64), ctypes.POINTER(I64)]
    lib.pulsar_strerror.argtypes = [ctypes.c_int]
    lib.pulsar_strerror.restype = ctypes.c_char_p
    lib.pulsar_debug_copy.argtypes = [P, ctypes.c_int, P, I64, P]
    lib.pulsar_debug_inject.argtypes = [P, ctypes.c_int, P]
    lib.pulsar_debug_copy.restype = I64
    lib.pulsar_render_noalloc.argtypes = [P, P, P, P, I64, ctypes.POINTER(Camera),
                                          ctypes.POINTER(Params), P, P, P]
    for name in EXPORTS:
        if name not in ("pulsar_strerror", "pulsar_debug_copy"):
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def strerror(code: int) -> str:
    return load().pulsar_strerror(int(code)).decode()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(code: int, what: str):
    if code != OK:
        raise PulsarError(code, what)


def camera(cam) -> Camera:
    """Camera struct from any object with R, t, fx, fy, cx, cy, width, height,
    znear, zfar attributes (and optionally orthographic)."""
    c = Camera()
    c.R[:] = [float(v) for v in np.asarray(cam.R, np.float32).reshape(9)]
    c.t[:] = [float(v) for v in np.asarray(cam.t, np.float32).reshape(3)]
    for k in ("fx", "fy", "cx", "cy", "znear", "zfar"):
        setattr(c, k, float(getattr(cam, k)))
    c.width, c.height = int(cam.width), int(cam.height)
    c.orthographic = 1 if getattr(cam, "orthographic", False) else 0
    return c


def params(p, count_hits: bool = False) -> Params:
    """Params struct from any object with gamma, bg_eps, stop_tau, kappa,
    geom_min_area, n_track, channels, geom_cutoff (and optionally
    normalize_grads, gaussian) attributes."""
    q = Params()
    q.gamma, q.bg_eps, q.stop_tau = float(p.gamma), float(p.bg_eps), float(p.stop_tau)
    q.kappa, q.geom_min_area = float(p.kappa), float(p.geom_min_area)
    q.n_track, q.channels = int(p.n_track), int(p.channels)
    q.flags = (FLAG_GEOM_CUTOFF if getattr(p, "geom_cutoff", True) else 0) | \
              (FLAG_COUNT_HITS if count_hits else 0) | \
              (FLAG_NORMALIZE_GRADS if getattr(p, "normalize_grads", False) else 0) | \
              (FLAG_GAUSSIAN if getattr(p, "gaussian", False) else 0)
    return q


# ------------------------------------------------------------ C entry points --
def create(device: int, max_spheres: int, max_pairs: int, max_width: int, max_height: int,
           max_channels: int, max_track: int, max_cams: int = 1) -> int:
    h = ctypes.c_void_p()
    if max_cams == 1:
        _check(load().pulsar_create(ctypes.byref(h), device, max_spheres, max_pairs, max_width,
                                    max_height, max_channels, max_track), "pulsar_create")
    else:
        _check(load().pulsar_create_cams(ctypes.byref(h), device, max_spheres, max_pairs,
                                         max_width, max_height, max_channels, max_track,
                                         max_cams), "pulsar_create_cams")
    return h.value


def destroy(ctx: int):
    _check(load().pulsar_destroy(ctx), "pulsar_destroy")


def project(ctx, pos, radius, opacity, n: int, cam: Camera, prm: Params, stream=None):
    _check(load().pulsar_project(ctx, _ptr(pos), _ptr(radius), _ptr(opacity), int(n),
                                 ctypes.byref(cam), ctypes.byref(prm), _stream(stream)),
           "pulsar_project")


def project_cams(ctx, pos, radius, opacity, n: int, cams, prm: Params, stream=None):
    """Project the spheres for a batch of cameras (list of Camera structs)."""
    arr = (Camera * len(cams))(*cams)
    _check(load().pulsar_project_cams(ctx, _ptr(pos), _ptr(radius), _ptr(opacity), int(n), arr,
                                      len(cams), ctypes.byref(prm), _stream(stream)),
           "pulsar_project_cams")


def shade_forward(ctx, features, params, rgb, stream=None):
    """Per-pixel shading MLP of the frame's feature images (see
    pulsar_shade_forward in include/pulsar.h)."""
    _check(load().pulsar_shade_forward(ctx, _ptr(features), _ptr(params), _ptr(rgb),
                                       _stream(stream)), "pulsar_shade_forward")


def shade_backward(ctx, features, params, grad_rgb, grad_features, grad_params, stream=None):
    """Gradients of the shading MLP (see pulsar_shade_backward in
    include/pulsar.h); grad_features may be None."""
    _check(load().pulsar_shade_backward(ctx, _ptr(features), _ptr(params), _ptr(grad_rgb),
                                        _ptr(grad_features), _ptr(grad_params),
                                        _stream(stream)), "pulsar_shade_backward")


def bin(ctx, stream=None):  # noqa: A001  (same name as the C entry point)
    _check(load().pulsar_bin(ctx, _stream(stream)), "pulsar_bin")


def forward(ctx, features, bg, image, stream=None):
    _check(load().pulsar_forward(ctx, _ptr(features), _ptr(bg), _ptr(image), _stream(stream)),
           "pulsar_forward")


def backward(ctx, features, bg, image, grad_image, grad_pos=None, grad_radius=None,
             grad_opacity=None, grad_features=None, grad_cam=None, stream=None):
    _check(load().pulsar_backward(ctx, _ptr(features), _ptr(bg), _ptr(image), _ptr(grad_image),
                                  _ptr(grad_pos), _ptr(grad_radius), _ptr(grad_opacity),
                                  _ptr(grad_features), _ptr(grad_cam), _stream(stream)),
           "pulsar_backward")


def status(ctx, stream=None, raise_on_error: bool = True):
    """(code, n_pairs, n_hits) after synchronising the stream."""
    m, h = ctypes.c_int64(), ctypes.c_int64()
    code = load().pulsar_status(ctx, _stream(stream), ctypes.byref(m), ctypes.byref(h))
    if raise_on_error:
        _check(code, "pulsar_status")
    return code, m.value, h.value


def render_noalloc(pos, radius, opacity, features, n: int, cam: Camera, prm: Params, bg, image,
                   stream=None):
    """Forward render of a small frame without any memory allocation (see
    pulsar_render_noalloc in include/pulsar.h for its limits).  For callers
    that cannot allocate device memory at render time; synchronises the stream."""
    _check(load().pulsar_render_noalloc(_ptr(pos), _ptr(radius), _ptr(opacity), _ptr(features),
                                        int(n), ctypes.byref(cam), ctypes.byref(prm), _ptr(bg),
                                        _ptr(image), _stream(stream)), "pulsar_render_noalloc")


def debug_copy(ctx, what: str, stream=None) -> np.ndarray:
    """Copy an internal array of the last frame to a numpy array (raw bytes)."""
    lib = load()
    size = lib.pulsar_debug_copy(ctx, DBG[what], None, 0, _stream(stream))
    if size < 0:
        raise PulsarError(int(size), "pulsar_debug_copy")
    buf = np.empty(max(size, 1), np.uint8)
    code = lib.pulsar_debug_copy(ctx, DBG[what], buf.ctypes.data_as(ctypes.c_void_p), size,
                                 _stream(stream))
    _check(int(code), "pulsar_debug_copy")
    return buf[:size]


# ---------------------------------------------------------------- helper --
class Renderer:
    """One context and its call sequence for torch tensors on one device.

        r = Renderer(max_spheres=..., max_pairs=..., max_width=..., max_height=...)
        image = r.render(pos, radius, opacity, features, cam, prm, bg)
        grads = r.backward(grad_image)
    """

    def __init__(self, max_spheres: int, max_pairs: int, max_width: int, max_height: int,
                 max_channels: int = 3, max_track: int = 8, device: int = 0,
                 max_cams: int = 1):
        self.device = device
        self.ctx = create(device, max_spheres, max_pairs, max_width, max_height, max_channels,
                          max_track, max_cams)
        self._frame = None

    def close(self):
        if self.ctx:
            destroy(self.ctx)
            self.ctx = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def render(self, pos, radius, opacity, features, cam, prm: Params, bg, image=None,
               stream=None):
        """Render one camera (a Camera struct; image [H,W,C]) or a batch (a list
        of Camera structs of equal size; image [K,H,W,C])."""
        import torch
        n = int(pos.shape[0])
        C = int(prm.channels)
        batch = isinstance(cam, (list, tuple))
        first = cam[0] if batch else cam
        shape = ((len(cam),) if batch else ()) + (first.height, first.width, C)
        if image is None:
            image = torch.empty(shape, device=f"cuda:{self.device}", dtype=torch.float32)
        if batch:
            project_cams(self.ctx, pos, radius, opacity, n, list(cam), prm, stream)
        else:
            project(self.ctx, pos, radius, opacity, n, cam, prm, stream)
        bin(self.ctx, stream)
        forward(self.ctx, features, bg, image, stream)
        self._frame = (pos, features, bg, image, n, C, len(cam) if batch else 0)
        return image

    def backward(self, grad_image, want=("pos", "radius", "opacity", "features", "cam"),
                 out=None, stream=None):
        import torch
        pos, features, bg, image, n, C, K = self._frame
        dev = image.device
        if out is None:
            out = {}
            shapes = dict(pos=(n, 3), radius=(n,), opacity=(n,), features=(n, C),
                          cam=(K, 16) if K else (16,))
            for k in want:
                out[k] = torch.empty(shapes[k], device=dev, dtype=torch.float32)
        backward(self.ctx, features, bg, image, grad_image, out.get("pos"), out.get("radius"),
                 out.get("opacity"), out.get("features"), out.get("cam"), stream)
        return out

    def shade(self, features, params, rgb=None, stream=None):
        """RGB of the per-pixel shading MLP over feature images [..., H, W, 16]
        of the current frame's camera(s)."""
        import torch
        if rgb is None:
            rgb = torch.empty(tuple(features.shape[:-1]) + (3,), device=features.device,
                              dtype=torch.float32)
        shade_forward(self.ctx, features, params, rgb, stream)
        return rgb

    def shade_backward(self, features, params, grad_rgb, grad_features=None, grad_params=None,
                       stream=None):
        """(dL/dfeatures, dL/dparams) of the shading for dL/drgb."""
        import torch
        if grad_features is None:
            grad_features = torch.empty_like(features)
        if grad_params is None:
            grad_params = torch.empty_like(params)
        shade_backward(self.ctx, features, params, grad_rgb, grad_features, grad_params, stream)
        return grad_features, grad_params

    def status(self, stream=None, raise_on_error: bool = True):
        return status(self.ctx, stream, raise_on_error)

    def debug(self, what: str, stream=None) -> np.ndarray:
        return debug_copy(self.ctx, what, stream)


INJECT_SHADE_TIMEOUT = 1


def debug_inject(ctx, what: int, stream=None):
    """Arm a test failure (see pulsar_debug_inject in include/pulsar.h)."""
    _check(load().pulsar_debug_inject(ctx, int(what), _stream(stream)), "pulsar_debug_inject")
