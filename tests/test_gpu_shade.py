"""Per-pixel shading MLP on the tensor cores (pulsar_shade_forward) against
the oracle (oracle/mlp.py) on seeded inputs.

Tolerance, derived from the arithmetic: both sides round the same operands
to bfloat16 and multiply them exactly; the GPU sums in fp32 (error below
1e-5 of the sum of absolute products) where the oracle sums in fp64.  That
difference can move a hidden activation across a bfloat16 rounding boundary
(or a pre-activation across 0): such pixels are rare and bounded by one
bfloat16 ulp (2^-8 relative) of every hidden activation, propagated.
"""
from __future__ import annotations

import numpy as np
import pytest

from oracle import mlp
from splat_rendering_gb300 import scenes

pytestmark = pytest.mark.gpu


def _bounds(ref, params):
    """Per-pixel tight and one-ulp bounds on |y_gpu - y_oracle| [P, 3]."""
    P = mlp.unpack(params)
    W3 = np.abs(mlp.bf16(P["W3"]))
    W2 = np.abs(mlp.bf16(P["W2"]))
    W1 = np.abs(mlp.bf16(P["W1"]))
    a1 = np.abs(ref["x"]) @ W1.T + np.abs(np.asarray(P["b1"], np.float32))
    a2 = np.abs(ref["h1"]) @ W2.T + np.abs(np.asarray(P["b2"], np.float32))
    a3 = np.abs(ref["h2"]) @ W3.T + np.abs(np.asarray(P["b3"], np.float32))
    tight = 1e-5 * (a3 + (a2 @ W3.T) + (a1 @ W2.T) @ W3.T) + 1e-6
    ulp = 2.0 ** -8
    # one ulp in x, h1 and h2 (and the accumulation error), propagated to y
    flip = ulp * (a3 + a2 @ W3.T + a1 @ W2.T @ W3.T) + tight
    return tight, flip


def _check(rgb, ref, params, what):
    tight, flip = _bounds(ref, params)
    err = np.abs(rgb.reshape(-1, 3).astype(np.float64) - ref["y"])
    over = (err > tight).any(1)
    assert (err <= flip).all(), f"{what}: beyond the one-ulp bound (worst {(err / flip).max():.3g}x)"
    assert over.mean() < 2e-3, f"{what}: {over.sum()} of {len(over)} pixels past the tight bound"
    return int(over.sum())


def _renderer_for(cams, C=16):
    from splat_rendering_gb300 import pulsar as pl
    return pl.Renderer(max_spheres=16, max_pairs=1 << 12, max_width=cams[0].width,
                       max_height=cams[0].height, max_channels=C, max_track=8,
                       max_cams=len(cams))


def _project(r, cams, C=16):
    """The shading takes the frame's cameras: project an (empty) scene."""
    import torch
    from splat_rendering_gb300 import pulsar as pl
    z = torch.zeros(48, device="cuda")
    p = scenes.Params(n_track=8, channels=C)
    if len(cams) == 1:
        pl.project(r.ctx, z, z, z, 0, pl.camera(cams[0]), pl.params(p))
    else:
        pl.project_cams(r.ctx, z, z, z, 0, [pl.camera(c) for c in cams], pl.params(p))


@pytest.mark.parametrize("ortho", [False, True])
def test_shading_matches_oracle(ortho):
    import torch
    cam = scenes._camera(np.eye(3), np.zeros(3), 180.0, 200, 150, 1.0, 9.0, fy=170.0,
                         cx=97.3, cy=77.1, orthographic=ortho)
    rng = np.random.default_rng(121 + ortho)
    F = rng.standard_normal((cam.height, cam.width, 16)).astype(np.float32)
    params = scenes.shading_mlp(6)
    r = _renderer_for([cam])
    _project(r, [cam])
    rgb = r.shade(torch.from_numpy(F).cuda(), torch.from_numpy(params).cuda())
    code = r.status(raise_on_error=False)[0]
    assert code == 0
    ref = mlp.forward(F.reshape(-1, 16), cam, params.astype(np.float64))
    _check(rgb.cpu().numpy(), ref, params.astype(np.float64), f"shade ortho={ortho}")
    r.close()


def test_shading_camera_batch_and_ragged_tile():
    """Three cameras in one batch (view directions from each camera), and a
    pixel count that is not a multiple of the 128-pixel tile."""
    import torch
    cams = [scenes._camera(np.eye(3), np.zeros(3), f, 37, 29, 1.0, 9.0, cx=cx, cy=14.2)
            for f, cx in ((30.0, 18.1), (45.0, 10.0), (60.0, 25.5))]
    rng = np.random.default_rng(123)
    F = rng.standard_normal((3, 29, 37, 16)).astype(np.float32)
    params = scenes.shading_mlp(7)
    r = _renderer_for(cams)
    _project(r, cams)
    rgb = r.shade(torch.from_numpy(F).cuda(), torch.from_numpy(params).cuda()).cpu().numpy()
    assert r.status(raise_on_error=False)[0] == 0
    for k, cam in enumerate(cams):
        ref = mlp.forward(F[k].reshape(-1, 16), cam, params.astype(np.float64))
        _check(rgb[k], ref, params.astype(np.float64), f"camera {k}")
    r.close()


def test_shading_full_size_frame():
    """1024 x 1024 features (the neural configuration's image size)."""
    import torch
    sc = scenes.make("neural", n=1000)
    cam = sc.cameras[0]
    rng = np.random.default_rng(124)
    F = rng.standard_normal((cam.height, cam.width, 16)).astype(np.float32)
    params = scenes.shading_mlp(8)
    r = _renderer_for([cam])
    _project(r, [cam])
    rgb = r.shade(torch.from_numpy(F).cuda(), torch.from_numpy(params).cuda())
    assert r.status(raise_on_error=False)[0] == 0
    ref = mlp.forward(F.reshape(-1, 16), cam, params.astype(np.float64))
    n = _check(rgb.cpu().numpy(), ref, params.astype(np.float64), "full size")
    print("pixels past the tight bound:", n)
    r.close()
