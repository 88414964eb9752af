"""The shading MLP's parity bounds (tests/shade_bounds.py) on the CPU: an
fp32 emulation of the tensor-core arithmetic -- the same bf16 operands, fp32
sums in another order, fp32 view directions -- lies inside them, and the
same emulation with a planted mistake does not."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import mlp
from splat_rendering_gb300 import scenes
import shade_bounds as sb

f32 = np.float32


def _q32(v):
    return mlp.bf16(v).astype(f32)


def _emulate(F, cam, params, dY, plant=None):
    """fp32 stand-in for the GPU kernels (bf16 operands, fp32 sums)."""
    P = {k: np.asarray(v, f32) for k, v in mlp.unpack(params).items()}
    W1, W2, W3 = (_q32(P[k]) for k in ("W1", "W2", "W3"))
    H, W = cam.height, cam.width
    a = (np.arange(W, dtype=f32) + f32(0.5) - f32(cam.cx)) / f32(cam.fx)
    b = (np.arange(H, dtype=f32) + f32(0.5) - f32(cam.cy)) / f32(cam.fy)
    A, B = np.meshgrid(a, b)
    inv = f32(1) / np.sqrt(A * A + B * B + f32(1))
    v = np.stack([A * inv, B * inv, inv], -1).reshape(-1, 3).astype(f32)
    if plant == "no view direction":
        v = np.zeros_like(v)
    x = _q32(np.concatenate([F.reshape(-1, 16).astype(f32), v], 1))
    z1 = x @ W1.T + P["b1"]
    h1 = _q32(np.maximum(z1, 0))
    if plant == "h1 one bf16 ulp high":
        h1 = _q32(h1 * f32(1 + 2.0 ** -7))
    z2 = h1 @ W2.T + (P["b2"] if plant != "drop b2" else f32(0))
    h2 = _q32(np.maximum(z2, 0))
    y = h2 @ W3.T + P["b3"]
    dy = _q32(dY.reshape(-1, 3))
    g2 = _q32((dy @ W3) * (z2 > 0))
    g1 = _q32((g2 @ W2) * (z1 > 0))
    dF = g1 @ W1[:, :16]
    if plant == "transpose W2 in the backward":
        g1 = _q32((g2 @ W2.T) * (z1 > 0))
    grads = dict(W1=g1.T @ x[:, :19], b1=g1.sum(0), W2=g2.T @ h1, b2=g2.sum(0),
                 W3=dy.T @ h2, b3=dy.sum(0))
    if plant == "bias rows swapped":
        grads["b1"], grads["b2"] = grads["b2"], grads["b1"]
    if plant == "one pixel missing":
        grads["W2"] = g2[1:].T @ h1[1:]
    return dict(y=y, dF=dF, params=mlp.pack(grads))


def _case(seed, ortho=False, H=40, W=56):
    cam = scenes._camera(np.eye(3), np.zeros(3), 50.0, W, H, 1.0, 9.0, fy=47.0, cx=27.3,
                         cy=19.1, orthographic=ortho)
    rng = np.random.default_rng(seed)
    F = rng.standard_normal((H, W, 16)).astype(f32)
    dY = rng.standard_normal((H, W, 3)).astype(f32)
    params = scenes.shading_mlp(seed).astype(np.float64)
    ref = sb.oracle_batch(F[None], [cam], params, dY[None])
    return cam, F, dY, params, ref


def test_fp32_emulation_inside_bounds():
    cam, F, dY, params, ref = _case(41)
    stats = sb.check(_emulate(F, cam, params, dY), ref, params, "emulation")
    # the bounds are not vacuous: their typical radius is far below the values
    for key, (_, med) in stats.items():
        assert med < 5e-3, (key, med)


@pytest.mark.parametrize("plant", ["drop b2", "transpose W2 in the backward",
                                   "one pixel missing", "h1 one bf16 ulp high",
                                   "no view direction", "bias rows swapped"])
def test_planted_mistake_outside_bounds(plant):
    cam, F, dY, params, ref = _case(42)
    with pytest.raises(AssertionError):
        sb.check(_emulate(F, cam, params, dY, plant), ref, params, plant)
