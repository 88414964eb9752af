"""Pins of the per-pixel shading MLP oracle (Pulsar Sec. 3.3, 5.2; reading in
oracle/mlp.py) against facts fixed outside it.  No GPU."""
from __future__ import annotations

import numpy as np
import pytest

import closed_form as cf
from oracle import mlp
from splat_rendering_gb300 import scenes


def _cam(W=24, H=20, ortho=False):
    return scenes._camera(np.eye(3), np.zeros(3), 30.0 if not ortho else 8.0, W, H, 1.0, 9.0,
                          fy=27.0, cx=11.3, cy=9.7, orthographic=ortho)


def test_bf16_rounding_matches_torch():
    """Round to nearest, ties to even, from float32 (torch's bfloat16)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-30, 30, 5000),
                        np.array([1.00390625, 1.01171875, 1.0 + 3 * 2 ** -9, -1.00390625,
                                  0.0, -0.0, 1e-40, 65519.0, 3.3895e38])])
    ref = torch.tensor(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(mlp.bf16(v), ref)


def test_view_directions():
    """Unit rays through the pixel centres (pinhole), +z (orthographic)."""
    cam = _cam()
    v = mlp.view_dirs(cam)
    q = cf.pixel_rays(cam).reshape(-1, 3)
    assert np.allclose(v, q / np.linalg.norm(q, axis=1, keepdims=True), rtol=0, atol=1e-15)
    assert np.array_equal(mlp.view_dirs(_cam(ortho=True)), np.tile([0.0, 0.0, 1.0], (480, 1)))


def test_linear_regime_is_one_composed_affine_map():
    """With the ReLUs inactive (large biases) the network is the affine map
    (W3 W2 W1) x + (W3 W2 b1 + W3 b2 + b3): matrices composed first, a
    different evaluation order than the layer-by-layer oracle."""
    cam = _cam()
    rng = np.random.default_rng(1)
    p = mlp.unpack(scenes.shading_mlp(3).astype(np.float64))
    p["b1"] = np.full(64, 50.0)
    p["b2"] = np.full(64, 500.0)
    flat = mlp.pack(p)
    F = rng.uniform(0, 1, (cam.width * cam.height, 16))
    out = mlp.forward(F, cam, flat, exact=True)
    assert (out["z1"] > 0).all() and (out["z2"] > 0).all()
    x = np.concatenate([F, mlp.view_dirs(cam)], 1)
    A = p["W3"] @ p["W2"] @ p["W1"]
    c = p["W3"] @ p["W2"] @ p["b1"].astype(np.float32) + p["W3"] @ p["b2"].astype(np.float32) + \
        p["b3"].astype(np.float32)
    assert np.allclose(out["y"], x @ A.T + c, rtol=1e-12, atol=1e-9)


def test_gradients_match_central_differences():
    """Exact-mode gradients of L = sum <dY, y> w.r.t. the features and every
    weight and bias agree with central finite differences (away from ReLU
    kinks: a check whose two step sizes disagree is skipped)."""
    cam = _cam(12, 10)
    rng = np.random.default_rng(2)
    params = scenes.shading_mlp(4).astype(np.float64)
    F = rng.uniform(-1, 1, (cam.width * cam.height, 16))
    dY = rng.standard_normal((cam.width * cam.height, 3))
    g = mlp.backward(F, cam, params, dY, exact=True)

    def loss(Fv, pv):
        return float((mlp.forward(Fv, cam, pv, exact=True)["y"] * dY).sum())

    def fd(which, idx, h):
        a = F.copy() if which == "F" else params.copy()
        b = a.copy()
        a[idx] += h
        b[idx] -= h
        la = loss(a, params) if which == "F" else loss(F, a)
        lb = loss(b, params) if which == "F" else loss(F, b)
        return (la - lb) / (2 * h)

    bad, checked = [], 0
    for which, ref, idxs in (("F", g["grad_features"], [tuple(rng.integers(0, s) for s in F.shape)
                                                       for _ in range(40)]),
                             ("P", g["grad_params"], [(int(i),) for i in
                                                      rng.choice(mlp.N_PARAMS, 120, replace=False)]
                              + [(mlp.N_PARAMS - 1,), (0,)])):
        for idx in idxs:
            f1, f2 = fd(which, idx, 1e-5), fd(which, idx, 2.5e-6)
            if abs(f1 - f2) > 1e-6 * (abs(f1) + 1):
                continue
            checked += 1
            if abs(ref[idx] - f2) > 1e-6 * (abs(f2) + 1):
                bad.append((which, idx, ref[idx], f2))
    assert not bad, bad
    assert checked > 120


def test_quantised_mode_rounds_every_operand():
    """In the tensor-core mode every matrix operand is a bfloat16 value."""
    cam = _cam()
    rng = np.random.default_rng(3)
    out = mlp.backward(rng.uniform(0, 1, (480, 16)), cam, scenes.shading_mlp(), rng.standard_normal((480, 3)))
    for k in ("x", "h1", "h2"):
        assert np.array_equal(mlp.bf16(out[k]), out[k]), k
