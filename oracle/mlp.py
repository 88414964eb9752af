"""Per-pixel shading MLP -- TEST INFRASTRUCTURE (CPU oracle, numpy fp64).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.

What it computes (Pulsar: Efficient Sphere-based Neural Rendering, the
paperlayer.ai summary of arXiv 2004.07484, Sec. 3.3 "Neural Shading": a
per-pixel network turns the rendered feature map into RGB; Sec. 5.2: a
shared per-pixel fully-connected model conditioned on the pixel's view
direction).  The pages give no architecture; reading:

  x  = [F_p (16 rendered channels), v_p (unit view direction, camera space)]
  h1 = ReLU(W1 x + b1)        W1 [64, 19]
  h2 = ReLU(W2 h1 + b2)       W2 [64, 64]
  y  = W3 h2 + b3             W3 [3, 64]    (RGB, linear)

computed the tensor-core way: every matrix operand (x, h1, h2, the weights,
and in the backward dY, g2, g1) is rounded to bfloat16 (round to nearest
even, from its float32 value), products are exact and sums are taken in
fp64 here (fp32 on the GPU), biases stay float32.  The backward of
L = sum_p <dY_p, y_p> treats the roundings as identities (straight
through):

  g2 = (W3^T Q(dY)) * [z2 > 0],   g1 = (W2^T Q(g2)) * [z1 > 0],
  dx = W1^T Q(g1)                 (dF = dx[:16]),
  dW3 = sum_p Q(dY) Q(h2)^T, dW2 = sum_p Q(g2) Q(h1)^T, dW1 = sum_p Q(g1) Q(x)^T,
  db3 = sum_p Q(dY), db2 = sum_p Q(g2), db1 = sum_p Q(g1).

``exact=True`` skips every rounding (the plain fp64 network; used by the
finite-difference pins).  Weights travel as one flat float32 vector in the
order W1, b1, W2, b2, W3, b3 (row-major).
"""
from __future__ import annotations

import numpy as np

N_FEAT, N_VIEW, N_IN, N_HID, N_OUT = 16, 3, 19, 64, 3
SHAPES = (("W1", (N_HID, N_IN)), ("b1", (N_HID,)), ("W2", (N_HID, N_HID)), ("b2", (N_HID,)),
          ("W3", (N_OUT, N_HID)), ("b3", (N_OUT,)))
N_PARAMS = sum(int(np.prod(s)) for _, s in SHAPES)


def unpack(flat):
    flat = np.asarray(flat, np.float64).reshape(-1)
    assert flat.size == N_PARAMS
    out, at = {}, 0
    for name, shape in SHAPES:
        k = int(np.prod(shape))
        out[name] = flat[at:at + k].reshape(shape)
        at += k
    return out


def pack(parts) -> np.ndarray:
    return np.concatenate([np.asarray(parts[name], np.float64).reshape(-1) for name, _ in SHAPES])


def bf16(v):
    """Round to bfloat16 (nearest, ties to even) from the value's float32
    rounding, returned as fp64."""
    f = np.asarray(v, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    nan = np.isnan(f)
    out = (r & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32).astype(np.float64)
    return np.where(nan, np.nan, out)


def view_dirs(cam) -> np.ndarray:
    """Unit view direction of every pixel ray in camera space, [H*W, 3]
    (pinhole: (a, b, 1)/|.| with a = (x + 1/2 - cx)/fx, b = (y + 1/2 - cy)/fy;
    orthographic: (0, 0, 1))."""
    H, W = cam.height, cam.width
    if getattr(cam, "orthographic", False):
        return np.tile(np.array([0.0, 0.0, 1.0]), (H * W, 1))
    xs = (np.arange(W) + 0.5 - cam.cx) / cam.fx
    ys = (np.arange(H) + 0.5 - cam.cy) / cam.fy
    a, b = np.meshgrid(xs, ys)
    q = np.stack([a.reshape(-1), b.reshape(-1), np.ones(H * W)], 1)
    return q / np.linalg.norm(q, axis=1, keepdims=True)


def _q(v, exact):
    return v if exact else bf16(v)


def forward(features, cam, params, exact: bool = False) -> dict:
    """features [H*W, 16] -> dict(y [H*W, 3], and the activations)."""
    P = unpack(params)
    F = np.asarray(features, np.float64).reshape(-1, N_FEAT)
    x = np.concatenate([F, view_dirs(cam)], 1)
    W1, W2, W3 = (_q(P[k], exact) for k in ("W1", "W2", "W3"))
    # biases: float32 values (fp64 in the exact mode)
    b1, b2, b3 = (P[k] if exact else np.asarray(P[k], np.float32).astype(np.float64)
                  for k in ("b1", "b2", "b3"))
    xq = _q(x, exact)
    z1 = xq @ W1.T + b1
    h1 = _q(np.maximum(z1, 0.0), exact)
    z2 = h1 @ W2.T + b2
    h2 = _q(np.maximum(z2, 0.0), exact)
    y = h2 @ W3.T + b3
    return dict(y=y, x=xq, z1=z1, h1=h1, z2=z2, h2=h2)


def backward(features, cam, params, grad_y, exact: bool = False) -> dict:
    """Gradients of L = sum_p <grad_y_p, y_p>: dF [H*W, 16] and the flat
    weight gradient (same layout as params), plus their per-entry sums of
    absolute per-pixel contributions (the scale of any summation's rounding),
    the rounded dY and the unrounded g2, g1 (where a rounding decision lies)."""
    P = unpack(params)
    fw = forward(features, cam, params, exact)
    W1, W2, W3 = (_q(P[k], exact) for k in ("W1", "W2", "W3"))
    dy = _q(np.asarray(grad_y, np.float64).reshape(-1, N_OUT), exact)
    g2 = (dy @ W3) * (fw["z2"] > 0)
    g2q = _q(g2, exact)
    g1 = (g2q @ W2) * (fw["z1"] > 0)
    g1q = _q(g1, exact)
    dx = g1q @ W1
    grads = dict(W1=g1q.T @ fw["x"], b1=g1q.sum(0), W2=g2q.T @ fw["h1"], b2=g2q.sum(0),
                 W3=dy.T @ fw["h2"], b3=dy.sum(0))
    absg = dict(W1=np.abs(g1q).T @ np.abs(fw["x"]), b1=np.abs(g1q).sum(0),
                W2=np.abs(g2q).T @ np.abs(fw["h1"]), b2=np.abs(g2q).sum(0),
                W3=np.abs(dy).T @ np.abs(fw["h2"]), b3=np.abs(dy).sum(0))
    return dict(grad_features=dx[:, :N_FEAT], grad_params=pack(grads), abs_params=pack(absg),
                abs_features=np.abs(g1q) @ np.abs(W1)[:, :N_FEAT], dy=dy, g2=g2, g1=g1, **fw)
