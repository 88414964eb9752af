"""Error bounds for the tensor-core shading MLP against the oracle
(oracle/mlp.py), derived from the arithmetic.

Both sides round the same operands to bfloat16 and multiply them exactly;
the GPU sums each dot product in fp32 (at most 64 terms: error below
REL = 3e-5 of the sum of absolute products and bias, with margin over
64 * 2^-23) where the oracle sums in fp64.  That difference can move a value
across a bfloat16 rounding boundary or a pre-activation across 0, and the
moved value then feeds the next layer.  The bounds follow every value as an
interval around the oracle's: a rounding or ReLU decision whose input
interval straddles a boundary widens the output interval to every result it
could take, and the widening propagates through the absolute weights.  The
weight gradients add ACC = 1e-4 of their absolute sums for the fp32
accumulation over a CTA's pixels.  A GPU value outside its interval is an
error, not rounding.
"""
from __future__ import annotations

import numpy as np

from oracle import mlp

REL = 3e-5
ACC = 1e-4


def _hull_q(center_q, lo, hi):
    """Radius around the rounded centre of the bf16 roundings of [lo, hi]."""
    return np.maximum(center_q - mlp.bf16(lo), mlp.bf16(hi) - center_q)


def _masked(pre, r_pre, z, r_z):
    """Interval of pre * [z > 0] with pre known within r_pre and z within r_z."""
    on, off = z - r_z > 0, z + r_z <= 0
    lo = np.where(on, pre - r_pre, np.where(off, 0.0, np.minimum(0.0, pre - r_pre)))
    hi = np.where(on, pre + r_pre, np.where(off, 0.0, np.maximum(0.0, pre + r_pre)))
    return lo, hi


def radii(ref, params, vdirs, backward: bool = True) -> dict:
    """Radii of y [P, 3] and, with backward, dF [P, 16] and the flat weight
    gradient, around the oracle's values (and under 'scale_<key>' the sums of
    absolute terms they are measured against).  ref: the oracle's backward (or
    forward) dict for the same pixels; vdirs [P, 3]: the unrounded view
    directions (the GPU computes them in fp32, a few ulp off)."""
    P = mlp.unpack(params)
    Wq = {k: mlp.bf16(P[k]) for k in ("W1", "W2", "W3")}
    W1, W2, W3 = (np.abs(Wq[k]) for k in ("W1", "W2", "W3"))
    b1, b2, b3 = (np.abs(np.asarray(P[k], np.float32)) for k in ("b1", "b2", "b3"))
    x, z1, h1, z2, h2 = (ref[k] for k in ("x", "z1", "h1", "z2", "h2"))
    rx = np.zeros_like(x)
    t = 1e-6 * np.abs(vdirs) + 1e-12
    rx[:, 16:19] = _hull_q(x[:, 16:19], vdirs - t, vdirs + t)
    rz1 = REL * (np.abs(x) @ W1.T + b1) + rx @ W1.T
    rh1 = _hull_q(h1, np.maximum(z1 - rz1, 0.0), np.maximum(z1 + rz1, 0.0))
    rz2 = REL * (np.abs(h1) @ W2.T + b2) + rh1 @ W2.T
    rh2 = _hull_q(h2, np.maximum(z2 - rz2, 0.0), np.maximum(z2 + rz2, 0.0))
    scale_y = np.abs(h2) @ W3.T + b3
    out = dict(y=REL * scale_y + rh2 @ W3.T, scale_y=scale_y)
    if not backward:
        return out
    dy = ref["dy"]
    lo, hi = _masked(dy @ Wq["W3"], REL * (np.abs(dy) @ W3), z2, rz2)
    g2q = mlp.bf16(ref["g2"])
    rg2 = _hull_q(g2q, lo, hi)
    lo, hi = _masked(g2q @ Wq["W2"], REL * (np.abs(g2q) @ W2) + rg2 @ W2, z1, rz1)
    g1q = mlp.bf16(ref["g1"])
    rg1 = _hull_q(g1q, lo, hi)
    out["scale_dF"] = np.abs(g1q) @ W1[:, :16]
    out["dF"] = REL * out["scale_dF"] + rg1 @ W1[:, :16]
    out["scale_params"] = ref["abs_params"]
    out["params"] = ACC * ref["abs_params"] + mlp.pack(dict(
        W1=np.abs(g1q).T @ rx + rg1.T @ (np.abs(x) + rx), b1=rg1.sum(0),
        W2=np.abs(g2q).T @ rh1 + rg2.T @ (np.abs(h1) + rh1), b2=rg2.sum(0),
        W3=np.abs(dy).T @ rh2, b3=np.zeros(3)))
    return out


def oracle_batch(F, cams, params, dY=None) -> dict:
    """The oracle over a batch of cameras, pixels camera after camera (the
    weight gradients summed); F [K, ..., 16], dY [K, ..., 3] or None (forward
    only).  Adds the unrounded view directions as 'vdirs'."""
    if dY is None:
        outs = [mlp.forward(F[k].reshape(-1, 16), cam, params) for k, cam in enumerate(cams)]
    else:
        outs = [mlp.backward(F[k].reshape(-1, 16), cam, params, dY[k].reshape(-1, 3))
                for k, cam in enumerate(cams)]
    ref = {key: np.concatenate([o[key] for o in outs], 0)
           for key, v in outs[0].items() if np.ndim(v) == 2 and key != "grad_params"}
    if dY is not None:
        ref["grad_params"] = sum(o["grad_params"] for o in outs)
        ref["abs_params"] = sum(o["abs_params"] for o in outs)
    ref["vdirs"] = np.concatenate([mlp.view_dirs(cam) for cam in cams], 0)
    return ref


def check(got: dict, ref: dict, params, what: str, backward: bool = True) -> dict:
    """Assert every GPU value lies in its interval; returns per-quantity
    statistics (worst error / radius, median radius / absolute scale)."""
    r = radii(ref, params, ref["vdirs"], backward)
    stats = {}
    for key in ("y", "dF", "params"):
        if key not in got or key not in r:
            continue
        want = {"y": ref["y"] if "y" in ref else None, "dF": ref.get("grad_features"),
                "params": ref.get("grad_params")}[key]
        g = np.asarray(got[key], np.float64).reshape(want.shape)
        err = np.abs(g - want)
        bound = r[key] * (1 + 1e-9) + 1e-12
        bad = err > bound
        if bad.any():
            i = np.unravel_index(np.argmax(err / bound), err.shape)
            raise AssertionError(f"{what}: {key} {int(bad.sum())} values outside the bound; worst "
                                 f"at {tuple(int(v) for v in i)}: got {g[i]:.9g}, oracle "
                                 f"{want[i]:.9g}, radius {r[key][i]:.3g}")
        stats[key] = (float((err / bound).max()),
                      float(np.median(r[key] / (r["scale_" + key] + 1e-30))))
    return stats
