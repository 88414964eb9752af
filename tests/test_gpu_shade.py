"""Per-pixel shading MLP on the tensor cores (pulsar_shade_forward,
pulsar_shade_backward) against the oracle (oracle/mlp.py) on seeded inputs.

Every GPU value must lie in the interval tests/shade_bounds.py derives from
the arithmetic (fp32 against fp64 sums of the same bf16 products, and every
rounding or ReLU decision that this difference can move).
"""
from __future__ import annotations

import numpy as np
import pytest

from splat_rendering_gb300 import scenes
import shade_bounds as sb

pytestmark = pytest.mark.gpu


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
    ref = sb.oracle_batch(F[None], [cam], params.astype(np.float64))
    sb.check(dict(y=rgb.cpu().numpy()), ref, params.astype(np.float64), f"shade ortho={ortho}",
             backward=False)
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
    ref = sb.oracle_batch(F, cams, params.astype(np.float64))
    sb.check(dict(y=rgb), ref, params.astype(np.float64), "camera batch", backward=False)
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
    ref = sb.oracle_batch(F[None], [cam], params.astype(np.float64))
    print(sb.check(dict(y=rgb.cpu().numpy()), ref, params.astype(np.float64), "full size",
                   backward=False))
    r.close()


# ------------------------------------------------------------------ backward --
def _run_backward(cams, F, dY, params):
    import torch
    r = _renderer_for(cams)
    _project(r, cams)
    Fd, Pd, dYd = (torch.from_numpy(a).cuda() for a in (F, params, dY))
    gF, gP = r.shade_backward(Fd, Pd, dYd)
    gP2 = torch.empty_like(gP)
    from splat_rendering_gb300 import pulsar as pl
    pl.shade_backward(r.ctx, Fd, Pd, dYd, None, gP2)   # dF skipped
    torch.cuda.synchronize()
    assert r.status(raise_on_error=False)[0] == 0
    gF, gP, gP2 = gF.cpu().numpy(), gP.cpu().numpy(), gP2.cpu().numpy()
    r.close()
    # the fixed summation order makes the weight gradient reproducible bit for bit
    assert np.array_equal(gP.view(np.uint32), gP2.view(np.uint32))
    return gF, gP


@pytest.mark.parametrize("ortho", [False, True])
def test_shading_backward_matches_oracle(ortho):
    cam = scenes._camera(np.eye(3), np.zeros(3), 180.0, 200, 150, 1.0, 9.0, fy=170.0,
                         cx=97.3, cy=77.1, orthographic=ortho)
    rng = np.random.default_rng(131 + ortho)
    F = rng.standard_normal((1, cam.height, cam.width, 16)).astype(np.float32)
    dY = rng.standard_normal((1, cam.height, cam.width, 3)).astype(np.float32)
    params = scenes.shading_mlp(9)
    gF, gP = _run_backward([cam], F, dY, params)
    ref = sb.oracle_batch(F, [cam], params.astype(np.float64), dY)
    print(sb.check(dict(dF=gF, params=gP), ref, params.astype(np.float64),
                   f"backward ortho={ortho}"))


def test_shading_backward_batch_many_tiles_per_cta():
    """Three 250 x 199 cameras: more tiles than resident CTAs (each CTA
    accumulates several tiles in tensor memory) and a ragged last tile."""
    cams = [scenes._camera(np.eye(3), np.zeros(3), f, 250, 199, 1.0, 9.0, cx=cx, cy=101.0)
            for f, cx in ((200.0, 120.0), (260.0, 131.5), (150.0, 100.0))]
    rng = np.random.default_rng(133)
    F = rng.standard_normal((3, 199, 250, 16)).astype(np.float32)
    dY = rng.standard_normal((3, 199, 250, 3)).astype(np.float32)
    params = scenes.shading_mlp(10)
    gF, gP = _run_backward(cams, F, dY, params)
    ref = sb.oracle_batch(F, cams, params.astype(np.float64), dY)
    print(sb.check(dict(dF=gF, params=gP), ref, params.astype(np.float64), "batch"))


def test_shading_backward_tiny_frame():
    """A 5 x 3 frame: one partly filled tile (rows past the frame add nothing)."""
    cam = scenes._camera(np.eye(3), np.zeros(3), 4.0, 5, 3, 1.0, 9.0, cx=2.6, cy=1.4)
    rng = np.random.default_rng(134)
    F = rng.standard_normal((1, 3, 5, 16)).astype(np.float32)
    dY = rng.standard_normal((1, 3, 5, 3)).astype(np.float32)
    params = scenes.shading_mlp(11)
    gF, gP = _run_backward([cam], F, dY, params)
    ref = sb.oracle_batch(F, [cam], params.astype(np.float64), dY)
    sb.check(dict(dF=gF, params=gP), ref, params.astype(np.float64), "tiny")


def test_shading_backward_full_size_frame():
    """1024 x 1024 (the neural configuration's image size): every CTA runs
    many tiles, the weight gradient sums a million pixels."""
    sc = scenes.make("neural", n=1000)
    cam = sc.cameras[0]
    rng = np.random.default_rng(135)
    F = rng.standard_normal((1, cam.height, cam.width, 16)).astype(np.float32)
    dY = rng.standard_normal((1, cam.height, cam.width, 3)).astype(np.float32)
    params = scenes.shading_mlp(12)
    gF, gP = _run_backward([cam], F, dY, params)
    ref = sb.oracle_batch(F, [cam], params.astype(np.float64), dY)
    print(sb.check(dict(dF=gF, params=gP), ref, params.astype(np.float64), "full size"))


def test_shading_errors_and_empty_frame():
    """Call order, channel count and alignment errors; a frame whose pixel
    count is 0 cannot be made (the ABI rejects width 0), so the smallest frame
    (1 x 1, one partly filled tile) stands for it."""
    import torch
    from splat_rendering_gb300 import pulsar as pl
    params = torch.from_numpy(scenes.shading_mlp(13)).cuda()
    cam = scenes._camera(np.eye(3), np.zeros(3), 2.0, 1, 1, 1.0, 9.0, cx=0.4, cy=0.6)
    r = _renderer_for([cam])
    F = torch.randn(1, 1, 16, device="cuda")
    rgb = torch.empty(1, 1, 3, device="cuda")
    with pytest.raises(pl.PulsarError) as e:      # no frame yet
        pl.shade_forward(r.ctx, F, params, rgb)
    assert e.value.code == pl.ERR_STATE
    with pytest.raises(pl.PulsarError) as e:
        pl.shade_backward(r.ctx, F, params, rgb, None, torch.empty_like(params))
    assert e.value.code == pl.ERR_STATE
    _project(r, [cam])
    raw = torch.randn(1 * 16 + 1, device="cuda")
    with pytest.raises(pl.PulsarError) as e:      # features not 16-byte aligned
        pl.shade_forward(r.ctx, raw[1:], params, rgb)
    assert e.value.code == pl.ERR_ARG
    gF = torch.empty(17, device="cuda")
    with pytest.raises(pl.PulsarError) as e:      # dF not 16-byte aligned
        pl.shade_backward(r.ctx, F, params, torch.zeros(1, 1, 3, device="cuda"), gF[1:],
                          torch.empty_like(params))
    assert e.value.code == pl.ERR_ARG
    # the 1 x 1 frame against the oracle
    y = r.shade(F, params)
    dY = torch.randn(1, 1, 3, device="cuda")
    gF1, gP1 = r.shade_backward(F, params, dY)
    assert r.status(raise_on_error=False)[0] == 0
    Fn, Pn, dYn = F.cpu().numpy(), params.cpu().numpy().astype(np.float64), dY.cpu().numpy()
    ref = sb.oracle_batch(Fn[None], [cam], Pn, dYn[None])
    sb.check(dict(y=y.cpu().numpy(), dF=gF1.cpu().numpy(), params=gP1.cpu().numpy()), ref, Pn,
             "1x1 frame")
    r.close()
    # a frame of 3 channels is not a shading input
    r3 = _renderer_for([cam], C=3)
    _project(r3, [cam], C=3)
    with pytest.raises(pl.PulsarError) as e:
        pl.shade_forward(r3.ctx, F, params, rgb)
    assert e.value.code == pl.ERR_ARG
    r3.close()


def test_shading_wait_timeout_is_reported_and_the_context_recovers():
    """Failure detection without a GPU fault: the injected failure makes the
    shading kernels issue no tensor-core work, so their bounded waits (0.25 s
    of wall time) run out; the call completes and frees its tensor memory,
    pulsar_status reports PULSAR_ERR_TIMEOUT (and disarms the injection), and
    the same context then shades correctly."""
    import time

    import torch
    from splat_rendering_gb300 import pulsar as pl
    cam = scenes._camera(np.eye(3), np.zeros(3), 40.0, 48, 40, 1.0, 9.0, cx=23.3, cy=19.9)
    rng = np.random.default_rng(141)
    F = rng.standard_normal((1, 40, 48, 16)).astype(np.float32)
    dY = rng.standard_normal((1, 40, 48, 3)).astype(np.float32)
    params = scenes.shading_mlp(14)
    r = _renderer_for([cam])
    _project(r, [cam])
    Fd, Pd, dYd = (torch.from_numpy(a).cuda() for a in (F[0], params, dY[0]))
    for backward in (False, True):
        pl.debug_inject(r.ctx, pl.INJECT_SHADE_TIMEOUT)
        t0 = time.perf_counter()
        if backward:
            r.shade_backward(Fd, Pd, dYd)
        else:
            r.shade(Fd, Pd)
        code = r.status(raise_on_error=False)[0]
        waited = time.perf_counter() - t0
        assert code == pl.ERR_TIMEOUT, pl.strerror(code)
        assert waited < 10.0, waited          # the waits are bounded
        # disarmed by the status call: the next call runs normally
        y = r.shade(Fd, Pd)
        gF, gP = r.shade_backward(Fd, Pd, dYd)
        assert r.status(raise_on_error=False)[0] == 0
        ref = sb.oracle_batch(F, [cam], params.astype(np.float64), dY)
        sb.check(dict(y=y.cpu().numpy(), dF=gF.cpu().numpy(), params=gP.cpu().numpy()), ref,
                 params.astype(np.float64), f"after an injected timeout (backward={backward})")
    r.close()
