"""The allocation-free render entry point (pulsar_render_noalloc) against the
context-based one (pulsar_project / pulsar_bin / pulsar_forward).

Some callers cannot allocate device memory while they render -- a stream being
captured into a graph, a plugin whose host owns the device memory budget, a
fixed-footprint real-time renderer -- so the library offers one entry point
whose scratch arrays live in a static device arena.  Its image must equal the
regular path's within the forward tolerance, call after call (the arena keeps
the previous call's contents).  This file is collected last on purpose.
"""
from __future__ import annotations

import numpy as np
import pytest

import gpu_helpers as gh
from splat_rendering_gb300 import scenes

pytestmark = pytest.mark.gpu


def _noalloc_image(sc):
    import torch
    from splat_rendering_gb300 import pulsar as pl
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()  # noqa: E731
    cam = sc.cameras[0]
    img = torch.full((cam.height, cam.width, sc.params.channels), float("nan"), device="cuda")
    pl.render_noalloc(t(sc.pos), t(sc.radius), t(sc.opacity), t(sc.features), sc.n,
                      pl.camera(cam), pl.params(sc.params), t(sc.bg), img)
    torch.cuda.synchronize()
    return img.cpu().numpy()


def test_noalloc_render_matches_context_path_on_consecutive_calls():
    # different frames in a row (different sizes, channels, n_track, an
    # orthographic camera), then the first again: each must match the context path
    first = scenes.random_scene(71, 3000, 200, 150, rot_deg=9, rrange=(0.01, 0.3))
    second = scenes.random_scene(72, 800, 96, 120, channels=5, n_track=7, fy=130.0, cx=40.0,
                                 rrange=(0.02, 0.4))
    third = scenes.random_scene(74, 1500, 120, 100, f=40.0, orthographic=True, rot_deg=12,
                                rrange=(0.01, 0.2))
    for sc in (first, second, third, first):
        ref = gh.run_gpu(sc, want=False, debug=False)
        assert ref["code"] == 0
        img = _noalloc_image(sc)
        gh.assert_close(img, ref["image"], gh.FWD_RTOL, gh.FWD_ATOL, f"noalloc {sc.name}")


def test_noalloc_rejects_sizes_beyond_its_arena():
    import torch
    from splat_rendering_gb300 import pulsar as pl
    sc = scenes.random_scene(73, 10, 300, 40)        # wider than 256 px
    img = torch.empty((40, 300, 3), device="cuda")
    z = torch.zeros(30, device="cuda")
    with pytest.raises(pl.PulsarError) as e:
        pl.render_noalloc(z, z, z, z, 10, pl.camera(sc.cameras[0]), pl.params(sc.params), z, img)
    assert e.value.code == pl.ERR_ARG
    with pytest.raises(pl.PulsarError) as e:                 # more spheres than the arena holds
        pl.render_noalloc(z, z, z, z, 16385, pl.camera(scenes.tiny().cameras[0]),
                          pl.params(sc.params), z, img)
    assert e.value.code == pl.ERR_ARG
