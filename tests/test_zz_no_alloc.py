"""The allocation-free render entry point (pulsar_render_noalloc) against the
context-based one (pulsar_project / pulsar_bin / pulsar_forward) and the
oracle.

Some callers cannot allocate device memory while they render -- a plugin
whose host framework owns the device memory budget, a fixed-footprint
real-time renderer that must not risk an allocation failure mid-frame -- so
the library offers one entry point whose scratch arrays live in a static
device arena.  Its image must equal the regular path's within the forward
tolerance, call after call (the arena keeps the previous call's contents),
and a frame that overflows the arena must be refused without disturbing the
next one.  This file is collected last on purpose.
"""
from __future__ import annotations

import numpy as np
import pytest

import gpu_helpers as gh
from splat_rendering_gb300 import scenes

pytestmark = pytest.mark.gpu

ARENA_PAIRS = 65536   # sphere-tile pairs the arena holds


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


def test_noalloc_render_matches_oracle(oracle_lib):
    sc = scenes.random_scene(75, 2500, 160, 130, rot_deg=6, rrange=(0.01, 0.25))
    img = _noalloc_image(sc)
    o = oracle_lib.render_scene(sc, with_grads=False)
    gh.assert_close(img, o["image"], gh.FWD_RTOL, gh.FWD_ATOL, "noalloc vs oracle")


def test_noalloc_capacity_overflow_then_recovers(oracle_lib):
    """A frame with more sphere-tile pairs than the arena holds is refused with
    PULSAR_ERR_CAPACITY and leaves the image untouched; the next call, on the
    arena the overflowing one left behind, renders correctly."""
    from splat_rendering_gb300 import pulsar as pl
    import torch
    big = scenes.random_scene(76, 2000, 256, 256, rrange=(0.5, 1.5))   # spheres of many tiles
    pairs = oracle_lib.tile_lists(big.pos, big.radius, big.opacity, big.cameras[0],
                                  big.params)[1].size
    assert pairs > ARENA_PAIRS
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()  # noqa: E731
    cam = big.cameras[0]
    img = torch.full((cam.height, cam.width, 3), float("nan"), device="cuda")
    with pytest.raises(pl.PulsarError) as e:
        pl.render_noalloc(t(big.pos), t(big.radius), t(big.opacity), t(big.features), big.n,
                          pl.camera(cam), pl.params(big.params), t(big.bg), img)
    assert e.value.code == pl.ERR_CAPACITY
    assert torch.isnan(img).all(), "an overflowing frame must not write the image"
    small = scenes.random_scene(77, 1200, 256, 200, rot_deg=4, rrange=(0.01, 0.2))
    ref = gh.run_gpu(small, want=False, debug=False)
    assert ref["code"] == 0
    gh.assert_close(_noalloc_image(small), ref["image"], gh.FWD_RTOL, gh.FWD_ATOL,
                    "noalloc after an overflow")


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
