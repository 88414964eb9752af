"""Normalised gradients (Pulsar Sec. B.2; PULSAR_FLAG_NORMALIZE_GRADS): the
CUDA path against the oracle's reading of them.  The oracle itself is
parity unpinned here (the quantities are not derivatives): these tests fix
that the two implementations of the one stated reading agree, within the
gradient tolerance of the plain path."""
from __future__ import annotations

from dataclasses import replace

import pytest

import gpu_helpers as gh
from splat_rendering_gb300 import scenes
from test_gpu_parity import _check_lists, _oracle_all

pytestmark = pytest.mark.gpu

CASES = {
    "pinhole": dict(seed=91, n=3000, width=96, height=80, rot_deg=14, shift=(0.1, 0.2, -0.1),
                    rrange=(0.005, 0.3)),
    "orthographic": dict(seed=92, n=2500, width=80, height=70, f=28.0, orthographic=True,
                         rot_deg=9, rrange=(0.005, 0.3)),
    "sixteen_channels": dict(seed=93, n=2000, width=72, height=64, channels=16, n_track=8,
                             rrange=(0.01, 0.3)),
    "no_cutoff_floor": dict(seed=94, n=2000, width=64, height=64, geom_cutoff=False,
                            rrange=(0.001, 0.02)),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_normalised_gradients(oracle_lib, case):
    sc = scenes.random_scene(**CASES[case])
    sc = replace(sc, params=replace(sc.params, normalize_grads=True))
    o, d, offs, ids = _oracle_all(oracle_lib, sc)
    g = gh.run_gpu(sc, max_pairs=len(ids) + 64)
    assert g["code"] == 0
    gh.assert_decisions_equal(g, d)
    _check_lists(g, offs, ids)
    gh.compare_frame(g, o, f"normalised {case}")


def test_normalisation_leaves_the_next_frame_plain(oracle_lib):
    """The per-sphere tracking counters are cleared by the frame that used
    them: a plain frame rendered next on the same context is unaffected."""
    from splat_rendering_gb300 import pulsar as pl
    base = scenes.random_scene(95, 1500, 64, 48, rrange=(0.01, 0.3))
    normed = replace(base, params=replace(base.params, normalize_grads=True))
    r = pl.Renderer(max_spheres=1500, max_pairs=1 << 16, max_width=64, max_height=48,
                    max_channels=3, max_track=5)
    for sc in (normed, base, normed):
        o, d, offs, ids = _oracle_all(oracle_lib, sc)
        g = gh.run_gpu(sc, renderer=r)
        assert g["code"] == 0
        gh.compare_frame(g, o, f"sequence normalize={sc.params.normalize_grads}")
    r.close()


def test_normalised_gradients_over_stale_culled_records(oracle_lib):
    """A culled sphere writes only the first half of its record, so one that
    the previous frame of the same context kept still holds that frame's
    geometry in the second half.  The normalised finalize reads a record's
    geometry only for spheres some pixel tracks: moving the camera 3 units
    forward culls about half the spheres of the first frame, and the
    normalised gradients of the second frame still match the oracle."""
    import numpy as np
    from splat_rendering_gb300 import pulsar as pl
    base = scenes.random_scene(96, 2000, 64, 48, rrange=(0.01, 0.3))
    cam = base.cameras[0]
    moved = replace(cam, t=(cam.t - np.array([0.0, 0.0, 3.0], np.float32)).astype(np.float32))
    second = replace(base, cameras=[moved], params=replace(base.params, normalize_grads=True))
    r = pl.Renderer(max_spheres=2000, max_pairs=1 << 16, max_width=64, max_height=48,
                    max_channels=3, max_track=5)
    culled = []
    for sc in (base, second):
        o, d, offs, ids = _oracle_all(oracle_lib, sc)
        culled.append(int((d["keep"] == 0).sum()))
        g = gh.run_gpu(sc, renderer=r)
        assert g["code"] == 0
        gh.assert_decisions_equal(g, d)
        gh.compare_frame(g, o, f"{sc.name} normalize={sc.params.normalize_grads}")
    r.close()
    assert culled[1] > culled[0] + 500, culled
