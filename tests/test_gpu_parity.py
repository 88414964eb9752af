"""CUDA path vs the CPU oracle, through the C ABI, on seeded inputs.

Bit-exact: per-sphere fp32 decisions, tile lists, tracked ids, hit counts.
Within tolerance: image, stabiliser and normaliser (1e-5 relative / 1e-6
absolute), gradients (1e-4 relative / 1e-5 absolute).
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest

import gpu_helpers as gh
from splat_rendering_gb300 import scenes

pytestmark = pytest.mark.gpu


def _oracle_all(oracle_lib, sc, cam_index=0, window=None, grad_image=None):
    cam = sc.cameras[cam_index]
    G = sc.grad_images[cam_index] if grad_image is None else grad_image
    o = oracle_lib.render(sc.pos, sc.radius, sc.opacity, sc.features, cam, sc.params, sc.bg,
                          grad_image=G, window=window)
    d = oracle_lib.project(sc.pos, sc.radius, sc.opacity, cam, sc.params)
    offs, ids = oracle_lib.tile_lists(sc.pos, sc.radius, sc.opacity, cam, sc.params)
    return o, d, offs, ids


def _check_lists(g, offs, ids):
    assert np.array_equal(g["tile_offsets"].astype(np.int64), offs), "tile offsets differ"
    assert np.array_equal(g["tile_ids"].astype(np.int64), ids.astype(np.int64)), "tile lists differ"


@pytest.mark.parametrize("name", ["tiny", "medium", "headline", "neural"])
def test_config_full_frame(oracle_lib, name):
    sc = scenes.make(name)
    o, d, offs, ids = _oracle_all(oracle_lib, sc)
    g = gh.run_gpu(sc, max_pairs=len(ids) + 1024)
    assert g["code"] == 0
    assert g["n_pairs"] == len(ids)
    assert g["hits"] == o["hits"]
    gh.assert_decisions_equal(g, d)
    _check_lists(g, offs, ids)
    gh.compare_frame(g, o, name)


@pytest.mark.parametrize("cam_index", range(6))
def test_driving_cameras(oracle_lib, cam_index):
    """Driving rig: full-frame decisions and tile lists; image and gradients on
    a 320x192 window (the upstream gradient is zero outside it)."""
    sc = scenes.driving()
    cam = sc.cameras[cam_index]
    win = (800, 560, 1120, 752)
    G = gh.windowed_grad(sc, cam_index, win)
    d = oracle_lib.project(sc.pos, sc.radius, sc.opacity, cam, sc.params)
    offs, ids = oracle_lib.tile_lists(sc.pos, sc.radius, sc.opacity, cam, sc.params)
    o = oracle_lib.render(sc.pos, sc.radius, sc.opacity, sc.features, cam, sc.params, sc.bg,
                          grad_image=G, window=win)
    g = gh.run_gpu(sc, cam_index, grad_image=G, max_pairs=len(ids) + 1024)
    assert g["code"] == 0 and g["n_pairs"] == len(ids)
    gh.assert_decisions_equal(g, d)
    _check_lists(g, offs, ids)
    gh.compare_frame(g, o, f"driving cam{cam_index}", window=win)


EDGE = {
    # ragged image, rotated and translated camera, fx != fy, off-centre principal point
    "ragged": dict(seed=51, n=300, width=37, height=23, rot_deg=15, shift=(0.2, -0.1, 0.3),
                   f=30.0, fy=41.0, cx=15.3, cy=9.1, rrange=(0.01, 0.3)),
    "one_channel": dict(seed=52, n=400, width=48, height=40, channels=1, n_track=1),
    "wide_payload": dict(seed=53, n=300, width=40, height=33, channels=33, n_track=16),
    # the largest payload and tracking depth the ABI accepts (98% of the pixels
    # fill all 16 slots), and the 17-32 channel build
    "max_payload": dict(seed=61, n=1500, width=40, height=33, channels=64, n_track=16,
                        rrange=(0.1, 0.5)),
    "payload_32": dict(seed=62, n=1200, width=45, height=31, channels=32, n_track=12,
                       rrange=(0.08, 0.4)),
    "five_channels": dict(seed=54, n=300, width=50, height=30, channels=5, n_track=9),
    "no_cutoff": dict(seed=55, n=500, width=64, height=48, geom_cutoff=False, rrange=(0.005, 0.2)),
    # big spheres: lists of ~4,200 keys, each sorted whole in shared memory
    "long_lists": dict(seed=56, n=20000, width=64, height=64, f=64.0, zrange=(2.5, 6.5),
                       rrange=(0.5, 1.5), spread=1.5),
    # many one-pixel spheres: lists of ~20,600 keys, past one shared-memory
    # sort, so sorted in chunks merged through global memory (four merge
    # passes), at ~150 hits per pixel
    "huge_lists": dict(seed=63, n=80000, width=32, height=32, f=32.0, zrange=(2.5, 6.5),
                       rrange=(0.001, 0.01)),
    "spill_outside": dict(seed=57, n=2000, width=80, height=60, spread=2.5, rrange=(0.01, 0.5)),
}


@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_cases(oracle_lib, case):
    sc = scenes.random_scene(**EDGE[case])
    o, d, offs, ids = _oracle_all(oracle_lib, sc)
    g = gh.run_gpu(sc, max_pairs=len(ids) + 64)
    assert g["code"] == 0
    gh.assert_decisions_equal(g, d)
    _check_lists(g, offs, ids)
    gh.compare_frame(g, o, case)
    if case == "long_lists":
        assert np.diff(offs).max() > 2048
    if case == "huge_lists":
        assert np.diff(offs).min() > 16384


@pytest.mark.parametrize("n", [3000, 6000, 12000])
def test_equal_depth_keys(oracle_lib, n):
    """Spheres on three depth planes with two radii: a handful of distinct
    sort keys, so every tile list is made of long runs of equal keys ordered
    by sphere id alone (Pulsar Sec. 3.2 sorts by earliest possible
    intersection; the id tie-break makes the list unique).  About 190, 375
    and 750 candidates per tile: one register network, two merged runs, the
    block sort."""
    sc = scenes.random_scene(59, n, 64, 64, f=64.0, zrange=(3.0, 4.5), rrange=(0.02, 0.08))
    rng = np.random.default_rng(60)
    sc.pos[:, 2] = rng.choice(np.float32([3.0, 4.0, 4.5]), n)
    sc.radius[:] = rng.choice(np.float32([0.03, 0.05]), n)
    o, d, offs, ids = _oracle_all(oracle_lib, sc)
    kept = d["key"][ids]
    assert len(np.unique(kept)) <= 6
    lens = np.diff(offs)
    lo, hi = {3000: (129, 256), 6000: (257, 512), 12000: (513, 2048)}[n]
    assert ((lens >= lo) & (lens <= hi)).sum() >= 4, lens
    g = gh.run_gpu(sc, max_pairs=len(ids) + 64)
    assert g["code"] == 0
    gh.assert_decisions_equal(g, d)
    _check_lists(g, offs, ids)
    gh.compare_frame(g, o, f"equal keys n={n}")


def test_zero_opacity_spheres(oracle_lib):
    sc = scenes.random_scene(58, 400, 48, 48, rrange=(0.02, 0.3))
    sc.opacity[::3] = 0.0
    o, d, offs, ids = _oracle_all(oracle_lib, sc)
    g = gh.run_gpu(sc)
    gh.assert_decisions_equal(g, d)
    gh.compare_frame(g, o, "zero opacity")


def test_empty_scene(oracle_lib):
    sc = scenes.random_scene(1, 0, 33, 17)
    sc.bg[:] = [0.5, -2.0, 1.25]
    g = gh.run_gpu(sc)
    assert g["code"] == 0 and g["n_pairs"] == 0 and g["hits"] == 0
    assert np.array_equal(g["image"], np.broadcast_to(sc.bg, g["image"].shape))
    assert (g["ids"] == -1).all()
    assert not g["grad_cam"].any()


def test_everything_culled(oracle_lib):
    sc = scenes.random_scene(2, 500, 40, 40)
    sc.pos[:, 2] *= -1.0
    g = gh.run_gpu(sc)
    assert g["code"] == 0 and g["n_pairs"] == 0 and g["hits"] == 0
    assert not g["grad_pos"].any() and not g["grad_cam"].any()


def test_early_stop_bound(oracle_lib):
    """With a small gamma the forward stops early once n_track hits are tracked;
    the image stays within tau * max|f - F| (plus fp32 rounding of the
    exponent, 2^-24 * 8 / gamma) of the exact blend and the tracked ids equal
    the oracle's (Pulsar Sec. 3.2, B.1.3)."""
    sc = scenes.random_scene(60, 20000, 48, 48, rrange=(0.05, 0.4), zrange=(2, 6),
                             gamma=0.01, n_track=2)
    sc.params.stop_tau = 1e-4
    o = oracle_lib.render(sc.pos, sc.radius, sc.opacity, sc.features, sc.cameras[0], sc.params,
                          sc.bg)
    g = gh.run_gpu(sc, want=False)
    assert np.array_equal(g["ids"], o["ids"])
    assert (g["nhits"] < o["nhits"]).any(), "early stop never triggered"
    spread = np.abs(sc.features).max() + np.abs(o["image"]).max()
    tol = 1e-4 * spread + 2.0 ** -24 * 8 / 0.01 * spread + 1e-6
    assert np.abs(g["image"] - o["image"]).max() <= tol


def test_capacity_overflow_and_recovery(oracle_lib):
    """Too many sphere-tile pairs: the frame reports PULSAR_ERR_CAPACITY without
    faulting; the same context then renders a fitting frame correctly."""
    from splat_rendering_gb300 import pulsar as pl
    big = scenes.random_scene(61, 3000, 64, 64, rrange=(0.1, 0.6))
    offs, ids = oracle_lib.tile_lists(big.pos, big.radius, big.opacity, big.cameras[0], big.params)
    r = pl.Renderer(max_spheres=3000, max_pairs=len(ids) // 2, max_width=64, max_height=64,
                    max_channels=3, max_track=5)
    g = gh.run_gpu(big, renderer=r, want=False, debug=False)
    assert g["code"] == pl.ERR_CAPACITY
    small = scenes.random_scene(62, 200, 64, 64, rrange=(0.01, 0.1))
    o, d, offs2, ids2 = _oracle_all(oracle_lib, small)
    assert len(ids2) <= len(ids) // 2
    g2 = gh.run_gpu(small, renderer=r)
    assert g2["code"] == 0
    _check_lists(g2, offs2, ids2)
    gh.compare_frame(g2, o, "after overflow")


def test_call_order_and_arguments():
    import torch
    from splat_rendering_gb300 import pulsar as pl
    r = pl.Renderer(max_spheres=10, max_pairs=100, max_width=16, max_height=16)
    img = torch.zeros((16, 16, 3), device="cuda")
    bg = torch.zeros(3, device="cuda")
    with pytest.raises(pl.PulsarError) as e:
        pl.forward(r.ctx, None, bg, img)
    assert e.value.code == pl.ERR_STATE
    with pytest.raises(pl.PulsarError) as e:
        pl.bin(r.ctx)
    assert e.value.code == pl.ERR_STATE
    sc = scenes.random_scene(3, 10, 16, 16)
    cam, prm = pl.camera(sc.cameras[0]), pl.params(sc.params)
    pos = torch.from_numpy(sc.pos).cuda()
    rad = torch.from_numpy(sc.radius).cuda()
    opa = torch.from_numpy(sc.opacity).cuda()
    with pytest.raises(pl.PulsarError) as e:
        pl.project(r.ctx, pos, rad, opa, 11, cam, prm)   # above max_spheres
    assert e.value.code == pl.ERR_ARG
    big = pl.camera(replace(sc.cameras[0], width=17))
    with pytest.raises(pl.PulsarError) as e:
        pl.project(r.ctx, pos, rad, opa, 10, big, prm)
    assert e.value.code == pl.ERR_ARG
    bad = pl.params(sc.params)
    bad.n_track = 9
    with pytest.raises(pl.PulsarError) as e:
        pl.project(r.ctx, pos, rad, opa, 10, cam, bad)
    assert e.value.code == pl.ERR_ARG
    pl.project(r.ctx, pos, rad, opa, 10, cam, prm)
    with pytest.raises(pl.PulsarError) as e:
        pl.backward(r.ctx, None, bg, img, img, grad_cam=torch.zeros(16, device="cuda"))
    assert e.value.code == pl.ERR_STATE
    pl.bin(r.ctx)
    with pytest.raises(pl.PulsarError) as e:
        pl.bin(r.ctx)
    assert e.value.code == pl.ERR_STATE
    assert r.status()[0] == 0


def test_partial_gradient_requests(oracle_lib):
    """Only the requested gradients are written (Pulsar Sec. B.2)."""
    sc = scenes.random_scene(63, 500, 48, 40, rrange=(0.02, 0.3))
    o, _, _, _ = _oracle_all(oracle_lib, sc)
    g = gh.run_gpu(sc, want=("opacity",))
    assert set(k for k in g if k.startswith("grad_")) == {"grad_opacity"}
    dF = gh.image_err(g["image"], o["image"])
    gh.assert_close(g["grad_opacity"], o["grad_opacity"], gh.GRAD_RTOL, gh.GRAD_ATOL, "opacity",
                    o["abs_grad_opacity"], o["sens_grad_opacity"], dF)
    g = gh.run_gpu(sc, want=("cam", "features"))
    dF = gh.image_err(g["image"], o["image"])
    gh.assert_close(g["grad_cam"], o["grad_cam"], gh.GRAD_RTOL, gh.GRAD_ATOL, "cam",
                    o["abs_grad_cam"], o["sens_grad_cam"], dF)
    gh.assert_close(g["grad_features"], o["grad_features"], gh.GRAD_RTOL, gh.GRAD_ATOL, "feat",
                    o["abs_grad_features"], o["sens_grad_features"], dF)


def test_repeat_frames_and_determinism(oracle_lib):
    """One context, frames of different scenes and cameras in a row: the
    zero-between-frames workspace invariants hold, and repeating a frame
    reproduces lists and image bit for bit."""
    from splat_rendering_gb300 import pulsar as pl
    r = pl.Renderer(max_spheres=5000, max_pairs=200000, max_width=96, max_height=80,
                    max_channels=4, max_track=8)
    a = scenes.random_scene(64, 3000, 96, 80, rrange=(0.01, 0.2), rot_deg=5)
    b = scenes.random_scene(65, 1000, 70, 50, channels=4, n_track=8, rrange=(0.02, 0.3))
    ga1 = gh.run_gpu(a, renderer=r)
    gb = gh.run_gpu(b, renderer=r)
    ga2 = gh.run_gpu(a, renderer=r)
    for k in ("tile_ids", "tile_offsets", "ids", "image", "mg", "wsum"):
        assert np.array_equal(ga1[k], ga2[k]), k
    # gradients are sums of atomics (order not fixed): both runs against the oracle
    oa, _, _, _ = _oracle_all(oracle_lib, a)
    gh.compare_frame(ga1, oa, "first run")
    gh.compare_frame(ga2, oa, "repeated run")
    o, _, _, _ = _oracle_all(oracle_lib, b)
    gh.compare_frame(gb, o, "second scene")


def test_unaligned_gradient_arrays(oracle_lib):
    """Gradient outputs that are not 16-byte aligned take the scalar path of the
    finalize kernel and give the same result."""
    import torch
    from splat_rendering_gb300 import pulsar as pl
    sc = scenes.random_scene(66, 777, 48, 40, rrange=(0.02, 0.3), rot_deg=8)
    o, _, _, _ = _oracle_all(oracle_lib, sc)
    r = pl.Renderer(max_spheres=sc.n, max_pairs=1 << 16, max_width=48, max_height=40)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    pos, feat, bg = t(sc.pos), t(sc.features), t(sc.bg)
    img = r.render(pos, t(sc.radius), t(sc.opacity), feat, pl.camera(sc.cameras[0]),
                   pl.params(sc.params), bg)
    buf = torch.zeros(3 * sc.n + 1, device="cuda")
    gpos = buf[1:].view(sc.n, 3)                      # 4-byte offset
    rbuf = torch.zeros(sc.n + 1, device="cuda")
    grad = rbuf[1:]
    pl.backward(r.ctx, feat, bg, img, t(sc.grad_images[0]), grad_pos=gpos, grad_radius=grad)
    assert r.status()[0] == 0
    dF = gh.image_err(img.cpu().numpy(), o["image"])
    gh.assert_close(gpos.cpu().numpy(), o["grad_pos"], gh.GRAD_RTOL, gh.GRAD_ATOL, "pos",
                    o["abs_grad_pos"], o["sens_grad_pos"], dF)
    gh.assert_close(grad.cpu().numpy(), o["grad_radius"], gh.GRAD_RTOL, gh.GRAD_ATOL, "radius",
                    o["abs_grad_radius"], o["sens_grad_radius"], dF)


def test_backward_twice_on_one_frame(oracle_lib):
    """The forward zeroes the backward's accumulators; a second backward of the
    same frame (another upstream gradient) must start from zero again, so both
    calls match the oracle."""
    import torch
    from splat_rendering_gb300 import pulsar as pl
    sc = scenes.random_scene(67, 1200, 64, 48, rrange=(0.02, 0.3), rot_deg=4)
    o, _, _, _ = _oracle_all(oracle_lib, sc)
    r = pl.Renderer(max_spheres=sc.n, max_pairs=1 << 16, max_width=64, max_height=48)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    img = r.render(t(sc.pos), t(sc.radius), t(sc.opacity), t(sc.features),
                   pl.camera(sc.cameras[0]), pl.params(sc.params), t(sc.bg))
    G = t(sc.grad_images[0])
    first = {k: v.cpu().numpy() for k, v in r.backward(G).items()}
    second = {k: v.cpu().numpy() for k, v in r.backward(G).items()}
    assert r.status()[0] == 0
    dF = gh.image_err(img.cpu().numpy(), o["image"])
    for g in (first, second):
        for k in ("pos", "radius", "opacity", "features", "cam"):
            gh.assert_close(g[k], o["grad_" + k], gh.GRAD_RTOL, gh.GRAD_ATOL, f"twice {k}",
                            o["abs_grad_" + k], o["sens_grad_" + k], dF)


def test_unaligned_sixteen_channel_rows(oracle_lib):
    """Rows of 16 channels that are not 16-byte aligned (features, image and
    image gradient at a 4-byte offset) take the scalar paths of the forward's
    feature staging and image stores and of the backward's feature staging and
    pixel loads: the image and the tracked ids come out bit for bit as with
    aligned rows, and the gradients match the oracle."""
    import torch
    from splat_rendering_gb300 import pulsar as pl
    sc = scenes.random_scene(67, 600, 48, 40, channels=16, n_track=8, rrange=(0.05, 0.4))
    o, _, _, _ = _oracle_all(oracle_lib, sc)
    r = pl.Renderer(max_spheres=sc.n, max_pairs=1 << 16, max_width=48, max_height=40,
                    max_channels=16, max_track=8)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731

    def offset(a):   # a copy of a at a 4-byte offset from a 16-byte boundary
        buf = torch.zeros(a.numel() + 1, device="cuda")
        v = buf[1:].view(a.shape)
        v.copy_(a)
        return v

    pos, rad, opa, bg = t(sc.pos), t(sc.radius), t(sc.opacity), t(sc.bg)
    cam, prm = pl.camera(sc.cameras[0]), pl.params(sc.params)
    feat = t(sc.features)
    img_aligned = r.render(pos, rad, opa, feat, cam, prm, bg)
    ids_aligned = r.debug("ids").copy()
    feat_u = offset(feat)
    img_u = offset(torch.zeros_like(img_aligned))
    r.render(pos, rad, opa, feat_u, cam, prm, bg, image=img_u)
    assert torch.equal(img_u, img_aligned)
    assert np.array_equal(r.debug("ids"), ids_aligned)
    grads = r.backward(offset(t(sc.grad_images[0])))
    assert r.status()[0] == 0
    dF = gh.image_err(img_u.cpu().numpy(), o["image"])
    for k in ("pos", "radius", "opacity", "features", "cam"):
        gh.assert_close(grads[k].cpu().numpy(), o["grad_" + k], gh.GRAD_RTOL, gh.GRAD_ATOL, k,
                        o["abs_grad_" + k], o["sens_grad_" + k], dF)
