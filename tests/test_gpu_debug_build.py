"""The debug build (device index checks that latch PULSAR_ERR_INTERNAL and skip
the access) with NVTX ranges compiled in: it must build, run the small
parity cases against the oracle through the C ABI, and report no failed
check.  The library is loaded in a child process so that it is the only
libpulsar in that process."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from splat_rendering_gb300 import pulsar as pl
pl.load({lib!r})
import numpy as np
import gpu_helpers as gh
import oracle
from splat_rendering_gb300 import scenes
oracle.build()
cases = [scenes.tiny(),
         scenes.random_scene(81, 3000, 150, 110, rot_deg=7, rrange=(0.01, 0.3)),
         scenes.random_scene(82, 400, 64, 48, channels=16, n_track=8, rrange=(0.2, 0.6)),
         scenes.random_scene(83, 1500, 100, 90, f=40.0, orthographic=True, rrange=(0.01, 0.2))]
for sc in cases:
    g = gh.run_gpu(sc)
    assert g["code"] == 0, (sc.name, pl.strerror(g["code"]))
    o = oracle.render_scene(sc)
    gh.compare_frame(g, o, sc.name)
print("debug build ok")
"""


def test_debug_build_runs_clean():
    from splat_rendering_gb300 import build as b
    lib = b.build(debug=True, nvtx=True)
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug build ok" in r.stdout
