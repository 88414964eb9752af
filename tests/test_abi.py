"""The C ABI library builds, loads and exports what include/pulsar.h declares
(no GPU needed: only host-side argument checks are called)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from splat_rendering_gb300 import build, pulsar
    build.build()
    return pulsar.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "pulsar.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|int64_t|const char\*)\s+(pulsar_\w+)\s*\(", src, re.M)))


def test_header_declares_the_path():
    names = _declared()
    for n in ("pulsar_create", "pulsar_project", "pulsar_bin", "pulsar_forward",
              "pulsar_backward", "pulsar_status", "pulsar_destroy"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_strerror_and_host_side_argument_errors(lib):
    from splat_rendering_gb300 import pulsar as pl
    assert pl.strerror(0) == "ok"
    assert "max_pairs" in pl.strerror(pl.ERR_CAPACITY)
    h = ctypes.c_void_p()
    # invalid limits are rejected before any CUDA call
    assert lib.pulsar_create(None, 0, 10, 10, 16, 16, 3, 5) == pl.ERR_ARG
    assert lib.pulsar_create(ctypes.byref(h), 0, 10, 10, 16, 16, 3, 0) == pl.ERR_ARG
    assert lib.pulsar_create(ctypes.byref(h), 0, 10, 10, 16, 16, 65, 5) == pl.ERR_ARG
    assert lib.pulsar_create(ctypes.byref(h), 0, 10, 0, 16, 16, 3, 5) == pl.ERR_ARG
    assert lib.pulsar_create(ctypes.byref(h), 0, 10, 10, 70000, 16, 3, 5) == pl.ERR_ARG
    # sphere indices are 32-bit with a launch's margin: at most 0x7fff0000 spheres
    assert lib.pulsar_create(ctypes.byref(h), 0, 0x7fff0001, 10, 16, 16, 3, 5) == pl.ERR_ARG
    # NULL context
    assert lib.pulsar_bin(None, None) == pl.ERR_ARG
    assert lib.pulsar_forward(None, None, None, None, None) == pl.ERR_ARG
    assert lib.pulsar_status(None, None, None, None) == pl.ERR_ARG
    assert lib.pulsar_destroy(None) == pl.ERR_ARG
    assert lib.pulsar_shade_forward(None, None, None, None, None) == pl.ERR_ARG
    assert lib.pulsar_shade_backward(None, None, None, None, None, None, None) == pl.ERR_ARG
    assert lib.pulsar_debug_inject(None, 1, None) == pl.ERR_ARG


def test_struct_layouts_match_header():
    from splat_rendering_gb300 import pulsar as pl
    assert ctypes.sizeof(pl.Camera) == 4 * (9 + 3 + 4) + 4 * 2 + 4 * 2 + 4
    assert pl.Camera.width.offset == 64 and pl.Camera.znear.offset == 72
    assert pl.Camera.orthographic.offset == 80
    assert ctypes.sizeof(pl.Params) == 4 * 5 + 4 * 3


def test_missing_library_fails_loudly(tmp_path):
    from splat_rendering_gb300 import pulsar as pl
    saved = pl._lib
    pl._lib = None
    try:
        with pytest.raises(RuntimeError, match="no CPU fallback"):
            pl.load(str(tmp_path / "libpulsar.so"))
    finally:
        pl._lib = saved


def test_debug_and_nvtx_builds_export_the_same_symbols():
    """The optional builds (device index checks; NVTX ranges) compile for sm_103a
    without a GPU and export every declared entry point."""
    from splat_rendering_gb300 import build
    path = build.build(debug=True, nvtx=True)
    dbg = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(dbg, name), name
    dbg.pulsar_strerror.restype = ctypes.c_char_p
    assert b"index check" in dbg.pulsar_strerror(-7)
