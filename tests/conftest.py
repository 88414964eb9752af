import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # never let a GPU test run (and fail) on a machine without a GPU
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # how much the gradient tolerance's widening terms did in this session
    try:
        import gpu_helpers
    except Exception:
        return
    rows = gpu_helpers.WIDENING
    if not rows:
        return
    tr = terminalreporter
    tr.section("gradient comparisons: entries passing only through the A or S terms")
    tr.write_line(f"{'comparison':58s} {'entries':>9s} {'> plain':>8s} {'worst/plain':>11s} "
                  f"{'cond needed':>11s} {'need S':>7s}")
    for what, n, wid, worst, need, no_s in rows:
        tr.write_line(f"{what[:58]:58s} {n:9d} {wid:8d} {worst:11.3g} {need:11.3g} {no_s:7d}")
    path = os.environ.get("PULSAR_WIDENING_LOG")
    if path:
        import json
        with open(path, "w") as f:
            json.dump([dict(what=r[0], entries=r[1], outside_plain=r[2], worst_over_plain=r[3],
                            cond_needed=r[4], outside_without_sens=r[5]) for r in rows], f,
                      indent=1)
