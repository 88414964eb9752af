"""Build the CUDA library libpulsar.so in-tree with nvcc for sm_103a.

    python -m splat_rendering_gb300.build [--verbose] [--ptxas-info] [--debug] [--nvtx]

Each translation unit under csrc/ is compiled in parallel, then linked into
splat_rendering_gb300/libpulsar.so (static CUDA runtime).  Nothing here needs
a GPU.  Two optional builds go to their own files next to it:
  --debug  libpulsar_debug.so: device index checks that latch an error
           (PULSAR_ERR_INTERNAL from pulsar_status) and skip the access;
  --nvtx   NVTX ranges around every C entry point (header-only NVTX3);
both together: libpulsar_debug_nvtx.so.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpulsar.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["project.cu", "bin.cu", "forward.cu", "backward.cu", "shade.cu", "pulsar.cu",
           "noalloc.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(ptxas_info: bool, debug: bool = False, nvtx: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-ffp-contract=off", f"-I{INCLUDE}", "--expt-relaxed-constexpr"]
    if ptxas_info:
        f += ["-Xptxas", "-v"]
    if debug:
        f += ["-DPULSAR_DEBUG"]
    if nvtx:
        f += ["-DPULSAR_NVTX"]
    return f


def lib_path(debug: bool = False, nvtx: bool = False) -> str:
    suffix = ("_debug" if debug else "") + ("_nvtx" if nvtx else "")
    return os.path.join(HERE, f"libpulsar{suffix}.so")


def _stale(lib: str, deps) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug: bool = False, nvtx: bool = False) -> str:
    lib = lib_path(debug, nvtx)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + [
        os.path.join(CSRC, "pulsar_internal.cuh"), os.path.join(INCLUDE, "pulsar.h"), __file__]
    if not force and not ptxas_info and not _stale(lib, deps):
        return lib
    out_dir = os.path.join(OUT_DIR, os.path.basename(lib)[:-3]) if (debug or nvtx) else OUT_DIR
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    flags = _flags(ptxas_info, debug, nvtx)

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, cmd, r

    objs = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for src, obj, cmd, r in ex.map(compile_one, SOURCES):
            if verbose or ptxas_info:
                print(" ".join(cmd), file=sys.stderr)
                if r.stderr:
                    print(r.stderr, file=sys.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
            objs.append(obj)
    tmp = lib + ".tmp"
    cmd = [cc, "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose="--verbose" in sys.argv, ptxas_info="--ptxas-info" in sys.argv,
                debug="--debug" in sys.argv, nvtx="--nvtx" in sys.argv))
