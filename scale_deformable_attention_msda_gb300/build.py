"""Build libmsda.so in-tree with nvcc for sm_103a (no cmake, no torch build).

Each translation unit under csrc/ is compiled twice in one parallel pool:
plainly into ``libmsda.so`` and with ``-DMSDA_CHECKED`` into
``libmsda_checked.so`` (every kernel access range-checked; see
msda_checked.cu), both next to this file. The CUDA runtime is linked
statically and its symbols are hidden, so each library exports only the
``msda_*`` C ABI of ``include/msda.h``. Rebuilds happen only when a source
is newer than a library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIBRARY = os.path.join(PKG, "libmsda.so")
CHECKED_LIBRARY = os.path.join(PKG, "libmsda_checked.so")
VARIANTS = {LIBRARY: ("plain", []), CHECKED_LIBRARY: ("checked", ["-DMSDA_CHECKED"])}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmsda")
    return path


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            [os.path.join(INCLUDE, "msda.h"), os.path.abspath(__file__)])


def stale(library: str = LIBRARY) -> bool:
    if not os.path.exists(library):
        return True
    t = os.path.getmtime(library)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src: str, variant: str, defines: list, verbose: bool) -> str:
    obj = os.path.join(BUILD_DIR, variant, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *defines, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    if verbose and r.stderr:
        print(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libmsda.so and libmsda_checked.so if needed; returns the path
    of libmsda.so."""
    todo = [lib for lib in VARIANTS if force or stale(lib)]
    if not todo:
        return LIBRARY
    srcs = sources()
    jobs = []
    for lib in todo:
        variant, defines = VARIANTS[lib]
        os.makedirs(os.path.join(BUILD_DIR, variant), exist_ok=True)
        jobs += [(lib, src, variant, defines) for src in srcs]
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda j: (j[0], _compile(j[1], j[2], j[3], verbose)), jobs))
    for lib in todo:
        tmp = lib + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-Xlinker", "--exclude-libs=ALL",
               "-o", tmp, *[o for l, o in objs if l == lib]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"linking {os.path.basename(lib)} failed:\n{r.stderr}")
        os.replace(tmp, lib)
    return LIBRARY


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
