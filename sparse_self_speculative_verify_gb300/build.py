"""Builds libssd.so (the CUDA kernels + C ABI) in-tree for sm_103a with nvcc.

Each translation unit under ``csrc/`` is compiled in parallel to an object file, then the
objects are linked into ``_build/<machine>/libssd.so``.  The library is rebuilt only when a
source or header is newer than it.  No CMake, no other architectures.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=default", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def build_dir(variant: str = "") -> str:
    return os.path.join(PKG, "_build", platform.machine() + (f"-{variant}" if variant else ""))


def lib_path(variant: str = "") -> str:
    return os.path.join(build_dir(variant), "libssd.so")


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit on PATH")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(variant: str = "") -> bool:
    out = lib_path(variant)
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(p) <= t for p in _deps())


# Diagnostic builds, each in a directory of its own beside the library proper (never loaded by the
# product path): "trace" records the tensor-core verify's per-block timeline (trace_verify.py).
VARIANT_FLAGS = {"trace": ["-DSSD_VERIFY_TRACE"]}


def build(force: bool = False, verbose: bool = False, extra_flags=None, variant: str = "") -> str:
    """Compile and link libssd.so (or a diagnostic variant of it); returns its path."""
    if not force and up_to_date(variant):
        return lib_path(variant)
    nvcc = _nvcc()
    odir = os.path.join(build_dir(variant), "obj")
    extra_flags = list(extra_flags or []) + VARIANT_FLAGS.get(variant, [])
    os.makedirs(odir, exist_ok=True)
    flags = ARCH + NVCC_FLAGS + ["-I", INCLUDE, "-I", CSRC] + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(odir, os.path.basename(src) + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib_path(variant) + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path(variant))
    return lib_path(variant)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
