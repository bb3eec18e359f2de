"""Builds libflashattn.so in-tree with nvcc for sm_103a (no cmake, parallel translation units).

``python -m exact_attention_89_gb300.build`` or ``build()`` compiles every ``csrc/*.cu`` into
``_build/`` and links ``exact_attention_89_gb300/libflashattn.so``.  Static CUDA runtime; the
driver's cuTensorMapEncodeTiled is obtained at run time, so no libcuda link is needed.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libflashattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libflashattn")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(src: str, extra, build_dir: str = BUILD_DIR) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + list(extra) + ["-I", INCLUDE, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return obj, r.stderr


def build(force: bool = False, extra_flags=(), verbose: bool = False, out_dir: str | None = None) -> str:
    """Compile and link libflashattn.so; returns its path. Skips work when up to date.

    With out_dir, objects and the library go there instead (used by tests for builds with extra
    macros); the in-tree library is left alone.
    """
    lib = LIB if out_dir is None else os.path.join(out_dir, "libflashattn.so")
    bdir = BUILD_DIR if out_dir is None else os.path.join(out_dir, "obj")
    if out_dir is None and not force and not extra_flags and up_to_date():
        return LIB
    os.makedirs(bdir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(lambda s: _compile(s, extra_flags, bdir), srcs))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib + ".%d.tmp" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
