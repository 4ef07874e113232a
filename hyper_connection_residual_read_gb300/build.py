"""Builds ``libhcread.so`` in-tree with nvcc for sm_103a (GB300).

Every ``csrc/*.cu`` file is compiled to an object in parallel, then linked into
one shared library next to this file. ``python -m
hyper_connection_residual_read_gb300.build`` runs it from the command line.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libhcread.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libhcread.so")
    return path


def _compile(src: str, extra: list[str], build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


# The bounds-checked variant (every hand-indexed global access range-checked; see
# hc_read_bounds_checked in include/hc_read.h), built on demand beside the objects.
BOUNDS_LIB = os.path.join(BUILD, "bounds", "libhcread_bounds.so")


def build(verbose: bool = False, extra: list[str] | None = None, out: str = LIB) -> str:
    """Compiles and links the library into `out`; returns its path."""
    build_dir = BUILD if out == LIB else os.path.join(os.path.dirname(out), "obj")
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    extra = list(extra or [])
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), srcs))
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    if verbose:
        print(f"built {out} from {len(srcs)} sources")
    if out == LIB:
        build_pycall(verbose)
    return out


def build_pycall(verbose: bool = False) -> str | None:
    """The CPython module behind the binding's hc_read / hc_read_path calls
    (csrc/hc_pycall.c, marshalling only). Without a C compiler or Python headers it
    is skipped and the binding calls the library through ctypes alone."""
    import sysconfig
    out = os.path.join(PKG, "_hcpycall" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))
    inc = sysconfig.get_paths()["include"]
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None or not os.path.exists(os.path.join(inc, "Python.h")):
        if verbose:
            print("skipped the Python call module (no C compiler or Python headers)")
        return None
    tmp = out + ".tmp"
    cmd = [cc, "-O2", "-shared", "-fPIC", "-I", inc, os.path.join(CSRC, "hc_pycall.c"), "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the Python call module failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    if verbose:
        print(f"built {out}")
    return out


def build_bounds_checked(verbose: bool = False) -> str:
    """The bounds-checked variant of the library (-DHC_BOUNDS_CHECK)."""
    return build(verbose, ["-DHC_BOUNDS_CHECK"], BOUNDS_LIB)


if __name__ == "__main__":
    if sys.argv[1:] == ["--bounds"]:
        build_bounds_checked(verbose=True)
    else:
        build(verbose=True, extra=sys.argv[1:])
