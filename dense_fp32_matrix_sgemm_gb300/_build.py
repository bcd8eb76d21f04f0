"""Builds libsgemm_gb300.so in-tree with nvcc for sm_103a (GB300).

Each .cu file under csrc/ is compiled to an object in parallel, then linked
into one shared library next to this file.  Objects are rebuilt only when a
source or header is newer.  No torch extension machinery is involved: the
library exposes a plain C ABI (include/sgemm_gb300.h).
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "sgemm_gb300")
LIB = os.path.join(PKG, "libsgemm_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Hidden visibility: the library exports only the C ABI that the public
# headers declare, so its kernels and host stubs cannot bind to, or be bound
# by, same-named symbols of another library in the process.
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-Xcompiler", "-fvisibility=hidden", "-Xptxas", "-O3", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the SGEMM library needs the CUDA toolkit to build")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _compile(src: str, ptxas_verbose: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    newest = max([os.path.getmtime(src)] + [os.path.getmtime(h) for h in _headers()])
    if os.path.exists(obj) and os.path.getmtime(obj) >= newest and not ptxas_verbose:
        return obj, ""
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj + ".tmp"]
    if ptxas_verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    os.replace(obj + ".tmp", obj)
    return obj, r.stderr


def build(verbose: bool = False, ptxas_verbose: bool = False, jobs: int | None = None) -> str:
    """Compile every csrc/*.cu for sm_103a and link the shared library."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    jobs = jobs or min(len(srcs), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose), srcs))
    objs = [o for o, _ in results]
    if ptxas_verbose or verbose:
        for src, (_, log) in zip(srcs, results):
            if log:
                sys.stderr.write(f"== {os.path.basename(src)}\n{log}")
    newest_obj = max(os.path.getmtime(o) for o in objs)
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < newest_obj:
        cmd = [nvcc(), *ARCH, "-shared", "-o", LIB + ".tmp", *objs, "-lcudart_static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(LIB + ".tmp", LIB)
    if verbose:
        sys.stderr.write(f"built {LIB}\n")
    _build_calls(verbose)
    return LIB


def _build_calls(verbose: bool = False):
    """Compile _calls.c, the CPython argument-marshalling module for the
    compute entry points (see that file), next to the library.  Without a C
    compiler or the Python headers nothing is built and the package marshals
    through ctypes instead; the library is the same either way."""
    import sysconfig
    src = os.path.join(PKG, "_calls.c")
    out = os.path.join(PKG, "_calls" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))
    inc = sysconfig.get_paths().get("include", "")
    cc = shutil.which("cc") or shutil.which("gcc")
    if not cc or not os.path.exists(os.path.join(inc, "Python.h")):
        if verbose:
            sys.stderr.write("note: no C compiler or Python headers; the binding uses ctypes\n")
        return None
    newest = max(os.path.getmtime(src), os.path.getmtime(os.path.join(INCLUDE, "sgemm_gb300.h")))
    if os.path.exists(out) and os.path.getmtime(out) >= newest:
        return out
    cmd = [cc, "-O2", "-std=gnu11", "-shared", "-fPIC", "-Wall", "-I", inc, "-I", INCLUDE, src,
           "-o", out + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        if verbose:
            sys.stderr.write(f"note: _calls.c did not build, the binding uses ctypes:\n{r.stderr}\n")
        return None
    os.replace(out + ".tmp", out)
    if verbose:
        sys.stderr.write(f"built {out}\n")
    return out


if __name__ == "__main__":
    build(verbose=True, ptxas_verbose="-v" in sys.argv)
