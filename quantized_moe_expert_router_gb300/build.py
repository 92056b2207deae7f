"""Build the CUDA libraries in-tree for sm_103a (nvcc, no cmake).

  _lib/libmoe.so        the product library (csrc/*.cu, C ABI of include/moe.h)
  _lib/libmoe_synth.so  the device twin of the synthetic input generator

Translation units compile in parallel; a library is rebuilt only when one of
its sources or headers is newer than it.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
OBJDIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]

MOE_LIB = os.path.join(LIBDIR, "libmoe.so")
SYNTH_LIB = os.path.join(LIBDIR, "libmoe_synth.so")


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def _build_lib(out, sources, headers, extra, force, verbose):
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= _newest(sources + headers)):
        return out
    os.makedirs(LIBDIR, exist_ok=True)
    os.makedirs(OBJDIR, exist_ok=True)
    objs = []
    cmds = []
    for s in sources:
        o = os.path.join(OBJDIR, os.path.basename(out) + "." + os.path.basename(s) + ".o")
        objs.append(o)
        cmds.append([NVCC, *ARCH, *COMMON, *extra, "-I", INCLUDE, "-I", CSRC, "-c", s, "-o", o])
    with ThreadPoolExecutor(max_workers=min(8, len(cmds))) as ex:
        logs = list(ex.map(_run, cmds))
    if verbose:
        for lg in logs:
            print(lg)
    tmp = out + f".tmp{os.getpid()}"
    _run([NVCC, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, out)
    return out


def build(force: bool = False, verbose: bool = False) -> None:
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdrs = sorted(glob.glob(os.path.join(CSRC, "*.h*"))) + [os.path.join(INCLUDE, "moe.h")]
    extra = ["-Xptxas", "-v"] if verbose else []
    _build_lib(MOE_LIB, srcs, hdrs, extra, force, verbose)
    synth_src = [os.path.join(PKG, "synth", "synth.cu")]
    _build_lib(SYNTH_LIB, synth_src, [], ["-fmad=false"], force, verbose)


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
