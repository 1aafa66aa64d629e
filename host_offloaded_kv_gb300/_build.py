"""In-tree build of the native parts of the package.

* ``_lib/libclo.so``       the CUDA library behind the C ABI (``include/clo.h``),
                             compiled for sm_103a only;
* ``synth/libclo_synth.so`` the seeded input generator (plain C).

Each translation unit is compiled in parallel and relinked only when a source
or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
CLO_LIB = os.path.join(LIBDIR, "libclo.so")
SYNTH_SRC = os.path.join(PKG, "synth", "synth.c")
SYNTH_LIB = os.path.join(PKG, "synth", "libclo_synth.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _nvcc() -> str:
    cand = [os.environ.get("NVCC", ""), shutil.which("nvcc") or "", "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run_parallel(cmds):
    procs = [(c, subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)) for c in cmds]
    errors = []
    for c, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"$ {' '.join(c)}\n{out}")
        elif out.strip() and os.environ.get("CLO_BUILD_VERBOSE"):
            sys.stderr.write(out)
    if errors:
        raise RuntimeError("build failed:\n" + "\n".join(errors))


def build_synth(force: bool = False) -> str:
    if force or _stale(SYNTH_LIB, [SYNTH_SRC]):
        cc = os.environ.get("CC", "gcc")
        _run_parallel([[cc, "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC", "-o", SYNTH_LIB,
                        SYNTH_SRC, "-lm"]])
    return SYNTH_LIB


def cuda_sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def build_clo(force: bool = False, extra_flags=None) -> str:
    srcs = cuda_sources()
    deps = srcs + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))
    if not (force or _stale(CLO_LIB, deps)):
        return CLO_LIB
    os.makedirs(LIBDIR, exist_ok=True)
    objdir = os.path.join(LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])
    objs, cmds = [], []
    for s in srcs:
        o = os.path.join(objdir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        cmds.append([nvcc, *ARCH, *flags, "-c", s, "-o", o])
    _run_parallel(cmds)
    tmp = CLO_LIB + ".tmp"
    _run_parallel([[nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]])
    os.replace(tmp, CLO_LIB)
    return CLO_LIB


def build_all(force: bool = False) -> None:
    build_synth(force)
    build_clo(force)
