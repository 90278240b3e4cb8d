"""Build libdgemm.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel to an object file
under _build/, then linked into dense_gemm_09_gb300/libdgemm.so against the
shared CUDA runtime (so the library shares the runtime state -- current
device, primary context -- of the process that loads it).

The checked build (libdgemm_checked.so, objects under _build/checked/) is
the same sources compiled with -DDGEMM_CHECKED: device-side bounds checks on
the indices the kernels compute (see csrc/checked.cuh).  build_all() compiles
both libraries' units at once.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdgemm.so")
LIB_CHECKED = os.path.join(PKG, "libdgemm_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
          "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    cand = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"),
            shutil.which("nvcc") or ""]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found (set CUDA_HOME)")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _variant(checked: bool):
    """(library path, object directory, extra nvcc flags) of one build."""
    if checked:
        return LIB_CHECKED, os.path.join(BUILD, "checked"), ["-DDGEMM_CHECKED"]
    return LIB, BUILD, []


def build_all(variants=(False, True), force: bool = False, verbose: bool = False,
              extra_flags: list[str] | None = None) -> list[str]:
    """Compile the requested builds (False: libdgemm.so, True: the checked
    libdgemm_checked.so), every translation unit of all of them in parallel,
    and link each library.  Returns the library paths."""
    cc = nvcc()
    jobs = []  # (lib, objs, procs)
    for checked in variants:
        lib, objdir, flags = _variant(checked)
        if not force and up_to_date(lib):
            continue
        os.makedirs(objdir, exist_ok=True)
        objs, procs = [], []
        for src in sources():
            obj = os.path.join(objdir, os.path.basename(src) + ".o")
            objs.append(obj)
            cmd = [cc, *ARCH, *CFLAGS, *flags, *(extra_flags or []), "-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                                text=True)))
        jobs.append((lib, objs, procs))
    failed = []
    for _, _, procs in jobs:
        for src, p in procs:
            out, _ = p.communicate()
            if p.returncode != 0:
                failed.append(src + "\n" + out)
            elif verbose and out.strip():
                print(out, file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    for lib, objs, _ in jobs:
        tmp = lib + ".tmp%d" % os.getpid()
        subprocess.check_call([cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return [_variant(c)[0] for c in variants]


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          checked: bool = False) -> str:
    """Compile one library: libdgemm.so, or with checked=True the checked build."""
    return build_all((checked,), force=force, verbose=verbose, extra_flags=extra_flags)[0]


if __name__ == "__main__":
    for path in build_all(force="--force" in sys.argv, verbose=True,
                          extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None):
        print(path)
