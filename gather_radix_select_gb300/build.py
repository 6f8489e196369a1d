"""Builds libsel.so (the CUDA kernels + C ABI) in-tree for sm_103a.

    python -m gather_radix_select_gb300.build [--force] [--debug] [-v]

Each .cu under csrc/ is compiled by its own nvcc process (in parallel), then
the objects are linked into gather_radix_select_gb300/_lib/libsel.so with the
CUDA runtime linked statically, so the library needs only the driver.

--debug builds libsel_debug.so instead: the same sources with SEL_DEBUG
defined, whose kernels check selected accesses (staged-list and region
offsets, workspace slots, output positions, gathered key rows), skip the ones
that would leave their buffer and report SEL_EBOUNDS in err_flag.  It is
loaded instead of libsel.so when SEL_LIBRARY=debug is set.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
SO = os.path.join(OUT_DIR, "libsel.so")
DEBUG_SO = os.path.join(OUT_DIR, "libsel_debug.so")
ROOT = os.path.dirname(HERE)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if not f.startswith(".")]
    files.append(os.path.join(ROOT, "include", "sel.h"))
    return files


def up_to_date(so: str = SO) -> bool:
    if not os.path.exists(so):
        return False
    t = os.path.getmtime(so)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          debug: bool = False) -> str:
    so = DEBUG_SO if debug else SO
    if not force and up_to_date(so):
        return so
    obj_dir = os.path.join(OUT_DIR, "debug" if debug else "release")
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (["-DSEL_DEBUG"] if debug else []) + list(extra_flags or [])
    objs = []
    cmds = []
    for src in sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmds.append([cc, *ARCH, *flags, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for " + cmd[-3])
        return r

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        list(ex.map(run, cmds))
    tmp = so + ".tmp%d" % os.getpid()
    run([cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, so)
    return so


def build_all(force: bool = False) -> list[str]:
    """libsel.so and libsel_debug.so, compiled side by side."""
    with concurrent.futures.ThreadPoolExecutor(max_workers=2) as ex:
        return list(ex.map(lambda d: build(force=force, debug=d), (False, True)))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
