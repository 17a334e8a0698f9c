"""Builds libkda.so in-tree with nvcc for sm_103a.

Each .cu file under csrc/ is compiled to an object in parallel, then linked
into ``gated_delta_rule_27_gb300/lib/libkda.so``.  A rebuild happens only when a
source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "lib", "libkda.so")
# the bounds-checking variant (every checked index is tested before its access; see csrc/kda_check.cuh)
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB = os.path.join(PKG, "lib", "libkda_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; libkda needs the CUDA toolkit to build")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs() + [os.path.abspath(__file__)])


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Builds libkda.so, or with `debug` the bounds-checking libkda_debug.so (-DKDA_DEBUG_BOUNDS)."""
    lib = DEBUG_LIB if debug else LIB
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    extra_flags = tuple(extra_flags) + (("-DKDA_DEBUG_BOUNDS",) if debug else ())
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    srcs = _sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


def _demangle(name: str) -> str:
    """The kernel's name and template arguments, without namespaces and parameter types."""
    try:
        full = subprocess.run(["c++filt", name], capture_output=True, text=True).stdout.strip() or name
    except OSError:
        return name
    full = full.replace("(anonymous namespace)::", "").split("(")[0]
    return full.replace("void ", "").split("::")[-1]


def resource_report() -> str:
    """Registers, spills, stack and shared memory of every kernel, as ptxas reports them for sm_103a
    (`-Xptxas -v`), one Markdown table row per kernel."""
    import re
    rows = []
    for src in _sources():
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-Xptxas", "-v", "-c", src, "-o", os.devnull]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s" % (src, r.stderr))
        name = None
        for line in r.stderr.splitlines():
            m = re.search(r"Compiling entry function '([^']+)'", line)
            if m:
                name = m.group(1)
                continue
            m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m and name:
                stack, st, ld = m.groups()
                continue
            m = re.search(r"Used (\d+) registers", line)
            if m and name:
                sm = re.search(r"(\d+) bytes smem", line)
                rows.append((os.path.basename(src), _demangle(name), m.group(1), stack, st, ld,
                             sm.group(1) if sm else "0"))
                name = None
    out = ["| source | kernel | registers | stack B | spill stores B | spill loads B | static smem B |",
           "|---|---|---|---|---|---|---|"]
    out += ["| %s | `%s` | %s | %s | %s | %s | %s |" % r for r in rows]
    return "\n".join(out)


if __name__ == "__main__":
    if "--resources" in sys.argv:
        print(resource_report())
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
