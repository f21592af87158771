"""Builds libgdn.so in-tree with nvcc for sm_103a (no cmake, no torch)."""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")


def _flags():
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


# Build variants: name -> extra nvcc flags.  "check" is the debug
# bounds-check build (csrc/gdn_check.cuh); its objects and library sit beside
# the normal ones under their own names.
VARIANTS = {"check": ["-DGDN_BOUNDS_CHECK"]}


def build_variant(name: str, force: bool = False, verbose: bool = False) -> str:
    return build(force=force, verbose=verbose, extra=VARIANTS[name], variant=name)


def build(force: bool = False, verbose: bool = False, extra=(), variant=None) -> str:
    build_dir = BUILD if variant is None else os.path.join(PKG, "_build_" + variant)
    lib_path = LIB if variant is None else os.path.join(PKG, "libgdn_%s.so" % variant)
    os.makedirs(build_dir, exist_ok=True)
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))
    objs = []
    jobs = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            jobs.append([NVCC] + _flags() + list(extra) + ["-c", src, "-o", obj])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n%s\n%s" % (" ".join(cmd), r.stdout + r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)

    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp%d" % os.getpid()
        run([NVCC] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
