"""Build libkvq.so (the CUDA library) in-tree with nvcc, for sm_103a only.

    python -m fp8_paged_kv_e4m3_gb300.build [--force] [--verbose-ptxas]

Each .cu file under csrc/ compiles in its own nvcc process (in parallel);
the objects link into fp8_paged_kv_e4m3_gb300/_build/libkvq.so with the
CUDA runtime linked statically.  No torch headers are involved: the library
is a plain C ABI.
"""
from __future__ import annotations

import argparse
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libkvq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) \
        + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    objs = []
    jobs = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        for src in _sources():
            obj = os.path.join(BUILD, os.path.basename(src) + ".o")
            objs.append(obj)
            cmd = [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
            jobs.append(ex.submit(subprocess.run, cmd, capture_output=True, text=True))
        results = [j.result() for j in jobs]
    for r in results:
        if r.returncode != 0 or (ptxas_verbose and r.stderr):
            sys.stderr.write(r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(r.args))
    tmp = LIB + f".{os.getpid()}.tmp"
    link = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    return LIB


def build_variant(tag: str, defines: dict, sources=("kvq_attn.cu",)) -> str:
    """A test build of the library at _build/<tag>/libkvq.so: the translation
    units `sources` compiled again with the preprocessor `defines` (name ->
    value), linked with the default build's other objects.  Used by tests
    that need an instrumented kernel; the default library never carries the
    defines."""
    build()
    out_dir = os.path.join(BUILD, tag)
    lib = os.path.join(out_dir, "libkvq.so")
    srcs = [os.path.join(CSRC, f) for f in sources]
    if os.path.exists(lib) and all(os.path.getmtime(p) <= os.path.getmtime(lib) for p in _deps() + [LIB]):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    dflags = [f"-D{k}={v}" for k, v in defines.items()]
    own = {}
    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, len(srcs)))) as ex:
        jobs = []
        for src in srcs:
            obj = os.path.join(out_dir, os.path.basename(src) + ".o")
            own[os.path.basename(src)] = obj
            jobs.append(ex.submit(subprocess.run, [cc, *ARCH, *FLAGS, *dflags, "-c", src, "-o", obj],
                                  capture_output=True, text=True))
        for j in jobs:
            r = j.result()
            if r.returncode != 0:
                sys.stderr.write(r.stderr)
                raise RuntimeError("nvcc failed:\n" + " ".join(r.args))
    objs = [own.get(os.path.basename(src), os.path.join(BUILD, os.path.basename(src) + ".o"))
            for src in _sources()]
    tmp = lib + f".{os.getpid()}.tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, ptxas_verbose=args.verbose_ptxas))
