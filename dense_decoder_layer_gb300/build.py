"""Build the in-tree CUDA libraries for sm_103a with nvcc.

* ``libpds.so`` (the product): every ``csrc/*.cu`` file, compiled to an
  object in parallel and linked into one shared library next to this file.
* ``tests/xcheck/libpds_xcheck.so`` (test-only): the independent mma.sync
  attention kernel the GPU tests compare the product's attention against.
  The product never loads it.

Objects go to ``_build/`` (ignored by git).  Run
``python -m dense_decoder_layer_gb300.build``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build", "pds")
LIB = os.path.join(HERE, "libpds.so")
XCHECK_DIR = os.path.join(ROOT, "tests", "xcheck")
XCHECK_LIB = os.path.join(XCHECK_DIR, "libpds_xcheck.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources(d=CSRC):
    return sorted(os.path.join(d, f) for f in os.listdir(d) if f.endswith(".cu"))


def _newer(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(ROOT, "include", "pds.h"))
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                    "-I" + os.path.join(ROOT, "include"), "-I" + CSRC, "--expt-relaxed-constexpr"]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    cc = nvcc()
    libs = {LIB: sources(), XCHECK_LIB: sources(XCHECK_DIR)}
    objs, jobs = {}, []
    for lib, srcs in libs.items():
        objs[lib] = []
        for src in srcs:
            obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
            objs[lib].append(obj)
            if force or _newer(obj, [src] + headers):
                jobs.append([cc, *flags, "-c", src, "-o", obj])

    def run(cmd):
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p

    failed = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for cmd, p in ex.map(run, jobs):
            if verbose or ptxas_verbose or p.returncode:
                sys.stderr.write(p.stdout + p.stderr)
            if p.returncode:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed on " + ", ".join(failed))
    for lib, lib_objs in objs.items():
        if force or jobs or _newer(lib, lib_objs):
            cmd = [cc, *ARCH, "-shared", "-o", lib, *lib_objs, "-lcudart"]
            p = subprocess.run(cmd, capture_output=True, text=True)
            if p.returncode:
                raise RuntimeError("link failed:\n" + p.stdout + p.stderr)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, ptxas_verbose="--ptxas" in sys.argv))
