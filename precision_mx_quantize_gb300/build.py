"""Build the in-tree CUDA library libmxq.so for sm_103a with nvcc.

Each translation unit under csrc/ compiles in parallel to an object file,
then nvcc links the shared library into _lib/.  Nothing is installed into
site-packages: the binding loads the library from this folder.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libmxq.so")
# bounds-checked variant: every kernel checks the global indices it computes
# and records MXQ_ERR_BOUNDS instead of accessing out of range
LIB_DEBUG = os.path.join(OUT_DIR, "libmxq_debug.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the MX library needs the CUDA toolkit to build")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile_cmds(nvcc, obj_dir, debug_bounds, ptxas_info):
    common = [
        "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
        "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr",
    ]
    if debug_bounds:
        common += ["-DMXQ_DEBUG_BOUNDS"]
    if ptxas_info:
        common += ["-Xptxas", "-v"]
    return [(src, [nvcc, *common, "-c", src, "-o",
                   os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")])
            for src in sources()]


def _link(nvcc, objs, lib):
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stderr}")
    os.replace(tmp, lib)


def build(verbose: bool = False, ptxas_info: bool = False, debug_bounds: bool = True) -> str:
    """Compile every csrc/*.cu for sm_103a and link _lib/libmxq.so (and, with
    debug_bounds, the bounds-checked _lib/libmxq_debug.so from the same
    sources, compiled in the same parallel batch); returns the main path."""
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    variants = [(LIB, os.path.join(OUT_DIR, "obj"), False)]
    if debug_bounds:
        variants.append((LIB_DEBUG, os.path.join(OUT_DIR, "obj_debug"), True))
    jobs = []
    for lib, obj_dir, dbg in variants:
        os.makedirs(obj_dir, exist_ok=True)
        jobs += [(lib, src, cmd) for src, cmd in _compile_cmds(nvcc, obj_dir, dbg, ptxas_info)]

    def compile_one(job):
        lib, src, cmd = job
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{p.stderr}")
        return lib, src, cmd[-1], p.stderr

    # the longest translation units first, so that they do not end last
    jobs.sort(key=lambda j: -os.path.getsize(j[1]))
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose or ptxas_info:
        for lib, src, _, log in results:
            if log.strip() and lib == LIB:
                sys.stderr.write(f"== {os.path.basename(src)}\n{log}\n")
    for lib, _, _ in variants:
        _link(nvcc, sorted(o for l, _, o, _ in results if l == lib), lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv))
