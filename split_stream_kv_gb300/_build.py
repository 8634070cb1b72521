"""Build liblynx.so in-tree: each csrc/*.cu compiled by nvcc for sm_103a in
parallel, then linked into one shared library next to this file.  The same
sources compiled with -DLYNX_CHECKED give liblynx_checked.so, the checked
build whose kernels verify their index arithmetic (see common.cuh)."""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_objs")
LIB = os.path.join(HERE, "liblynx.so")
OBJ_CHECKED = os.path.join(HERE, "_objs_checked")
LIB_CHECKED = os.path.join(HERE, "liblynx_checked.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: no scalar multiply/add pair is contracted into a fused
# multiply-add behind the source's back.  The codec's binary32 statistics
# follow a fixed operation order (one rounding per step); every fma the
# kernels want is written explicitly (fmaf, fma.rn.f32x2, fma.rm.f32).  (The
# flag does not cover packed f32x2 pairs, so products that feed an add are
# computed with scalar __fmul_rn in the kernels.)
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-Wall", "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _build_one(lib: str, objdir: str, extra, force: bool, verbose: bool, pool) -> list:
    """Compile jobs for one library (the stale objects) and the link step."""
    os.makedirs(objdir, exist_ok=True)
    hdrs = _headers()
    objs, jobs = [], []
    for src in _sources():
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + hdrs):
            jobs.append((src, obj, extra))
    return objs, jobs


def _compile_one(job, verbose=False):
    src, obj, extra = job
    tmp = obj + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    os.replace(tmp, obj)
    return r.stderr


def _link(lib: str, objs, force: bool, built: bool):
    if force or built or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, checked: bool = True) -> str:
    """Compile and link if anything changed; return the library path.  With
    `checked`, also the checked build (compiled in the same parallel pass)."""
    targets = [(LIB, OBJ, [])]
    if checked:
        targets.append((LIB_CHECKED, OBJ_CHECKED, ["-DLYNX_CHECKED"]))
    plans = [(lib, *_build_one(lib, od, extra, force, verbose, None)) for lib, od, extra in targets]
    jobs = [j for _, _, js in plans for j in js]
    if jobs:
        with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            for log in ex.map(lambda j: _compile_one(j, verbose), jobs):
                if verbose and log:
                    sys.stderr.write(log)
    for lib, objs, js in plans:
        _link(lib, objs, force, bool(js))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
