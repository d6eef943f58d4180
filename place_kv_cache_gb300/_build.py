"""Build the CUDA library in-tree: every translation unit of csrc/ compiled
for sm_103a in parallel with nvcc, linked into ``libol.so`` beside this file.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_objs")
LIB = os.path.join(HERE, "libol.so")
OBJ_PHASE = os.path.join(HERE, "_objs_phase")
LIB_PHASE = os.path.join(HERE, "libol_phase.so")
SOURCES = ["ol_api.cpp", "ol_append.cu", "ol_generic.cu", "ol_fast_bf16.cu", "ol_fast_int4.cu", "ol_noalloc.cu",
           "ol_hpaged.cu", "ol_fast_hpaged.cu"]
HEADERS = ["ol_internal.h", "ol_launch.h", "ol_common.cuh", "ol_merge.cuh", "ol_fast_bf16_kernel.inc", "ol_hpaged.cuh",
           os.path.join("..", "..", "include", "ol.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose: bool, obj_dir: str = OBJ, defines=()) -> str:
    path = os.path.join(CSRC, src)
    obj = os.path.join(obj_dir, src + ".o")
    deps = [path] + [os.path.join(CSRC, h) for h in HEADERS]
    if not _stale(obj, deps):
        return obj
    cmd = [nvcc(), *ARCH, *FLAGS, *[f"-D{d}" for d in defines], "-c", path, "-o", obj]
    if src.endswith(".cpp"):
        cmd[1:1] = ["-x", "cu"]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, variant: str = "") -> str:
    """Build libol.so; variant "phase" builds libol_phase.so instead, the timing
    build whose decode kernel records per-CTA phase stamps (OL_PHASE_STAMPS)."""
    obj_dir, lib, defines = (OBJ_PHASE, LIB_PHASE, ("OL_PHASE_STAMPS=1",)) if variant == "phase" else (OBJ, LIB, ())
    os.makedirs(obj_dir, exist_ok=True)
    if force:
        for f in os.listdir(obj_dir):
            os.remove(os.path.join(obj_dir, f))
    # the stamps live in ol_fast_bf16.cu only: the timing build shares every other object
    stamped = ("ol_fast_bf16.cu",) if variant == "phase" else ()

    def one(src):
        return _compile(src, verbose, obj_dir, defines) if src in stamped else _compile(src, verbose)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(one, SOURCES))
    if force or _stale(lib, objs):
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", lib + ".tmp", *objs, "-lpthread", "-ldl", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
