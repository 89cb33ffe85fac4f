"""Build libmla.so in-tree from csrc/*.cu for sm_103a (nvcc, no cmake).

Each translation unit is compiled in parallel, then linked into
mla_attention_gb300/libmla.so against the shared CUDA runtime (the same one
PyTorch loads).  Objects go to mla_attention_gb300/_build/.

build(guard=True) makes the guarded library instead (libmla_guard.so, objects in
_build_guard/): compiled with -DMLA_GUARD, every plain global load and store of the
kernels is checked against the extent of its buffer, skipped when outside it, and
the first such access is recorded in the status word (mla_check_device_status).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmla.so")
OBJ_GUARD = os.path.join(PKG, "_build_guard")
LIB_GUARD = os.path.join(PKG, "libmla_guard.so")
ROOT = os.path.dirname(PKG)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + os.path.join(ROOT, "include"),
                     "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libmla needs the CUDA toolkit to build")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _needs_rebuild(lib) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(ROOT, "include", "mla.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, guard: bool = False) -> str:
    nvcc = _nvcc()
    obj_dir, lib = (OBJ_GUARD, LIB_GUARD) if guard else (OBJ, LIB)
    flags = NVCC_FLAGS + (["-DMLA_GUARD"] if guard else [])
    os.makedirs(obj_dir, exist_ok=True)
    srcs = sources()
    objs = [os.path.join(obj_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    if not force and not _needs_rebuild(lib):
        return lib

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r.returncode, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, zip(srcs, objs)))
    for src, rc, log in results:
        if verbose or rc != 0:
            sys.stderr.write(f"[libmla] {os.path.basename(src)}:\n{log}")
        if rc != 0:
            raise RuntimeError(f"nvcc failed on {src}")
    tmp = lib + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "shared",
                                                           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("linking libmla.so failed")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, guard="--guard" in sys.argv))
