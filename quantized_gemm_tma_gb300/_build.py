"""Build ``libhq.so`` in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel, then linked
into one shared library next to this file.  Rebuilds only what changed
(source or header newer than its object).
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
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libhq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-I", INCLUDE]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; set NVCC or put the CUDA toolkit on PATH")
    return cand


def sources(src_dir: str = CSRC):
    return sorted(os.path.join(src_dir, f) for f in os.listdir(src_dir) if f.endswith((".cu", ".cpp")))


def _headers(src_dir: str = CSRC):
    hs = [os.path.join(src_dir, f) for f in os.listdir(src_dir) if f.endswith((".h", ".cuh"))]
    hs.append(os.path.join(INCLUDE, "hq.h"))
    return hs


def _stale(src: str, obj: str, newest_header: float) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return os.path.getmtime(src) > t or newest_header > t


def build(verbose: bool = False, jobs: int | None = None, extra: list[str] | None = None,
          out: str | None = None, obj_dir: str | None = None, csrc: str | None = None) -> str:
    """Compile and link; returns the path of the library (libhq.so unless `out` is given).

    `extra` adds nvcc flags (e.g. -D tuning macros); give such builds their own
    `out` and `obj_dir` (and `csrc` for a modified source tree) so they do not
    mix with the default objects.
    """
    nvcc = _nvcc()
    src_dir = csrc or CSRC
    lib_path = out or LIB
    obj_root = obj_dir or OBJ
    os.makedirs(obj_root, exist_ok=True)
    newest_header = max(os.path.getmtime(h) for h in _headers(src_dir))
    srcs = sources(src_dir)
    objs = [os.path.join(obj_root, os.path.basename(s) + ".o") for s in srcs]
    todo = [(s, o) for s, o in zip(srcs, objs) if _stale(s, o, newest_header)]

    def compile_one(so):
        s, o = so
        cmd = [nvcc, *ARCH, *FLAGS, "-I", src_dir, *(extra or []), "-c", s, "-o", o]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(s)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return o

    if todo:
        with ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            list(ex.map(compile_one, todo))
    if todo or not os.path.exists(lib_path) or any(os.path.getmtime(o) > os.path.getmtime(lib_path) for o in objs):
        cmd = [nvcc, *ARCH, "-shared", "-o", lib_path + ".tmp", *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(lib_path + ".tmp", lib_path)
    return lib_path


if __name__ == "__main__":
    build(verbose="-v" in sys.argv)
    print(LIB)
