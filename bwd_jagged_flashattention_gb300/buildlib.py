"""Build libjfa.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel; the result is linked into
``bwd_jagged_flashattention_gb300/libjfa.so`` (git-ignored).  No cmake and
no torch extension machinery: the library is a plain C-ABI shared object.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB_PATH = os.path.join(HERE, "libjfa.so")
BUILD_DIR = os.path.join(ROOT, "_build")

SOURCES = ["jfa_api.cu", "fwd.cu", "bwd.cu", "mxfp8.cu", "host_util.cu", "selftest.cu", "scheduler.cpp", "noalloc.cu"]
HEADERS = ["ptx.cuh", "kernels.h", "scheduler.h", "host_util.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libjfa.so")


def _flags(verbose_ptxas: bool) -> list[str]:
    f = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "-I", os.path.join(ROOT, "include")]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    """Compile (if stale) and link libjfa.so.  Returns its path."""
    nvcc = _nvcc()
    build_dir, lib_path = BUILD_DIR, LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "jfa.h"),
                                                        os.path.join(ROOT, "include", "jfa_selftest.h")]
    objs, cmds = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(build_dir, src.replace(".", "_") + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + hdrs):
            cmds.append([nvcc] + _flags(verbose_ptxas) + ["-c", path, "-o", obj])
    if cmds:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(cmds), os.cpu_count() or 4)) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), cmds))
        for c, r in zip(cmds, results):
            if verbose_ptxas or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(c)}")
    if force or cmds or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link of libjfa.so failed")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
