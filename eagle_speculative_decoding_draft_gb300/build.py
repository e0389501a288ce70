"""Builds the CUDA library (libeagle_tree.so) in-tree for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked into one shared object whose only
exported symbols are the C ABI of include/eagle_tree.h.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
OUT_DIR = PKG / "lib"
LIB = OUT_DIR / "libeagle_tree.so"
# the same library with the device-side checks of the kernels' own index invariants
# (-DEAGLE_CHECKS): a separate build, used by the tests
CHECKS_DIR = OUT_DIR / "checks"
CHECKS_LIB = CHECKS_DIR / "libeagle_tree.so"
SOURCES = ["api.cu", "gemm.cu", "topk.cu", "tree.cu", "sample.cu", "noalloc.cu", "decoder.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = Path(cand) / "bin" / "nvcc"
    return str(p) if p.exists() else "nvcc"


def _stale(lib: Path = LIB) -> bool:
    if not lib.exists():
        return True
    t = lib.stat().st_mtime
    deps = list(CSRC.glob("*.cu")) + list(CSRC.glob("*.cuh")) + [ROOT / "include" / "eagle_tree.h",
                                                                  Path(__file__)]
    return any(d.stat().st_mtime > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), checks: bool = False) -> Path:
    """Compiles the library (or, with checks, its checking variant) unless it is up to date;
    returns its path."""
    out_dir, lib = (CHECKS_DIR, CHECKS_LIB) if checks else (OUT_DIR, LIB)
    if checks:
        extra_flags = (*extra_flags, "-DEAGLE_CHECKS")
    if not force and not _stale(lib):
        return lib
    out_dir.mkdir(parents=True, exist_ok=True)
    obj_dir = out_dir / "obj"
    obj_dir.mkdir(exist_ok=True)
    common = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              f"-I{ROOT / 'include'}", *extra_flags]

    def compile_one(src: str) -> Path:
        obj = obj_dir / (Path(src).stem + ".o")
        cmd = common + ["-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0 or verbose:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}")
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib.with_suffix(f".so.tmp{os.getpid()}")
    cmd = [nvcc(), *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
