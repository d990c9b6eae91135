"""Build libla.so (the C-ABI linear-attention library) in-tree with nvcc for sm_103a.

Each CUDA source compiles to its own object in parallel; the objects link into
``efficient_transformer_gb300/_lib/libla.so`` (git-ignored).  Nothing is installed.

``build(variant="test")`` builds the same sources with ``-DLA_TEST_HOOKS`` into
``_lib/libla_test.so``: bounded waits give up after 5 ms instead of 2 s, and one exported
switch makes a kernel withhold a barrier arrival, so that a test can check the timeout
path end to end.  The product library never contains these hooks.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libla.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libla.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hdrs + [os.path.abspath(__file__)]


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


# "timeline": block 0 of the forward and backward kernels records clock64() at fixed events
# of its first 64 chunks (read back with la_timeline_read*), for pipeline studies.
VARIANTS = {"": [], "test": ["-DLA_TEST_HOOKS"], "timeline": ["-DLA_TIMELINE"]}


def lib_path(variant: str = "") -> str:
    return LIB_PATH if not variant else os.path.join(LIB_DIR, f"libla_{variant}.so")


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          variant: str = "") -> str:
    """Compile every ``csrc/*.cu`` and link ``libla.so`` (or the named variant); returns
    the library path."""
    nvcc = _nvcc()
    obj_dir = OBJ_DIR if not variant else OBJ_DIR + "_" + variant
    out_lib = lib_path(variant)
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    common = _deps()
    flags = NVCC_FLAGS + VARIANTS[variant] + (extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        if force or _stale(obj, common + [src]):
            cmd = [nvcc] + ARCH + flags + ["-c", src, "-o", obj + ".tmp.o"]
            if verbose:
                print(" ".join(cmd))
            subprocess.run(cmd, check=True)
            os.replace(obj + ".tmp.o", obj)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    if force or _stale(out_lib, objs):
        cmd = [nvcc] + ARCH + ["-shared", "-o", out_lib + ".tmp", *objs]
        subprocess.run(cmd, check=True)
        os.replace(out_lib + ".tmp", out_lib)
    return out_lib


if __name__ == "__main__":
    print(build(verbose=True))
