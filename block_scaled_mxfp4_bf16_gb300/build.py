"""Build the in-tree CUDA library libmxfp4_gb300.so for sm_103a (nvcc, no cmake).

Each .cu under csrc/ is compiled in parallel into an object file, then linked into one
shared library next to this file. The CUDA runtime is linked statically; the driver API is
reached through cudaGetDriverEntryPointByVersion, so loading the library needs no GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB_NAME = "libmxfp4_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
BUILD_DIR = os.path.join(HERE, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              f"-I{INCLUDE}", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the MXFP4 library needs the CUDA toolkit to build")


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                               + glob.glob(os.path.join(INCLUDE, "*.h")))


FLAGS_STAMP = os.path.join(BUILD_DIR, "lib.flags")   # the extra flags of the last link


def up_to_date() -> bool:
    """The in-tree library exists, is newer than every source and was built without extra flags
    (a phase-trace build, say, is never taken for the product build)."""
    if not os.path.exists(LIB_PATH) or not os.path.exists(FLAGS_STAMP):
        return False
    with open(FLAGS_STAMP) as fh:
        if fh.read().strip():
            return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _deps())


def variant_path(variant: str) -> str:
    """Path of a separately built variant of the library (for example the test-hook build)."""
    return os.path.join(HERE, f"libmxfp4_gb300_{variant}.so")


def build_variant(variant: str, extra_flags: list[str]) -> str:
    """Build a variant of the library with extra flags into its own file and object directory,
    leaving the product library alone; rebuilt only when a source is newer. Returns its path."""
    path = variant_path(variant)
    if os.path.exists(path) and all(os.path.getmtime(d) <= os.path.getmtime(path) for d in _deps()):
        return path
    return build(force=True, extra_flags=extra_flags, lib_path=path, obj_dir=os.path.join(BUILD_DIR, variant))


def build(force: bool = False, extra_flags: list[str] | None = None, verbose: bool = False,
          lib_path: str | None = None, obj_dir: str | None = None) -> str:
    """Compile and link the library if any source is newer than it. Returns its path."""
    if lib_path is None and not force and not extra_flags and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    out_path = lib_path or LIB_PATH
    objs_dir = obj_dir or BUILD_DIR
    os.makedirs(objs_dir, exist_ok=True)
    flags = NVCC_FLAGS + (extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(objs_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_path)
    if lib_path is None:
        with open(FLAGS_STAMP, "w") as fh:
            fh.write(" ".join(extra_flags or []))
    return out_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
