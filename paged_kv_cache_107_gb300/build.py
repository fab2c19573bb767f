"""Build the CUDA library in-tree: paged_kv_cache_107_gb300/lib/libpagedkv.so.

Every .cu file under csrc/ is compiled for sm_103a only (one -gencode), in parallel, then
linked into one shared library with a plain C ABI (include/pa.h). No torch headers are
involved; the CUDA runtime is linked statically.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB_DIR = os.path.join(HERE, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libpagedkv.so")
OBJ_DIR = os.path.join(LIB_DIR, "obj")
GENCODE = "arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    cuda_home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    cand = os.path.join(cuda_home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: set CUDA_HOME")
    return found


def _flags(extra=()):
    return ["-gencode", GENCODE, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
            "--expt-relaxed-constexpr", *extra]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + [os.path.join(os.path.dirname(HERE), "include", "pa.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib_path: str = None) -> str:
    """Compile csrc/*.cu for sm_103a and link lib/libpagedkv.so. Returns its path.

    lib_path: build a separate library there instead (always rebuilt, objects beside it),
    for example a test build with extra preprocessor flags; the in-tree library is left
    alone."""
    if lib_path is not None:
        return _build_to(lib_path, lib_path + ".obj", verbose, extra_flags)
    if not force and up_to_date():
        return LIB_PATH
    return _build_to(LIB_PATH, OBJ_DIR, verbose, extra_flags)


def _build_to(lib_path: str, obj_dir: str, verbose: bool, extra_flags) -> str:
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()
    srcs = sources()

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *_flags(extra_flags), "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, "-gencode", GENCODE, "-shared", "-Xcompiler", "-fPIC", "-o", tmp,
           *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
