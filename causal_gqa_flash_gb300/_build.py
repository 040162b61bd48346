"""In-tree build of the CUDA library (sm_103a only).

Each translation unit in ``csrc/`` is compiled by nvcc in parallel and the
objects are linked into ``_build/libgqa_attn.so`` next to this file. Nothing is
installed anywhere else.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libgqa_attn.so"
SOURCES = ["attn_fwd.cu", "attn_bwd.cu", "rope.cu", "naive.cu", "probe.cu", "api.cu", "api_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", f"-I{INCLUDE}"]


def library_path() -> str:
    return os.path.join(BUILD_DIR, LIB_NAME)


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand) and shutil.which(cand) is None:
        raise RuntimeError("nvcc not found; set NVCC or put the CUDA toolkit on PATH")
    return cand


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return files


def up_to_date() -> bool:
    lib = library_path()
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if any source is newer than it; return its path."""
    if not force and up_to_date():
        return library_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    tmpdir = tempfile.mkdtemp(dir=BUILD_DIR)
    try:
        def compile_one(src):
            obj = os.path.join(tmpdir, os.path.splitext(src)[0] + ".o")
            cmd = [nvcc] + NVCC_FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose:
                print(r.stdout + r.stderr)
            return obj

        with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            objs = list(ex.map(compile_one, SOURCES))
        out_tmp = os.path.join(tmpdir, LIB_NAME)
        cmd = [nvcc] + ARCH + ["-shared", "-o", out_tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(out_tmp, library_path())
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)
    return library_path()
