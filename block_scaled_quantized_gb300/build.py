"""Build librs.so (the C-ABI CUDA library) in-tree for sm_103a.

Each .cu translation unit is compiled by nvcc in parallel, then linked into
``block_scaled_quantized_gb300/_build/librs.so``.  A stamp holding the hash
of the sources and flags skips the build when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "librs.so")
SOURCES = ["rs_api.cu", "rs_quant.cu", "rs_gemm.cu", "rs_noalloc.cu", "rs_kext.cu", "rs_attn.cu", "rs_gemm_pair.cu",
           "rs_tactics.cu"]
HEADERS = ["rs_device.cuh", "rs_internal.h", "rs_quant_core.cuh", "rs_tactics_gb300.inc"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: librs needs the CUDA 13 toolkit")


def _digest(extra: list[str]) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(INCLUDE, "rs.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + extra).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          name: str = "librs") -> str:
    """Compile <name>.so if its sources changed; returns the library path.
    ``name``/``extra`` select a variant, e.g. the trace build
    (``name="librs_trace", extra=["-DRS_TRACE"]``)."""
    extra = list(extra or [])
    os.makedirs(BUILD, exist_ok=True)
    lib_path = os.path.join(BUILD, name + ".so")
    stamp = os.path.join(BUILD, name + ".stamp")
    digest = _digest(extra)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return lib_path
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, name + "_" + src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr, flush=True)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None))
