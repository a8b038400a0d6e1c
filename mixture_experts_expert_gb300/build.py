"""Builds libmoe_gb300.so in-tree with nvcc (sm_103a only).

Each CUDA translation unit is compiled in parallel into ``_build/`` and linked
into ``mixture_experts_expert_gb300/libmoe_gb300.so``.  Only the ``moe_*``
symbols are exported.  The library is rebuilt unless a stamp file beside it holds the
SHA-256 of every source, the header, this script, the compiler flags, the nvcc version
and the host architecture it was built from; ``build()`` reports which of the two
happened (``last_status``: "compiled" or "reused").
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libmoe_gb300.so")
STAMP_PATH = LIB_PATH + ".sha256"
last_status = None   # "compiled" or "reused", set by build()

SOURCES = ["moe_api.cu", "route.cu", "router.cu", "gemm_fwd.cu", "gemm_bwd.cu", "gemm_dw.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I" + CSRC, "-I" + INCLUDE]


def _nvcc() -> str:
    cand = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"),
            shutil.which("nvcc") or ""]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "moe_gb300.h"))
    files.append(os.path.abspath(__file__))
    return files


def source_key(flags: list[str]) -> str:
    """SHA-256 over the sources, the header, this script, the flags, nvcc's version
    and the host architecture."""
    h = hashlib.sha256()
    for f in sorted(_deps()):
        h.update(os.path.basename(f).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + flags).encode())
    h.update(platform.machine().encode())
    try:
        ver = subprocess.run([_nvcc(), "--version"], capture_output=True, text=True).stdout
    except Exception:
        ver = ""
    h.update(ver.encode())
    return h.hexdigest()


def up_to_date(flags: list[str] | None = None) -> bool:
    if not (os.path.exists(LIB_PATH) and os.path.exists(STAMP_PATH)):
        return False
    with open(STAMP_PATH) as fh:
        return fh.read().strip() == source_key(NVCC_FLAGS + list(flags or []))


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compiles (unless the stamped build matches the sources) and returns the path of
    libmoe_gb300.so; ``last_status`` says which happened."""
    global last_status
    if not force and up_to_date(extra_flags):
        last_status = "reused"
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-Xlinker", "--exclude-libs,ALL"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(STAMP_PATH, "w") as fh:
        fh.write(source_key(flags) + "\n")
    last_status = "compiled"
    return LIB_PATH


if __name__ == "__main__":
    import sys
    path = build(force="--force" in sys.argv, verbose=True,
                 extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None)
    print(last_status, path)
