"""Build libspecdec.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", f) for f in ("specdec_verify.cu", "specdec_ngram.cu", "specdec_bitmask.cu")]
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libspecdec.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")


def build_library(out: str = LIB_PATH, extra_flags=(), verbose: bool = False) -> str:
    tmp = f"{out}.tmp{os.getpid()}"          # write then rename: concurrent builders never see a partial file
    cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-o", tmp, *SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({' '.join(cmd)}):\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, out)
    if verbose:
        print(res.stdout, res.stderr)
    return out


def needs_rebuild(out: str = LIB_PATH) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    deps = SOURCES + [os.path.join(INCLUDE, "specdec.h")]
    return any(os.path.getmtime(d) > t for d in deps)


if __name__ == "__main__":
    print(build_library(verbose=True))
