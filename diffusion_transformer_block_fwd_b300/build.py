"""Builds libflux3.so in-tree with nvcc for sm_103a.

    python -m diffusion_transformer_block_fwd_b300.build [--verbose-ptxas]

The library is one translation unit (csrc/flux3_api.cu includes the kernel
headers); the C ABI is include/flux3.h.
"""

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "flux3_api.cu")
OUT = os.path.join(PKG, "libflux3.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def sources():
    d = os.path.join(PKG, "csrc")
    files = [os.path.join(d, f) for f in os.listdir(d) if f.endswith((".cu", ".cuh", ".h"))]
    return files + [os.path.join(ROOT, "include", "flux3.h")]


def up_to_date():
    if not os.path.exists(OUT):
        return False
    t = os.path.getmtime(OUT)
    return all(os.path.getmtime(f) <= t for f in sources())


def build(force=False, ptxas_verbose=False):
    if not force and up_to_date():
        return OUT
    cmd = [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-shared",
           "-I", os.path.join(ROOT, "include"), "-o", OUT + ".tmp", SRC]
    if ptxas_verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    subprocess.run(cmd, check=True)
    os.replace(OUT + ".tmp", OUT)
    return OUT


if __name__ == "__main__":
    build(force=True, ptxas_verbose="--verbose-ptxas" in sys.argv)
    print(OUT)
