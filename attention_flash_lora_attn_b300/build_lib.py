"""Compile the CUDA library in-tree for sm_103a.

    python -m attention_flash_lora_attn_b300.build_lib [--debug]

Produces attention_flash_lora_attn_b300/_lib/libflashlora.so (one unity
translation unit, csrc/api.cu, that includes every kernel).  The runtime is
linked statically; the driver API is reached through
cudaGetDriverEntryPointByVersion, so the library loads on a machine without
a GPU (every call then returns FLA_ERR_CUDA).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libflashlora.so")
ROOT = os.path.dirname(HERE)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh")))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    deps = sources() + [os.path.join(ROOT, "include", "flash_lora_attn.h"), __file__]
    return all(os.path.getmtime(f) <= t for f in deps)


def build(force: bool = False, debug: bool = False, verbose: bool = False) -> str:
    if not force and not debug and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-std=c++17", "-O3", "-lineinfo", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-Xcompiler", "-Wall",
           "-I", os.path.join(ROOT, "include"), "-I", CSRC,
           "-DFLA_BUILD", "-o", tmp, os.path.join(CSRC, "api.cu")]
    if debug:
        cmd += ["-DFLA_DEBUG"]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed building libflashlora.so")
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, debug="--debug" in sys.argv, verbose="-v" in sys.argv))
