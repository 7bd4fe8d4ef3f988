"""Builds the CUDA library in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libspec_verify.so")
SOURCES = [os.path.join(CSRC, "spec_verify.cu"), os.path.join(CSRC, "spec_verify_noalloc.cu"),
           os.path.join(CSRC, "telemetry.cu"), os.path.join(CSRC, "lm_head.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "sv_device.cuh"), os.path.join(CSRC, "keyhist.cuh"),
                  os.path.join(CSRC, "launch_cache.h"), os.path.join(CSRC, "fstream.cuh"),
                  os.path.join(os.path.dirname(HERE), "include", "spec_verify.h"),
                  os.path.join(os.path.dirname(HERE), "include", "spec_lm_head.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "--expt-relaxed-constexpr",
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile libspec_verify.so next to this file; returns its path."""
    if not force and up_to_date():
        return LIB
    cmd = [nvcc(), *NVCC_FLAGS, *(extra or []), "-o", LIB + ".tmp", *SOURCES]
    if verbose:
        print(" ".join(cmd))
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout, res.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose=True, extra=sys.argv[1:]))
