"""Builds the two shared libraries of the package in-tree with nvcc:

  libswaattn.so       bf16 tensors, tcgen05 kernels (the product path)
  libswaattn_fp32.so  fp32 tensors, SIMT debug kernels

Both come from csrc/swa_attn.cu, compiled for sm_103a only.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")

LIBS = {
    "bf16": ("libswaattn.so", []),
    "fp32": ("libswaattn_fp32.so", ["-DSWA_ELEM_FP32"]),
}

NVCC_FLAGS = [
    "-std=c++17", "-O3", "-lineinfo",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def lib_path(kind: str) -> str:
    return os.path.join(PKG, LIBS[kind][0])


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> None:
    """Compiles every library that is missing or older than its sources,
    in parallel. Raises RuntimeError with nvcc's output on failure."""
    nvcc = nvcc_path()
    procs = []
    for kind, (name, defs) in LIBS.items():
        out = os.path.join(PKG, name)
        if not force and not _stale(out):
            continue
        tmp = out + ".tmp"
        cmd = [nvcc, *NVCC_FLAGS, *defs, "-o", tmp, os.path.join(CSRC, "swa_attn.cu")]
        if verbose:
            print(" ".join(cmd))
        procs.append((out, tmp, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.STDOUT, text=True)))
    errors = []
    for out, tmp, p in procs:
        log, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"{os.path.basename(out)}:\n{log}")
        else:
            os.replace(tmp, out)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))


if __name__ == "__main__":
    build(force=True, verbose=True)
