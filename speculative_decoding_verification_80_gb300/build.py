"""Builds libspecdec.so in-tree from csrc/ with nvcc for sm_103a.

Translation units compile in parallel; the library links the CUDA runtime
statically, so it needs only the driver at run time.
"""
from __future__ import annotations

import concurrent.futures
import glob
import hashlib
import re
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libspecdec.so")
BUILD_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecdec.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _code_only(text: str) -> str:
    """C/C++ source without its comments (string literals kept)."""
    return re.sub(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"',
                  lambda m: m.group(0) if m.group(0).startswith('"') else " ", text, flags=re.S)


def source_digest(skip=()) -> str:
    """Hash of the code the library is built from (kernels, headers, flags),
    comments aside, so an edit to comments keeps the recorded measurements of
    the same code valid.  `skip` leaves out source files by name (the verify
    kernel's digest leaves out the MTP kernel's and the sharded verify's
    files, which it does not include)."""
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(CSRC, "*"))) + sorted(glob.glob(os.path.join(INCLUDE, "*.h")))
    for f in files:
        if os.path.basename(f) in skip:
            continue
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    h.update(" ".join(ARCH + NVCC_FLAGS[:-2]).encode())
    return h.hexdigest()[:16]


def verify_digest() -> str:
    """Digest of the sources the verify kernel is built from."""
    return source_digest(skip=("mtp_kernel.cuh", "shard_kernels.cuh", "shard_api.cu", "specdec_shard.h"))


def _up_to_date() -> bool:
    stamp = LIB + ".digest"
    if not (os.path.exists(LIB) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        return f.read().strip() == source_digest()


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and _up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs = []
    cmds = []
    for src in sources():
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmds.append([nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(cmds))) as ex:
        list(ex.map(run, cmds))
    tmp = LIB + f".tmp{os.getpid()}"
    run([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    with open(LIB + ".digest", "w") as f:
        f.write(source_digest())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
