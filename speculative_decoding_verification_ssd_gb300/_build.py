"""Builds libssd.so (the C-ABI CUDA library) in-tree for sm_103a.

Each translation unit is compiled in parallel with nvcc
(-gencode arch=compute_103a,code=sm_103a), then linked into
``speculative_decoding_verification_ssd_gb300/libssd.so`` with the CUDA
runtime linked statically.  No cmake, no torch extension machinery.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libssd.so")

SOURCES = ["ssd_unit.cu", "ssd_stream.cu", "ssd_stream_wide.cu", "ssd_slice.cu", "ssd_reshape.cu", "ssd_api.cu", "ssd_fanout.cpp", "ssd_backup.cu",
           "ssd_diag.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libssd")


def _inputs_digest() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            p = os.path.join(d, name)
            if os.path.isfile(p):
                h.update(name.encode())
                h.update(open(p, "rb").read())
    h.update(" ".join(ARCH).encode())
    h.update(open(__file__, "rb").read())
    return h.hexdigest()


def source_digest(names=None) -> str:
    """Digest of kernel sources (used to tag profiles taken of a build): all of csrc/,
    or only the named files."""
    h = hashlib.sha256()
    for name in sorted(names if names is not None else os.listdir(CSRC)):
        p = os.path.join(CSRC, name)
        if os.path.isfile(p):
            h.update(name.encode())
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def stream_kernel_digest() -> str:
    """Digest of the streaming kernel's translation unit: ssd_stream.cu and the
    device headers it includes."""
    return source_digest(["ssd_stream.cu"] + [n for n in os.listdir(CSRC) if n.endswith(".cuh")])


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    stamp = os.path.join(BUILD, "stamp")
    digest = _inputs_digest()
    if (not force and os.path.exists(LIB) and os.path.exists(stamp)
            and open(stamp).read().strip() == digest):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
              "--expt-relaxed-constexpr", "-Xcompiler", "-Wall"]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, src + ".o")
        cmd = [cc] + ARCH + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
