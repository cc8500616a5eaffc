"""Build ``_build/libdg.so`` from ``csrc/`` with nvcc for sm_103a (parallel translation units); rebuilt
whenever the digest of its sources differs from the one recorded beside it."""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libdg.so")

SOURCES = ["dg_api.cu", "dg_inst_normal.cu", "dg_inst_contiguous.cu", "dg_inst_masked.cu", "dg_inst_kgrouped.cu",
           "dg_inst_bs.cu", "dg_inst_decode.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdg")


STAMP = LIB + ".sha256"
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC"]


def source_digest() -> str:
    """SHA-256 over every input of the build: the CUDA sources and headers, the public headers, this
    script and the compiler flags. The library is rebuilt whenever it differs from the digest recorded
    beside it (file times are not trusted: a copied tree can carry a library newer than its sources)."""
    h = hashlib.sha256()
    files = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC))
    files += sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE))
    files.append(os.path.abspath(__file__))
    for f in files:
        h.update(os.path.relpath(f, ROOT).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(FLAGS + SOURCES).encode())
    return h.hexdigest()


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(STAMP)):
        return False
    with open(STAMP) as f:
        return f.read().strip() == source_digest()


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every translation unit in parallel and link the shared library; returns its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and up_to_date():
        return LIB
    digest = source_digest()
    cc = nvcc()
    flags = FLAGS + ["-I", INCLUDE, "-I", CSRC]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or ptxas_info or p.returncode != 0:
            sys.stderr.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [cc, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "--no-undefined", *objs, "-o", tmp]
    subprocess.run(link, check=True)
    os.replace(tmp, LIB)
    with open(STAMP + f".tmp{os.getpid()}", "w") as f:
        f.write(digest + "\n")
    os.replace(STAMP + f".tmp{os.getpid()}", STAMP)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv))
