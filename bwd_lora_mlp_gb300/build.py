"""Build liblora_mlp.so in-tree with nvcc for sm_103a.

    python -m bwd_lora_mlp_gb300.build          # build unless the library matches the sources

The library is reused only when the digest stored beside it (liblora_mlp.so.digest) equals the
digest of the current sources (every file of csrc/, the public header, this script) and of the
compiler flags; file times play no part, so a library copied in from elsewhere, or left over from
other sources, is rebuilt.

The translation units compile in parallel; the library links the CUDA runtime statically and
reaches the driver only through cudaGetDriverEntryPointByVersion, so it loads on machines
without a GPU (the host-side argument checks and the NF4 code table work there).
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
LIB = os.path.join(PKG, "liblora_mlp.so")
DIGEST = LIB + ".digest"

SOURCES = ["lm_api.cu", "lm_aux.cu", "lm_gemm_fwd.cu", "lm_gemm_bwd.cu", "lm_gemm2.cu", "lm_gemm2_nf4.cu", "lm_static_ws.cu",
           "lm_dual.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblora_mlp.so")


def _deps() -> list:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "lora_mlp.h"),
                                                                  os.path.abspath(__file__)]
    return sorted(f for f in files if os.path.isfile(f))


def source_digest(extra_flags=None) -> str:
    """sha256 over the build inputs: each source file's name and bytes, the target and the flags."""
    h = hashlib.sha256()
    for f in _deps():
        h.update(os.path.relpath(f, ROOT).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
        h.update(b"\0")
    # the flags without the include paths, which name this checkout's location
    flags = [f for f in ARCH + FLAGS + list(extra_flags or []) if not f.startswith("-I")]
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def up_to_date(extra_flags=None) -> bool:
    if not (os.path.exists(LIB) and os.path.exists(DIGEST)):
        return False
    with open(DIGEST) as f:
        return f.read().strip() == source_digest(extra_flags)


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    digest = source_digest(extra_flags)
    if not force and up_to_date(extra_flags):
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    flags = FLAGS + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB)
    with open(DIGEST + ".tmp", "w") as f:
        f.write(digest + "\n")
    os.replace(DIGEST + ".tmp", DIGEST)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
