"""Build libfo.so (the sm_103a CUDA library) in-tree with nvcc.

Each ``csrc/*.cu`` translation unit is compiled in parallel, then linked into
``quantized_state_optimizer_gb300/_build/libfo.so`` with the CUDA runtime
linked statically.  No fast-math: IEEE division, square root and
round-to-nearest are what the method's definition requires, and
``-fmad=false`` forbids multiply-add contraction in the parity-critical
arithmetic.
"""

from __future__ import annotations

import glob
import hashlib
import os
import shutil
import subprocess
import sys
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libfo.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-I", INCLUDE, "-I", CSRC,
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfo.so")


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _fingerprint() -> str:
    h = hashlib.sha256()
    h.update(" ".join(NVCC_FLAGS).encode())
    files = _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                                + glob.glob(os.path.join(INCLUDE, "*.h")))
    for f in files:
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile and link libfo.so unless an up-to-date copy exists; return its path."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "libfo.fingerprint")
    fp = _fingerprint()
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == fp:
        return LIB
    tmpdir = tempfile.mkdtemp(dir=BUILD)
    try:
        procs = []
        objs = []
        extra = ["-Xptxas", "-v"] if verbose_ptxas else []
        for src in _sources():
            obj = os.path.join(tmpdir, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        failed = []
        for cmd, p in procs:
            out, _ = p.communicate()
            if verbose_ptxas or p.returncode != 0:
                sys.stderr.write(out.decode(errors="replace"))
            if p.returncode != 0:
                failed.append(" ".join(cmd))
        if failed:
            raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
        tmp_lib = os.path.join(tmpdir, "libfo.so")
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp_lib, *objs], check=True)
        os.replace(tmp_lib, LIB)
        with open(stamp, "w") as fh:
            fh.write(fp)
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
