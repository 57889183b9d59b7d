"""Build ``libtq.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process, in parallel, then one
link step produces the shared library next to this file.  Objects go to
``_build/`` beside it.  Nothing here needs a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtq.so")
# (source, extra flags, object name); the kernels of each key width 1 .. 8 are
# one compilation of tq_inst.cu, so the widths build in parallel
SOURCES = [("tq_host.cpp", [], "tq_host.o"), ("tq_encode.cu", [], "tq_encode.o"), ("tq_decode.cu", [], "tq_decode.o"),
           ("tq_octopus.cu", [], "tq_octopus.o"), ("tq_selftest.cu", [], "tq_selftest.o"),
           ("tq_prefill_tc.cu", [], "tq_prefill_tc.o")]
SOURCES += [("tq_inst.cu", [f"-DTQ_KB={kb}"], f"tq_inst_k{kb}.o") for kb in range(1, 9)]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    nv = shutil.which("nvcc")
    if nv is None and os.path.exists("/usr/local/cuda/bin/nvcc"):
        nv = "/usr/local/cuda/bin/nvcc"
    if nv is None:
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libtq.so")
    return nv


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "tq.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-I", INCLUDE, "-Xcompiler", "-fPIC,-fvisibility=hidden"]
    procs = []
    objs = []
    for src, flags, name in SOURCES:
        obj = os.path.join(BUILD, name)
        objs.append(obj)
        cmd = [nvcc] + common + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((cmd, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = LIB + ".tmp"
    link = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
