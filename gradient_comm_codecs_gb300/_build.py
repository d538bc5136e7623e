"""In-tree build of libzpp.so (sm_103a) with nvcc.

    python -m gradient_comm_codecs_gb300._build [--force]

Each .cu translation unit is compiled in parallel to an object under
``_build/``; the objects are linked with the static CUDA runtime into
``libzpp.so`` next to this file.  ``-Xptxas -v`` register/spill reports go to
``_build/ptxas.log``.
"""
from __future__ import annotations

import fcntl
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libzpp.so")
SOURCES = ["zpp_abi.cu", "quant.cu", "hop.cu", "adam.cu", "ring.cu"]
HEADERS = [os.path.join(CSRC, "zpp_device.cuh"), os.path.join(CSRC, "zpp_launch.h"),
           os.path.join(INCLUDE, "zpp.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "-fmad=false", "-I", INCLUDE, "-I", CSRC, "-Xptxas", "-v"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, quiet: bool = True) -> str:
    os.makedirs(BUILD, exist_ok=True)
    with open(os.path.join(BUILD, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and not _stale():
            return LIB
        nvcc = _nvcc()
        procs = []
        for s in SOURCES:
            obj = os.path.join(BUILD, s.replace(".cu", ".o"))
            cmd = [nvcc, *NVCC_FLAGS, "-c", os.path.join(CSRC, s), "-o", obj]
            procs.append((s, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                   stderr=subprocess.STDOUT, text=True)))
        log, objs, failed = [], [], []
        for s, obj, p in procs:
            out, _ = p.communicate()
            log.append(f"==== {s}\n{out}")
            objs.append(obj)
            if p.returncode != 0:
                failed.append(s)
        with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
            f.write("\n".join(log))
        if failed:
            raise RuntimeError(f"nvcc failed for {failed}:\n" + "\n".join(log))
        tmp = LIB + f".{os.getpid()}.tmp"
        subprocess.check_call([nvcc, "-shared", *ARCH, "--cudart", "static", "-o", tmp, *objs])
        os.replace(tmp, LIB)
        if not quiet:
            print("\n".join(log))
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, quiet="-v" not in sys.argv)
    print(LIB)
