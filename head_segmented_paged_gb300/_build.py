"""Build libsegkv.so in-tree for sm_103a with nvcc (no CMake)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsegkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_SOURCES = ["append.cu", "prefill.cu", "decode.cu", "decode_mma.cu", "decode_noalloc.cu", "rope.cu",
              "transfer.cu",
              "ffn.cu", "mass.cu", "topk.cu"]
CPP_SOURCES = ["segkv_host.cpp"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _cuda_home(nvcc: str) -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _deps() -> list[str]:
    out = [os.path.join(ROOT, "include", "segkv.h")]
    for f in os.listdir(CSRC):
        out.append(os.path.join(CSRC, f))
    out.append(__file__)
    return out


def _stale(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and not _stale(LIB):
        return LIB
    nvcc = _nvcc()
    home = _cuda_home(nvcc)
    os.makedirs(BUILD, exist_ok=True)
    cmds = []
    objs = []
    for s in CU_SOURCES:
        o = os.path.join(BUILD, s + ".o")
        objs.append(o)
        cmd = [nvcc, "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
               "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, s), "-o", o]
        if ptxas_verbose:
            cmd.insert(1, "-Xptxas=-v")
        cmds.append(cmd)
    for s in CPP_SOURCES:
        o = os.path.join(BUILD, s + ".o")
        objs.append(o)
        cmds.append(["g++", "-O2", "-std=c++17", "-fPIC", "-I", os.path.join(home, "include"),
                     "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, s),
                     "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        for cmd, r in ex.map(run, cmds):
            if verbose or ptxas_verbose or r.returncode != 0:
                print(" ".join(cmd))
                print(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"compile failed: {cmd[-3]}")
    tmp = LIB + f".{os.getpid()}.tmp"
    link = [nvcc, "-shared", *ARCH, "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        print(" ".join(link))
        print(r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    build(force=True, verbose=True, ptxas_verbose="-v" in sys.argv)
    print(LIB)
