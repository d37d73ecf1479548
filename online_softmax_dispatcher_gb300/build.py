"""Build libosd_softmax.so in-tree (online_softmax_dispatcher_gb300/_build/).

Every CUDA translation unit is compiled for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``), in parallel, then linked with
nvcc into one shared library.  The C ABI it exports is include/softmax.h.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_NAME = "libosd_softmax.so"
LIB_PATH = os.path.join(BUILD, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_SOURCES = ["abi.cu", "k_rowgroup_f32.cu", "k_rowgroup_f16.cu", "k_rowgroup_bf16.cu", "k_block.cu",
                "k_stream.cu", "k_splitk.cu", "k_tma.cu", "k_bwd.cu", "k_wide.cu",
                "noalloc.cu", "k_masked.cu", "k_norm_f32.cu", "k_norm_f16.cu", "k_norm_bf16.cu", "k_grid.cu"]
HOST_SOURCES = ["plan.cpp"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libosd_softmax.so")


def _fingerprint() -> str:
    h = hashlib.sha256()
    files = sorted(os.listdir(CSRC)) + ["../../include/softmax.h", "../build.py"]
    for name in files:
        path = os.path.normpath(os.path.join(CSRC, name))
        if os.path.isfile(path):
            h.update(name.encode())
            with open(path, "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def _compile(cmd: list[str]) -> tuple[list[str], int, str]:
    p = subprocess.run(cmd, capture_output=True, text=True)
    return cmd, p.returncode, p.stdout + p.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link; skipped when the sources are unchanged since the last build."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "fingerprint")
    fp = _fingerprint()
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == fp:
                return LIB_PATH
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC]
    cmds, objs = [], []
    for src in CUDA_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj, *ARCH, "-lineinfo", *common,
               "-Xcompiler", "-fPIC,-fvisibility=hidden"]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        cmds.append(cmd)
    for src in HOST_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        cmds.append(["g++", "-c", os.path.join(CSRC, src), "-o", obj, "-O2", "-std=c++17", "-fPIC",
                     "-fvisibility=hidden", "-Wall", "-I", INCLUDE, "-I", CSRC])
    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        results = list(ex.map(_compile, cmds))
    failed = False
    for cmd, rc, out in results:
        if verbose or rc != 0 or ptxas_info:
            sys.stderr.write(" ".join(cmd) + "\n" + out)
        failed |= rc != 0
    if failed:
        raise RuntimeError("libosd_softmax.so: compilation failed (see stderr)")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, "-shared", *ARCH, "-o", tmp, *objs, "-cudart", "static"]
    _, rc, out = _compile(link)
    if rc != 0:
        sys.stderr.write(" ".join(link) + "\n" + out)
        raise RuntimeError("libosd_softmax.so: link failed")
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(fp)
    return LIB_PATH


if __name__ == "__main__":
    import argparse

    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=True, ptxas_info=a.ptxas_info))
