"""In-tree build of the moestep CUDA library (nvcc, sm_103a) and its loader path."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB_DIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIB_DIR, "libmoestep.so")
SOURCES = ["api.cu", "route.cu", "misc.cu", "expert_gemm.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_flags() -> list[str]:
    return ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
            "-I", CSRC, *ARCH]


def build(quiet: bool = True, extra: list[str] | None = None) -> str:
    """Compile every translation unit in parallel, then link libmoestep.so."""
    os.makedirs(LIB_DIR, exist_ok=True)
    objs, procs = [], []
    out = subprocess.DEVNULL if quiet else None
    for src in SOURCES:
        obj = os.path.join(LIB_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = ["nvcc", *nvcc_flags(), *(extra or []), "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=out, stderr=subprocess.PIPE, text=True)))
    errs = []
    for cmd, p in procs:
        _, err = p.communicate()
        if p.returncode != 0:
            errs.append(f"{' '.join(cmd)}\n{err}")
    if errs:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errs))
    link = ["nvcc", "-shared", *ARCH, *objs, "-o", LIB, "-lcudart"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {r.stderr}")
    return LIB
