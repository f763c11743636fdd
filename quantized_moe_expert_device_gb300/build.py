"""Builds libgqmm.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles in parallel to an object under _build/, then nvcc links the shared
library next to this file.  Usage:  python -m quantized_moe_expert_device_gb300.build
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libgqmm.so")
SOURCES = ["api.cu", "quantize.cu", "route.cu", "gemm_tc.cu", "gemm_simt.cu", "noalloc.cu", "gemv.cu", "gemv_mma.cu", "mlp.cu", "gemm_nn.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; libgqmm needs the CUDA 13 toolkit")


def _cuda_lib_dirs(nvcc: str):
    root = os.path.dirname(os.path.dirname(nvcc))
    dirs = []
    for d in ("lib64", "lib64/stubs", "targets/sbsa-linux/lib", "targets/sbsa-linux/lib/stubs",
              "targets/x86_64-linux/lib", "targets/x86_64-linux/lib/stubs"):
        p = os.path.join(root, d)
        if os.path.isdir(p):
            dirs.append(p)
    return dirs


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    common = ["-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if ptxas_info:
        common += ["-Xptxas", "-v"]
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    headers.append(os.path.join(ROOT, "include", "gqmm.h"))
    newest_header = max(os.path.getmtime(h) for h in headers)

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        if (not ptxas_info and os.path.exists(o) and os.path.getmtime(o) > os.path.getmtime(s)
                and os.path.getmtime(o) > newest_header):
            return o, ""
        r = subprocess.run([nvcc, *common, "-c", s, "-o", o], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return o, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    logs = "".join(log for _, log in results)
    if verbose and logs:
        print(logs, file=sys.stderr)
    objs = [o for o, _ in results]
    link = [nvcc, "-shared", *ARCH, "-o", LIB + ".tmp", *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv))
