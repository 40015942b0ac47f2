"""In-tree build of the CUDA libraries (nvcc for sm_103a, no cmake).

``libdllm.so``        the decoder (include/dllm.h)
``libdllm_synth.so``  the seeded input generator (include/dllm_synth.h)

Translation units compile in parallel; a unit is rebuilt when it or any
header of the source directory is newer than its object.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_lib")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-cudart", "shared"]
LIB_UNITS = ["api", "attention", "gemm_plain", "gemm_qkv", "gemm_resid", "gemm_swiglu", "gemm_lmhead",
             "step_hd64", "step_hd128"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_header() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(HERE, "..", "include", "*.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(unit: str, nvcc: str, hdr_time: float, verbose: bool) -> str:
    src = os.path.join(CSRC, unit + ".cu")
    obj = os.path.join(OUT, unit + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_time):
        return obj
    cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {unit}.cu:\n{r.stdout}\n{r.stderr}")
    return obj


def _link(objs, out, nvcc, verbose):
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", out]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {out} failed:\n{r.stdout}\n{r.stderr}")


def build(verbose: bool = False) -> None:
    os.makedirs(OUT, exist_ok=True)
    nvcc = _nvcc()
    hdr = _newest_header()
    units = LIB_UNITS + ["synth_fill"]
    with ThreadPoolExecutor(max_workers=len(units)) as ex:
        objs = dict(zip(units, ex.map(lambda u: _compile(u, nvcc, hdr, verbose), units)))
    lib = os.path.join(OUT, "libdllm.so")
    lib_objs = [objs[u] for u in LIB_UNITS]
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in lib_objs):
        _link(lib_objs, lib, nvcc, verbose)
    synth = os.path.join(OUT, "libdllm_synth.so")
    if not os.path.exists(synth) or os.path.getmtime(synth) < os.path.getmtime(objs["synth_fill"]):
        _link([objs["synth_fill"]], synth, nvcc, verbose)


if __name__ == "__main__":
    build(verbose=True)
