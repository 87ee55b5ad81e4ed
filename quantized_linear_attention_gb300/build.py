"""In-tree builds: the CUDA C-ABI library ``liblq.so`` (sm_103a) and the workload generator.

``liblq.so`` is built with nvcc directly (no torch extension machinery): every
translation unit is compiled for ``sm_103a`` only, in parallel, then linked as a
shared library. Outputs go to ``quantized_linear_attention_gb300/_build/``.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")

CUDA_SOURCES = ["lq_kernels.cu", "lq_append.cu", "lq_step.cu", "lq_fp32.cu", "lq_api.cu"]
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    # IEEE division and square root, denormals kept, and no contraction of a*b+c:
    # the pinned path spells out every fma it wants.
    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
    "-Xptxas", "-v",
]


def nvcc() -> str:
    cand = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    p = os.path.join(cand, "bin", "nvcc")
    return p if os.path.exists(p) else (shutil.which("nvcc") or "nvcc")


def lq_library_path() -> str:
    return os.path.join(OUT_DIR, "liblq.so")


def workload_library_path() -> str:
    return os.path.join(OUT_DIR, "libqla_workload.so")


def _newer(out, srcs):
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(s) <= t for s in srcs)


def _deps():
    srcs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    srcs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return srcs


def build_workload(force: bool = False) -> str:
    out = workload_library_path()
    src = os.path.join(CSRC, "workload_gen.c")
    if not force and _newer(out, [src]):
        return out
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O3", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", src, "-o", tmp,
                    "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build_lq(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link ``liblq.so``."""
    out = lq_library_path()
    if not force and _newer(out, _deps()):
        return out
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.basename(src) + ".o")
        cmd = [cc, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with _cf.ThreadPoolExecutor(max_workers=len(CUDA_SOURCES)) as ex:
        results = list(ex.map(compile_one, CUDA_SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *[o for o, _ in results], "-o", tmp,
           "-lcudart"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
        for _, log in results:
            f.write(log)
    return out


def build_all(force: bool = False, verbose: bool = False):
    return build_workload(force), build_lq(force, verbose)


if __name__ == "__main__":
    print(build_all(force=True, verbose=True))
