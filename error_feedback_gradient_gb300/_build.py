"""Build libefgrad.so in-tree with nvcc for sm_103a.

Each CUDA source compiles to an object in parallel, then the objects link
into ``error_feedback_gradient_gb300/lib/libefgrad.so`` with the CUDA runtime
linked statically (the library then needs only the driver at run time).
Register / spill / shared-memory usage from ``-Xptxas -v`` is written to
``lib/ptxas.log``.
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
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "lib")
BUILD_DIR = os.path.join(ROOT, "_build")
SOURCES = ["ef_api.cu", "ef_sign.cu", "ef_topk.cu", "ef_aggregate.cu", "ef_quant.cu", "ef_codec.cu", "ef_randk.cu",
           "ef_exchange.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if p.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + p.stdout)
    return p.stdout


def build(verbose: bool = False) -> str:
    """Compile every CUDA source and link the shared library; returns its path."""
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(BUILD_DIR, exist_ok=True)
    common = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
              "-Xptxas", "-v"]
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "efgrad.h"))
    newest_header = max(os.path.getmtime(h) for h in headers)

    def compile_one(src):
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        if (os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(path)
                and os.path.getmtime(obj) >= newest_header):
            return obj, ""
        log = _run(common + ["-c", path, "-o", obj])
        return obj, log

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    logs = "".join(f"== {SOURCES[i]}\n{log}" for i, (_, log) in enumerate(results) if log)
    if logs:
        with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
            f.write(logs)
    lib = os.path.join(OUT_DIR, "libefgrad.so")
    tmp = lib + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, lib)
    if verbose:
        print(logs)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
