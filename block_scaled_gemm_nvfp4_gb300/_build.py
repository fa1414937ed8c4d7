"""Build libnvfp4 (the CUDA kernels and the C ABI) in-tree for sm_103a.

One nvcc invocation per translation unit, run in parallel, then one link
step into ``_lib/libnvfp4.so``.  The quantiser is compiled without FMA
contraction (every FP32 step there is a single IEEE round-to-nearest
operation); nothing is built with fast-math.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT, "libnvfp4.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
UNITS = {
    "api.cu": [],
    "quantize.cu": ["-fmad=false"],
    "dequantize.cu": ["-fmad=false"],
    "gemm.cu": [],
    "qadamw.cu": ["-fmad=false"],
    "lora.cu": ["-fmad=false"],
    "ns.cu": ["-fmad=false"],
    "mma_rate.cu": [],
}


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _sources_newest():
    newest = 0.0
    for name in os.listdir(CSRC):
        newest = max(newest, os.path.getmtime(os.path.join(CSRC, name)))
    newest = max(newest, os.path.getmtime(os.path.join(ROOT, "include", "nvfp4.h")))
    return newest


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _sources_newest():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_unit(item):
        name, flags = item
        obj = os.path.join(OUT, name.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *COMMON, *flags, *extra, "-c", os.path.join(CSRC, name), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (name, res.stdout, res.stderr))
        return obj, res.stderr

    with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(compile_unit, UNITS.items()))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (res.stdout, res.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
