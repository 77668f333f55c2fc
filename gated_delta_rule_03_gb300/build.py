"""Build libgdr.so, the sm_103a CUDA library, in-tree with nvcc.

Each translation unit under csrc/ is compiled in parallel into _build/, then
linked into gated_delta_rule_03_gb300/libgdr.so with the CUDA runtime linked
statically (the library then needs only the driver). The driver API entry
points the library uses are fetched at run time through the runtime, so no
-lcuda is needed. Register and spill counts from ptxas go to _build/ptxas.log.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgdr.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["gdr_api.cu", "decode.cu", "prefill_exact.cu", "solve_tc.cu", "prefill_tc.cu", "channel_tc.cu", "noalloc.cu",
           "epilogue.cu"]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libgdr.so")


def _compile(src):
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v", "-I", os.path.join(HERE, "..", "include"), "-c",
           os.path.join(CSRC, src), "-o", obj]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{proc.stderr}")
    return obj, proc.stderr


def build(verbose=False):
    """Compile every CUDA source and link libgdr.so; returns the library path."""
    os.makedirs(BUILD, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as log:
        for obj, err in results:
            log.write(f"== {os.path.basename(obj)}\n{err}\n")
            if verbose:
                print(err, file=sys.stderr)
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[r[0] for r in results]]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
