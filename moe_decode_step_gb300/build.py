"""Build the CUDA extension in tree: moe_decode_step_gb300/libmoe_decode.so (sm_103a)."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libmoe_decode.so")
SOURCES = ["csrc/moe_decode.cu", "csrc/noalloc.cu"]
HEADERS = ["csrc/common.cuh", "csrc/mxfp4.cuh", "csrc/planes.cuh", "csrc/stream.cuh",
           "csrc/tc.cuh", "csrc/topk.cuh", "csrc/tail.cuh"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = SOURCES + HEADERS + [os.path.join(ROOT, "include", "moe_decode.h")]
    return any(os.path.getmtime(os.path.join(HERE, p)) > t for p in deps)


def build(force=False, verbose=False):
    if force or _stale():
        cmd = ["nvcc", *NVCC_FLAGS, "-I" + os.path.join(ROOT, "include"), "-o", LIB,
               *[os.path.join(HERE, s) for s in SOURCES]]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.check_call(cmd)
    return LIB
