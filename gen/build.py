"""Compile the generator's host library (gcc) and device library (nvcc), in tree."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "libmoegen.so")
DEVICE_LIB = os.path.join(HERE, "libmoegen_cuda.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(os.path.join(HERE, s)) > t for s in sources)


def build_host(force=False):
    srcs = ["moegen.c", "moegen_core.h"]
    if force or _stale(HOST_LIB, srcs):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", HOST_LIB,
                               os.path.join(HERE, "moegen.c"), "-lpthread"])
    return HOST_LIB


def build_device(force=False):
    srcs = ["moegen_cuda.cu", "moegen_core.h"]
    if force or _stale(DEVICE_LIB, srcs):
        subprocess.check_call(["nvcc", *ARCH, "-O3", "-fmad=false", "-lineinfo",
                               "-Xcompiler", "-fPIC", "-shared", "-o", DEVICE_LIB,
                               os.path.join(HERE, "moegen_cuda.cu")])
    return DEVICE_LIB
