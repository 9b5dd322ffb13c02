"""Seeded synthetic-input generator shared by the oracle side and the GPU side.

Holds no MoE arithmetic: only Philox4x32-10 integers turned into normal draws
(see moegen_core.h).  `normal_host` runs on CPU threads, `normal_device` fills
a CUDA float32 tensor; both give bit-identical values for the same element.
"""
import ctypes
import os

import numpy as np

from . import build as _build
from .configs import (CONFIGS, LayerConfig, activation_seed, f32, T_ROUTER_W, T_ROUTER_BIAS,
                      T_GAMMA, T_SHARED_GU, T_SHARED_D, T_X, T_RESIDUAL, T_EXPERT_GU,
                      T_EXPERT_D)

_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(_build.build_host())
        lib.moegen_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                          ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                                          ctypes.c_float, ctypes.c_void_p, ctypes.c_int]
        lib.moegen_philox.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.moegen_ln_u_host.argtypes = [ctypes.c_uint32]
        lib.moegen_ln_u_host.restype = ctypes.c_float
        lib.moegen_cos2pi_u_host.argtypes = [ctypes.c_uint32]
        lib.moegen_cos2pi_u_host.restype = ctypes.c_float
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(_build.DEVICE_LIB):
            raise RuntimeError("gen/libmoegen_cuda.so is not built (run __graft_entry__.build())")
        lib = ctypes.CDLL(_build.DEVICE_LIB)
        lib.moegen_normal_f32_device.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                                 ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                                                 ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
        lib.moegen_normal_f32_device.restype = ctypes.c_int
        _dev = lib
    return _dev


def host_threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def philox4x32_10(ctr, key):
    c = (ctypes.c_uint32 * 4)(*ctr)
    k = (ctypes.c_uint32 * 2)(*key)
    o = (ctypes.c_uint32 * 4)()
    _host_lib().moegen_philox(c, k, o)
    return list(o)


def ln_u(r):
    return _host_lib().moegen_ln_u_host(r)


def cos2pi_u(r):
    return _host_lib().moegen_cos2pi_u_host(r)


def normal_host(seed, tensor, sub, n, mean, std, start=0, nthreads=None):
    out = np.empty(int(n), dtype=np.float32)
    _host_lib().moegen_normal_f32(int(seed), int(tensor), int(sub), int(start), int(n),
                                  f32(mean), f32(std), out.ctypes.data,
                                  nthreads or host_threads())
    return out


def normal_device(seed, tensor, sub, out, mean, std, start=0, stream=None):
    """Fill the contiguous CUDA float32 tensor `out` (all of it)."""
    import torch
    assert out.is_cuda and out.dtype == torch.float32 and out.is_contiguous()
    s = stream if stream is not None else torch.cuda.current_stream(out.device)
    rc = _dev_lib().moegen_normal_f32_device(int(seed), int(tensor), int(sub), int(start),
                                             out.numel(), f32(mean), f32(std),
                                             ctypes.c_void_p(out.data_ptr()),
                                             ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"moegen device launch failed: cudaError {rc}")
    return out


def activation_x(cfg, seed, B=None):
    """x rows [B, d] as float32 (before the bf16 rounding both sides apply).

    Uncorrelated configs: the N(0, 1) draws of tensor T_X, sub-stream 0.  A
    verify batch (cfg.drafts > 0, correlation rho = cfg.corr): row r of group
    g = r // (1 + drafts) is rho * z_g + sqrt(1 - rho^2) * n_r, with n_r the
    same sub-stream-0 draws and z_g the draws of sub-stream 1 (one row per
    group), each product and the sum rounded to float32 (numpy float32
    arithmetic, no fused multiply-add), so every row is still N(0, 1) and two
    rows of a group correlate by rho**2."""
    B = cfg.B if B is None else B
    n = normal_host(seed, T_X, 0, B * cfg.d, 0.0, 1.0).reshape(B, cfg.d)
    if cfg.drafts <= 0 or cfg.corr == 0.0:
        return n
    gsize = 1 + cfg.drafts
    groups = (B + gsize - 1) // gsize
    z = normal_host(seed, T_X, 1, groups * cfg.d, 0.0, 1.0).reshape(groups, cfg.d)
    rho = np.float32(cfg.corr)
    sig = np.float32(np.sqrt(1.0 - float(cfg.corr) ** 2))
    zr = z[np.arange(B) // gsize]
    return (rho * zr + sig * n).astype(np.float32)

