"""GB300-native (sm_103a) MoE decode layer: router + biased top-k, MXFP4 routed
SwiGLU experts with weighted combine, bf16 shared expert, residual + RMSNorm.

The compute path is the CUDA library `libmoe_decode.so` behind the C ABI in
include/moe_decode.h; this package only marshals arguments (PyTorch tensors
supply device memory and streams).
"""
import ctypes

import torch

from ._binding import (MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA,
                       MOE_ERR_ALLOC, MOE_ERR_TIMEOUT, MoEDims, MoEError, MoEWeights, check, lib,
                       status_string)

__all__ = ["MoELayer", "MoEDims", "MoEWeights", "MoEError", "mxfp4_pack", "mxfp4_pack_device",
           "mxfp4_repack", "mxfp4_retile_device",
           "mxfp4_packed_bytes", "status_string", "lib", "MOE_OK", "MOE_ERR_INVALID_ARG",
           "MOE_ERR_UNSUPPORTED", "MOE_ERR_CUDA", "MOE_ERR_ALLOC", "MOE_ERR_TIMEOUT"]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(None)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _expect(t, dtype, shape, name, device=True):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name}: want {dtype} {tuple(shape)} contiguous, "
                         f"got {t.dtype} {tuple(t.shape)}")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


class MoELayer:
    """One MoE decode layer bound to borrowed device weight tensors.

    weights: dict with router_w bf16 [E,d], router_bias f32 [E], w_gu_q u8
    [E,2f,d/2], w_gu_s u8 [E,2f,d/32], w_d_q u8 [E,d,f/2], w_d_s u8 [E,d,f/32],
    shared_gu bf16 [2fs,d], shared_d bf16 [d,fs], rms_gamma bf16 [d].
    mxfp4_layout: how the expert bytes are laid out: 0 canonical, 1 tiled (FC1
    in layout 2, FC2 in layout 1), 3 UMMA (FC1 in layout 4, FC2 in layout 3);
    by default the dict's "mxfp4_layout" entry, else 0.  Weights not in the
    chosen path's layouts are relaid into a copy the layer owns.
    expert_path: 1 = mma.sync tensor cores with register dequantisation
    (tiled layouts), 2 = tcgen05 block-scaled MMAs (UMMA layouts), 0 (default)
    = both kept, path 1 at B = 1 and path 2 from B = 2.
    """

    def __init__(self, d, f, n_experts, top_k, f_shared, max_batch, weights,
                 routed_scale=2.5, rms_eps=1e-6, mxfp4_layout=None, expert_path=0):
        if mxfp4_layout is None:
            mxfp4_layout = int(weights.get("mxfp4_layout", 0))
        self.dims = MoEDims(d, f, n_experts, top_k, f_shared, max_batch, routed_scale, rms_eps,
                            mxfp4_layout, int(expert_path))
        E, fs = n_experts, f_shared
        spec = {
            "router_w": (torch.bfloat16, (E, d)), "router_bias": (torch.float32, (E,)),
            "w_gu_q": (torch.uint8, (E, 2 * f, d // 2)), "w_gu_s": (torch.uint8, (E, 2 * f, d // 32)),
            "w_d_q": (torch.uint8, (E, d, f // 2)), "w_d_s": (torch.uint8, (E, d, f // 32)),
            "shared_gu": (torch.bfloat16, (2 * fs, d)), "shared_d": (torch.bfloat16, (d, fs)),
            "rms_gamma": (torch.bfloat16, (d,)),
        }
        for name, (dt, shape) in spec.items():
            _expect(weights[name], dt, shape, name)
        self._weights = dict(weights)   # keep the borrowed tensors alive
        w = MoEWeights(*[weights[n].data_ptr() for n in spec])
        h = ctypes.c_void_p()
        check(lib().moe_layer_create(ctypes.byref(self.dims), ctypes.byref(w), ctypes.byref(h)),
              "moe_layer_create")
        self._h = h
        self.device = weights["router_w"].device
        self._next = None

    # -- lifetime ---------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().moe_layer_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # -- calls --------------------------------------------------------------
    def router_topk(self, x, idx=None, w=None, stream=None):
        B = x.shape[0]
        k = self.dims.top_k
        _expect(x, torch.bfloat16, (B, self.dims.d), "x")
        if idx is None:
            idx = torch.empty((B, k), dtype=torch.int32, device=x.device)
        if w is None:
            w = torch.empty((B, k), dtype=torch.float32, device=x.device)
        check(lib().moe_router_topk(self._h, _stream(stream), _ptr(x), B, _ptr(idx), _ptr(w)),
              "moe_router_topk")
        return idx, w

    def forward(self, x, residual, out=None, stream=None):
        B = x.shape[0]
        _expect(x, torch.bfloat16, (B, self.dims.d), "x")
        _expect(residual, torch.bfloat16, (B, self.dims.d), "residual")
        if out is None:
            out = torch.empty_like(x)
        check(lib().moe_decode_forward(self._h, _stream(stream), _ptr(x), B, _ptr(residual),
                                       _ptr(out)), "moe_decode_forward")
        return out

    def forward_host(self, x, residual, out, stream=None):
        """Host (CPU) bf16 tensors; residual and out are written in place."""
        B = x.shape[0]
        for t, n in ((x, "x"), (residual, "residual"), (out, "out")):
            _expect(t, torch.bfloat16, (B, self.dims.d), n, device=False)
            if t.is_cuda:
                raise ValueError(f"{n} must be a host tensor")
        check(lib().moe_decode_forward_host(self._h, _stream(stream), _ptr(x), B, _ptr(residual),
                                            _ptr(out)), "moe_decode_forward_host")
        return out

    def forward_debug(self, x, residual, out=None, stream=None):
        B = x.shape[0]
        d, k, f = self.dims.d, self.dims.top_k, self.dims.f
        if out is None:
            out = torch.empty_like(x)
        y_r = torch.empty((B, d), dtype=torch.float32, device=x.device)
        y_s = torch.empty((B, d), dtype=torch.float32, device=x.device)
        h = torch.empty((B, k, f), dtype=torch.float32, device=x.device)
        z = torch.empty((B, d), dtype=torch.float32, device=x.device)
        o32 = torch.empty((B, d), dtype=torch.float32, device=x.device)
        check(lib().moe_decode_forward_debug(self._h, _stream(stream), _ptr(x), B, _ptr(residual),
                                             _ptr(out), _ptr(y_r), _ptr(y_s), _ptr(h), _ptr(z),
                                             _ptr(o32)),
              "moe_decode_forward_debug")
        return dict(out=out, y_routed=y_r, y_shared=y_s, h=h, z=z, out_f32=o32)

    def debug_dequant(self, expert, which, stream=None):
        d, f = self.dims.d, self.dims.f
        shape = (2 * f, d) if which == 0 else (d, f)
        out = torch.empty(shape, dtype=torch.float32, device=self.device)
        check(lib().moe_debug_dequant(self._h, _stream(stream), int(expert), int(which), _ptr(out)),
              "moe_debug_dequant")
        return out

    def set_prefetch_next(self, other):
        self._next = other
        check(lib().moe_set_prefetch_next(self._h, other._h if other is not None else None),
              "moe_set_prefetch_next")

    def status(self):
        v = ctypes.c_int()
        check(lib().moe_layer_status(self._h, ctypes.byref(v)), "moe_layer_status")
        return v.value

    def set_act_format(self, fmt):
        """Routed experts' activations: 0 exact (default), 1 MXFP8 (the
        tensor-core path at any B, the mma.sync path at B = 1; see
        moe_set_act_format)."""
        check(lib().moe_set_act_format(self._h, int(fmt)), "moe_set_act_format")

    def debug_set_fault(self, fault, wait_ns=0):
        """Failure-detection test hook (see moe_debug_set_fault): fault 1 makes
        the one-row expert kernel's grid-wide barrier wait expire after
        wait_ns (one CTA does not arrive)."""
        check(lib().moe_debug_set_fault(self._h, int(fault), int(wait_ns)),
              "moe_debug_set_fault")

    def set_timing(self, enable):
        check(lib().moe_set_timing(self._h, int(bool(enable))), "moe_set_timing")

    def get_timing(self):
        """[router + top-k, FC1, FC2, 0 (no phase of its own), tail, layer] in us
        (see moe_get_timing)."""
        arr = (ctypes.c_float * 6)()
        check(lib().moe_get_timing(self._h, arr, 6), "moe_get_timing")
        return list(arr)

    def set_trace(self, enable):
        check(lib().moe_set_trace(self._h, int(bool(enable))), "moe_set_trace")

    def get_trace(self):
        """{kernel: (start_us, end_us)} of the last traced forward, relative to
        the earliest kernel start; kernels that did not run are left out."""
        arr = (ctypes.c_ulonglong * 10)()
        check(lib().moe_get_trace(self._h, arr, 10), "moe_get_trace")
        names = ["router", "topk", "fc1", "fc2", "tail"]
        ran = [i for i in range(5) if arr[2 * i] <= arr[2 * i + 1]]
        if not ran:
            return {}
        t0 = min(arr[2 * i] for i in ran)
        return {names[i]: ((arr[2 * i] - t0) / 1e3, (arr[2 * i + 1] - t0) / 1e3) for i in ran}

    def launches_per_forward(self, B):
        return lib().moe_launches_per_forward(self._h, int(B))


def mxfp4_packed_bytes(rows, k, layout=0):
    sb = ctypes.c_size_t()
    qb = lib().mxfp4_packed_bytes(int(rows), int(k), int(layout), ctypes.byref(sb))
    return qb, sb.value


def mxfp4_pack(w, layout=0):
    """Host packer: w CPU float32 [rows, k] -> (q uint8 [rows, k/2], s uint8 [rows, k/32])
    in the given layout (0 canonical, 1 tiled rows, 2 tiled gate/up pairs, 3 UMMA
    rows, 4 UMMA gate/up pairs)."""
    if w.is_cuda or w.dtype != torch.float32 or w.dim() != 2:
        raise ValueError("mxfp4_pack wants a CPU float32 matrix")
    w = w.contiguous()
    rows, k = w.shape
    q = torch.empty((rows, k // 2), dtype=torch.uint8)
    s = torch.empty((rows, k // 32), dtype=torch.uint8)
    check(lib().mxfp4_pack(_ptr(w), rows, k, _ptr(q), _ptr(s), int(layout)), "mxfp4_pack")
    return q, s


def mxfp4_pack_device(w, q=None, s=None, stream=None, layout=0):
    """Device packer: w CUDA float32 [rows, k] -> q, s on the same device."""
    if not w.is_cuda or w.dtype != torch.float32 or w.dim() != 2:
        raise ValueError("mxfp4_pack_device wants a CUDA float32 matrix")
    w = w.contiguous()
    rows, k = w.shape
    if q is None:
        q = torch.empty((rows, k // 2), dtype=torch.uint8, device=w.device)
    if s is None:
        s = torch.empty((rows, k // 32), dtype=torch.uint8, device=w.device)
    check(lib().mxfp4_pack_device(_stream(stream), _ptr(w), rows, k, _ptr(q), _ptr(s),
                                  int(layout)), "mxfp4_pack_device")
    return q, s


def mxfp4_repack(q, s, src, dst):
    """Host conversion of one matrix's packed bytes (CPU uint8 [rows, k/2] and
    [rows, k/32]) from layout `src` to layout `dst` (0 to 4)."""
    if q.is_cuda or s.is_cuda or q.dtype != torch.uint8 or s.dtype != torch.uint8:
        raise ValueError("mxfp4_repack wants CPU uint8 tensors")
    q = q.contiguous()
    s = s.contiguous()
    rows, k = q.shape[0], q.shape[1] * 2
    qo = torch.empty_like(q)
    so = torch.empty_like(s)
    check(lib().mxfp4_repack(_ptr(q), _ptr(s), rows, k, int(src), int(dst), _ptr(qo), _ptr(so)),
          "mxfp4_repack")
    return qo, so


def mxfp4_retile_device(q, s, layout, stream=None):
    """Canonical packed bytes (CUDA uint8 [..., rows, k/2] and [..., rows, k/32],
    matrices stacked on the leading dims) -> new tensors in tiled or UMMA layout 1 to 4."""
    if not (q.is_cuda and s.is_cuda) or q.dtype != torch.uint8 or s.dtype != torch.uint8:
        raise ValueError("mxfp4_retile_device wants CUDA uint8 tensors")
    q = q.contiguous()
    s = s.contiguous()
    rows, k = q.shape[-2], q.shape[-1] * 2
    n_mat = q.numel() // (rows * (k // 2))
    qo = torch.empty_like(q)
    so = torch.empty_like(s)
    check(lib().mxfp4_retile_device(_stream(stream), _ptr(q), _ptr(s), n_mat, rows, k, int(layout),
                                    _ptr(qo), _ptr(so)), "mxfp4_retile_device")
    return qo, so
