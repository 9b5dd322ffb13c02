"""ctypes binding of libmoe_decode.so (argument marshalling only).

Every compute step runs in the CUDA library; if the library is missing this
module raises instead of falling back to anything else.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_decode.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_ALLOC = 4
MOE_ERR_TIMEOUT = 5

_P = ctypes.c_void_p


class MoEDims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("f", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("f_shared", ctypes.c_int32),
                ("max_batch", ctypes.c_int32), ("routed_scale", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("mxfp4_layout", ctypes.c_int32),
                ("expert_path", ctypes.c_int32)]


class MoEWeights(ctypes.Structure):
    _fields_ = [("router_w", _P), ("router_bias", _P), ("w_gu_q", _P), ("w_gu_s", _P),
                ("w_d_q", _P), ("w_d_s", _P), ("shared_gu", _P), ("shared_d", _P),
                ("rms_gamma", _P)]


class MoEError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        cuda = ""
        if code == MOE_ERR_CUDA and _lib is not None:
            cuda = f" (cudaError {_lib.moe_last_cuda_error()})"
        super().__init__(f"{what}: {status_string(code)}{cuda}")


_lib = None

# name -> (restype, argtypes)
_PROTOS = {
    "moe_layer_create": (ctypes.c_int, [ctypes.POINTER(MoEDims), ctypes.POINTER(MoEWeights),
                                        ctypes.POINTER(_P)]),
    "moe_layer_destroy": (ctypes.c_int, [_P]),
    "moe_router_topk": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _P, _P]),
    "moe_decode_forward": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _P, _P]),
    "moe_decode_forward_host": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _P, _P]),
    "moe_decode_forward_debug": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _P, _P, _P, _P, _P,
                                                _P, _P]),
    "moe_debug_dequant": (ctypes.c_int, [_P, _P, ctypes.c_int, ctypes.c_int, _P]),
    "moe_set_prefetch_next": (ctypes.c_int, [_P, _P]),
    "moe_layer_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int)]),
    "moe_set_timing": (ctypes.c_int, [_P, ctypes.c_int]),
    "moe_debug_set_fault": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_ulonglong]),
    "moe_set_act_format": (ctypes.c_int, [_P, ctypes.c_int]),
    "moe_get_timing": (ctypes.c_int, [_P, _P, ctypes.c_int]),
    "moe_launches_per_forward": (ctypes.c_int, [_P, ctypes.c_int]),
    "moe_set_trace": (ctypes.c_int, [_P, ctypes.c_int]),
    "moe_get_trace": (ctypes.c_int, [_P, _P, ctypes.c_int]),
    "mxfp4_packed_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_size_t)]),
    "mxfp4_pack": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int64, _P, _P, ctypes.c_int]),
    "mxfp4_pack_device": (ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int64, _P, _P,
                                         ctypes.c_int]),
    "mxfp4_repack": (ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                    ctypes.c_int, _P, _P]),
    "mxfp4_retile_device": (ctypes.c_int, [_P, _P, _P, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_int, _P, _P]),
    "moe_router_topk_noalloc": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_float, _P,
                                               _P]),
    "moe_router_topk_noalloc_status": (ctypes.c_int, [_P]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_last_cuda_error": (ctypes.c_int, []),
}


def lib():
    """Load the in-tree CUDA library; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _PROTOS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(code):
    return lib().moe_status_string(int(code)).decode()


def check(code, what):
    if code != MOE_OK:
        raise MoEError(code, what)
