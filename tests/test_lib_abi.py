"""The C-ABI library loads, exports every declared symbol, and its host-side
logic (MXFP4 host packer, argument validation) works without a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import moe_decode_step_gb300 as M
from moe_decode_step_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from moe_decode_step_gb300 import build
    build.build()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_decode.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w\*]+\s+\**\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ("moe_layer_create", "moe_layer_destroy", "moe_router_topk", "moe_decode_forward",
                 "moe_decode_forward_host", "mxfp4_pack", "mxfp4_pack_device", "mxfp4_repack",
                 "mxfp4_retile_device"):
        assert want in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(_binding.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    assert set(_declared_functions()) <= set(_binding._PROTOS)


def test_status_strings():
    assert M.status_string(0) == "ok"
    assert "unsupported" in M.status_string(2)
    assert M.status_string(99) == "unknown status"


def test_packed_bytes():
    assert M.mxfp4_packed_bytes(3072, 7168) == (3072 * 3584, 3072 * 224)
    assert M.mxfp4_packed_bytes(10, 33)[0] == 0


def _edge_matrix():
    rng = np.random.default_rng(11)
    rows = []
    base = rng.standard_normal((8, 64)).astype(np.float32)
    rows.extend(base)
    # exact midpoints of the E2M1 grid at scale 2^0 (amax pinned to 6 -> e = 0)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 4, np.float32)
    rows.append(np.concatenate([mids, -mids]))
    rows.append(np.zeros(64, np.float32))
    rows.append(np.concatenate([np.full(32, -0.0, np.float32), np.full(32, 1e-40, np.float32)]))
    rows.append((rng.standard_normal(64) * 1e30).astype(np.float32))
    rows.append((rng.standard_normal(64) * 1e-39).astype(np.float32))
    big = rng.standard_normal(64).astype(np.float32)
    big[3] = 7.9
    big[40] = -100.0
    rows.append(big)
    return np.stack(rows).astype(np.float32)


def test_library_host_packer_matches_oracle_bytes():
    for w in (_edge_matrix(), np.random.default_rng(3).standard_normal((37, 1024)).astype(np.float32)):
        q, s = M.mxfp4_pack(torch.from_numpy(w))
        qo, so = oracle.mxfp4_pack(w)
        assert np.array_equal(s.numpy(), so)
        assert np.array_equal(q.numpy(), qo)


def test_create_rejects_bad_dims_and_null_weights_before_touching_the_gpu():
    L = M.lib()
    w = M.MoEWeights()
    h = ctypes.c_void_p()
    good = dict(d=1024, f=256, n_experts=64, top_k=4, f_shared=256, max_batch=1,
                routed_scale=2.5, rms_eps=1e-6, mxfp4_layout=0)
    for bad in (dict(d=1000), dict(f=100), dict(f=384), dict(top_k=0), dict(top_k=65), dict(n_experts=2),
                dict(max_batch=65), dict(max_batch=0), dict(f_shared=0), dict(d=16384),
                dict(d=7936), dict(f=3328), dict(f=4096), dict(f_shared=4352),
                dict(expert_path=3), dict(expert_path=-1)):
        dims = M.MoEDims(**{**good, **bad})
        assert L.moe_layer_create(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(h)) == \
            M.MOE_ERR_INVALID_ARG, bad
    for layout in (2, 4, 5):
        dims = M.MoEDims(**{**good, "mxfp4_layout": layout})
        assert L.moe_layer_create(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(h)) == \
            M.MOE_ERR_UNSUPPORTED
    dims = M.MoEDims(**good)
    assert L.moe_layer_create(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(h)) == \
        M.MOE_ERR_INVALID_ARG   # null weight pointers
    assert L.moe_layer_create(None, ctypes.byref(w), ctypes.byref(h)) == M.MOE_ERR_INVALID_ARG


def test_calls_on_a_null_handle_are_rejected():
    L = M.lib()
    x = ctypes.c_void_p(16)
    assert L.moe_decode_forward(None, None, x, 1, x, x) == M.MOE_ERR_INVALID_ARG
    assert L.moe_router_topk(None, None, x, 1, x, x) == M.MOE_ERR_INVALID_ARG
    assert L.moe_debug_dequant(None, None, 0, 0, x) == M.MOE_ERR_INVALID_ARG
    assert L.moe_layer_destroy(None) == M.MOE_OK
    v = ctypes.c_int()
    assert L.moe_layer_status(None, ctypes.byref(v)) == M.MOE_ERR_INVALID_ARG
    assert L.moe_launches_per_forward(None, 1) == -1
    assert L.mxfp4_pack(None, 1, 32, x, x, 0) == M.MOE_ERR_INVALID_ARG
