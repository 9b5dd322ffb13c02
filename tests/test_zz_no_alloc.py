"""The allocation-free router + top-k entry point (for callers that cannot call
cudaMalloc) must give the same routing as the layer's moe_router_topk.

It is called through the C ABI with plain device pointers; every buffer here
is allocated by the test, never by the entry point.  Two calls in a row check
that the shared scratch array carries nothing over from one call to the next.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import gen
import oracle
import moe_decode_step_gb300 as M
from gen.configs import CONFIGS, T_ROUTER_W, T_ROUTER_BIAS, T_X
from moe_decode_step_gb300 import synthetic

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(router_w, bias, x, k, routed_scale):
    B, d = x.shape
    E = router_w.shape[0]
    idx = torch.full((B, k), -1, dtype=torch.int32, device=x.device)
    w = torch.full((B, k), -1.0, dtype=torch.float32, device=x.device)
    rc = M.lib().moe_router_topk_noalloc(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), _ptr(router_w), _ptr(bias),
        _ptr(x), B, d, E, k, float(routed_scale), _ptr(idx), _ptr(w))
    return rc, idx, w


def _status():
    v = ctypes.c_int(-1)
    rc = M.lib().moe_router_topk_noalloc_status(ctypes.byref(v))
    assert rc == M.MOE_OK, M.status_string(rc)
    return v.value


def _check_against_oracle(idx, w, ref_idx, ref_w, gap):
    """Expert sets equal to the oracle's for every row whose k-th vs (k+1)-th
    biased-score gap is at least 1e-5, and each weight within 1e-6 of the
    oracle's weight for the same expert."""
    idx = idx.cpu().numpy()
    w = w.cpu().numpy().astype(np.float64)
    checked = 0
    for b in range(idx.shape[0]):
        if gap[b] < 1e-5:
            continue
        assert sorted(idx[b].tolist()) == sorted(ref_idx[b].tolist()), b
        order = {int(e): j for j, e in enumerate(ref_idx[b])}
        for j in range(idx.shape[1]):
            assert abs(w[b, j] - ref_w[b, order[int(idx[b, j])]]) <= 1e-6
        checked += 1
    return checked


def _check_same_routing(layer_idx, layer_w, idx, w):
    assert torch.equal(idx.cpu(), layer_idx.cpu())
    np.testing.assert_allclose(w.cpu().numpy(), layer_w.cpu().numpy(), rtol=0, atol=1e-6)


@pytest.mark.parametrize("B", [1, 5, 64])
def test_noalloc_router_matches_layer_router_tiny(B):
    cfg = CONFIGS["tiny_b1"]
    weights = synthetic.make_weights(cfg)
    layer = synthetic.make_layer(cfg, max_batch=64, weights=weights)
    x, _ = synthetic.make_activations(cfg, B=B)
    ref_idx, ref_w = layer.router_topk(x)
    for _ in range(2):   # two calls in a row share the scratch array
        rc, idx, w = _noalloc(weights["router_w"], weights["router_bias"], x, cfg.top_k,
                              cfg.routed_scale)
        torch.cuda.synchronize()
        assert rc == M.MOE_OK, M.status_string(rc)
        _check_same_routing(ref_idx, ref_w, idx, w)
    assert _status() == 0
    layer.close()


def test_noalloc_router_full_size_matches_oracle():
    """Full-size router (896 experts, d = 7168, top-16) at B = 8 straight
    against the oracle's fp64 routing, on the oracle's tie-free draw."""
    cfg = CONFIGS["full_b8"]
    inp = oracle.clean_inputs(cfg)
    ref_logits, ref_idx, ref_w, gap = oracle.route(inp)
    dev = torch.device("cuda")
    rw = torch.from_numpy(inp.wr.astype(np.float32)).to(dev).to(torch.bfloat16)
    bias = torch.from_numpy(np.asarray(inp.bias, np.float32)).to(dev)
    x, _ = synthetic.make_activations(cfg, attempt=inp.attempt)
    assert np.array_equal(x.float().cpu().numpy().astype(np.float64), inp.x)
    for _ in range(2):
        rc, idx, w = _noalloc(rw, bias, x, cfg.top_k, cfg.routed_scale)
        torch.cuda.synchronize()
        assert rc == M.MOE_OK, M.status_string(rc)
        assert _check_against_oracle(idx, w, ref_idx, ref_w, gap) == cfg.B
    assert _status() == 0


def test_noalloc_router_largest_hidden_size_matches_oracle():
    """d = 7680, the largest hidden size the entry point accepts, 64 experts,
    top-4, B = 5, against the oracle's fp64 routing."""
    d, E, k, B = 7680, 64, 4, 5
    dev = torch.device("cuda")
    rw = torch.empty((E, d), dtype=torch.float32, device=dev)
    gen.normal_device(21, T_ROUTER_W, 0, rw, 0.0, float(np.float32(1 / np.sqrt(d))))
    rw = rw.to(torch.bfloat16)
    bias = torch.empty(E, dtype=torch.float32, device=dev)
    gen.normal_device(21, T_ROUTER_BIAS, 0, bias, 0.0, 0.01)
    x = torch.empty((B, d), dtype=torch.float32, device=dev)
    gen.normal_device(21, T_X, 0, x, 0.0, 1.0)
    x = x.to(torch.bfloat16)
    _, ref_idx, ref_w, gap = oracle.router(x.float().cpu().numpy(), rw.float().cpu().numpy(),
                                           bias.cpu().numpy(), k, 2.5)
    rc, idx, w = _noalloc(rw, bias, x, k, 2.5)
    torch.cuda.synchronize()
    assert rc == M.MOE_OK, M.status_string(rc)
    assert _check_against_oracle(idx, w, ref_idx, ref_w, gap) >= B - 1
    assert _status() == 0


def test_noalloc_router_full_size_router_weights():
    """Full-size router (896 experts, d = 7168, top-16) at B = 8, against the
    layer entry point on the same router weights."""
    c = CONFIGS["full_b8"]
    small = dict(d=c.d, f=256, n_experts=c.n_experts, top_k=c.top_k, f_shared=256, max_batch=8)
    dev = torch.device("cuda")
    rw = torch.empty((c.n_experts, c.d), dtype=torch.float32, device=dev)
    gen.normal_device(2, T_ROUTER_W, 0, rw, 0.0, c.std_router())
    bias = torch.empty(c.n_experts, dtype=torch.float32, device=dev)
    gen.normal_device(2, T_ROUTER_BIAS, 0, bias, 0.0, 0.01)
    rw = rw.to(torch.bfloat16)
    E, d, f = c.n_experts, c.d, 256
    weights = {
        "router_w": rw, "router_bias": bias,
        "w_gu_q": torch.zeros((E, 2 * f, d // 2), dtype=torch.uint8, device=dev),
        "w_gu_s": torch.zeros((E, 2 * f, d // 32), dtype=torch.uint8, device=dev),
        "w_d_q": torch.zeros((E, d, f // 2), dtype=torch.uint8, device=dev),
        "w_d_s": torch.zeros((E, d, f // 32), dtype=torch.uint8, device=dev),
        "shared_gu": torch.zeros((2 * f, d), dtype=torch.bfloat16, device=dev),
        "shared_d": torch.zeros((d, f), dtype=torch.bfloat16, device=dev),
        "rms_gamma": torch.ones(d, dtype=torch.bfloat16, device=dev),
    }
    layer = M.MoELayer(weights=weights, **small)
    x, _ = synthetic.make_activations(c)
    ref_idx, ref_w = layer.router_topk(x)
    for _ in range(2):
        rc, idx, w = _noalloc(rw, bias, x, c.top_k, c.routed_scale)
        torch.cuda.synchronize()
        assert rc == M.MOE_OK, M.status_string(rc)
        _check_same_routing(ref_idx, ref_w, idx, w)
    layer.close()


def test_noalloc_router_rejects_sizes_beyond_its_scratch():
    cfg = CONFIGS["tiny_b1"]
    weights = synthetic.make_weights(cfg)
    x = torch.zeros((65, cfg.d), dtype=torch.bfloat16, device="cuda")
    rc, _, _ = _noalloc(weights["router_w"], weights["router_bias"], x, cfg.top_k, 2.5)
    assert rc == M.MOE_ERR_UNSUPPORTED
    rc, _, _ = _noalloc(weights["router_w"], weights["router_bias"], x[:2], 33, 2.5)
    assert rc == M.MOE_ERR_UNSUPPORTED
    # hidden size past the largest accepted (7680)
    big = torch.zeros((64, 7936), dtype=torch.bfloat16, device="cuda")
    rc, _, _ = _noalloc(big, weights["router_bias"], big[:1], cfg.top_k, 2.5)
    assert rc == M.MOE_ERR_UNSUPPORTED
