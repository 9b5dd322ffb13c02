"""Pins for the oracle's layer composition on the tiny seeded layer."""
import numpy as np
import pytest

import oracle
from gen.configs import CONFIGS


@pytest.fixture(scope="module")
def tiny():
    inp = oracle.clean_inputs(CONFIGS["tiny_b1"])
    return inp, oracle.forward(inp)


def test_layer_equals_numpy_composition(tiny):
    """Recompute the whole layer with numpy matmuls on the oracle-dequantised
    weights; every intermediate must agree to fp64 rounding."""
    inp, r = tiny
    c = inp.cfg
    x = inp.x[0]
    logits = inp.wr @ x
    s = 1 / (1 + np.exp(-logits))
    key = (s + inp.bias.astype(np.float64)).astype(np.float32)
    order = sorted(range(c.n_experts), key=lambda e: (-key[e], e))[:c.top_k]
    assert list(r["idx"][0]) == order
    w = c.routed_scale * s[order] / s[order].sum()
    np.testing.assert_allclose(r["w"][0], w, rtol=1e-14)
    y_r = np.zeros(c.d)
    for j, e in enumerate(order):
        q_gu, s_gu, q_d, s_d = inp.expert_packed(e)
        Wgu = oracle.mxfp4_dequant(q_gu, s_gu)
        Wd = oracle.mxfp4_dequant(q_d, s_d)
        g, u = Wgu[:c.f] @ x, Wgu[c.f:] @ x
        h = g / (1 + np.exp(-g)) * u
        np.testing.assert_allclose(r["h"][0, j], h, rtol=1e-11, atol=1e-13)
        y_r += w[j] * (Wd @ h)
    np.testing.assert_allclose(r["y_r"][0], y_r, rtol=1e-10, atol=1e-12)
    gs = inp.shared_gu[:c.f_shared] @ x
    us = inp.shared_gu[c.f_shared:] @ x
    y_s = inp.shared_d @ (gs / (1 + np.exp(-gs)) * us)
    np.testing.assert_allclose(r["y_s"][0], y_s, rtol=1e-10, atol=1e-12)
    z = inp.residual[0] + y_r + y_s
    out = z / np.sqrt((z**2).mean() + c.rms_eps) * inp.gamma
    np.testing.assert_allclose(r["z"][0], z, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r["out"][0], out, rtol=1e-10, atol=1e-12)


def test_zero_down_weights_reduce_to_rmsnorm_of_residual_plus_shared(tiny):
    inp, r = tiny
    c = inp.cfg
    zero = np.zeros((c.B, c.top_k, c.d))
    y_r = oracle.combine(zero, r["w"])
    assert np.all(y_r == 0)
    z, out = oracle.tail(inp.residual, y_r, r["y_s"], inp.gamma, c.rms_eps)
    zz = inp.residual + r["y_s"]
    np.testing.assert_allclose(out, zz / np.sqrt((zz**2).mean(axis=1, keepdims=True) + c.rms_eps)
                               * inp.gamma, rtol=1e-12)


def test_outputs_are_bf16_rounded_versions(tiny):
    _, r = tiny
    assert np.array_equal(r["out_bf16"], oracle.round_bf16(r["out"]))
    err = np.abs(r["out_bf16"] - r["out"])
    # half a bf16 ulp: 2^(floor(log2|v|) - 8)
    ulp_half = np.exp2(np.floor(np.log2(np.abs(r["out"]))) - 8)
    assert np.all(err <= ulp_half)


def test_routing_is_clean(tiny):
    _, r = tiny
    assert np.all(r["gap"] >= 1e-5)
    assert r["w"].sum() == pytest.approx(2.5)
