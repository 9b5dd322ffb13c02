"""Pins for the oracle's SwiGLU experts (MXFP4 and dense) and the tail."""
import math

import numpy as np
import pytest
import torch

import oracle


def _bf(a):
    return oracle.round_bf16(a)


def test_swiglu_closed_forms():
    assert oracle.swiglu(0.0, 3.0) == 0.0
    assert oracle.swiglu(2.0, 0.0) == 0.0
    assert oracle.swiglu(1.0, 1.0) == pytest.approx(1 / (1 + math.exp(-1)), rel=1e-15)
    assert oracle.swiglu(40.0, 0.5) == pytest.approx(20.0, rel=1e-15)
    assert oracle.swiglu(-40.0, 1.0) == pytest.approx(-40 * math.exp(-40), rel=1e-6)


def _expert(rng, d, f):
    gu = (rng.standard_normal((2 * f, d)) / math.sqrt(d)).astype(np.float32)
    dn = (rng.standard_normal((d, f)) / math.sqrt(f)).astype(np.float32)
    return oracle.mxfp4_pack(gu) + oracle.mxfp4_pack(dn)


def test_fc1_one_hot_input_returns_weight_columns():
    rng = np.random.default_rng(0)
    d, f = 128, 64
    q_gu, s_gu, _, _ = _expert(rng, d, f)
    W = oracle.mxfp4_dequant(q_gu, s_gu)
    for j in (0, 31, 32, 127):
        x = np.zeros((1, d))
        x[0, j] = 1.0
        h = oracle.mxfp4_fc1(q_gu, s_gu, x)
        g, u = W[:f, j], W[f:, j]
        np.testing.assert_array_equal(h[0], g / (1 + np.exp(-g)) * u)


def test_fc1_fc2_match_numpy_matmul_on_dequantised_weights():
    rng = np.random.default_rng(1)
    d, f = 256, 96
    q_gu, s_gu, q_d, s_d = _expert(rng, d, f)
    x = _bf(rng.standard_normal((3, d)))
    Wgu = oracle.mxfp4_dequant(q_gu, s_gu)
    Wd = oracle.mxfp4_dequant(q_d, s_d)
    g = x @ Wgu[:f].T
    u = x @ Wgu[f:].T
    h_ref = g / (1 + np.exp(-g)) * u
    h = oracle.mxfp4_fc1(q_gu, s_gu, x)
    np.testing.assert_allclose(h, h_ref, rtol=1e-12, atol=1e-13)
    y = oracle.mxfp4_fc2(q_d, s_d, h)
    np.testing.assert_allclose(y, h @ Wd.T, rtol=1e-12, atol=1e-13)


def test_gate_and_up_rows_are_not_swapped():
    rng = np.random.default_rng(2)
    d, f = 64, 32
    q_gu, s_gu, _, _ = _expert(rng, d, f)
    W = oracle.mxfp4_dequant(q_gu, s_gu)
    x = _bf(rng.standard_normal((1, d)))
    h = oracle.mxfp4_fc1(q_gu, s_gu, x)[0]
    g, u = W[:f] @ x[0], W[f:] @ x[0]
    swapped = u / (1 + np.exp(-u)) * g
    np.testing.assert_allclose(h, g / (1 + np.exp(-g)) * u, rtol=1e-12)
    assert not np.allclose(h, swapped, rtol=1e-3)


def test_dense_matches_numpy():
    rng = np.random.default_rng(3)
    d, f = 96, 40
    wgu = _bf(rng.standard_normal((2 * f, d)) / 10)
    wd = _bf(rng.standard_normal((d, f)) / 6)
    x = _bf(rng.standard_normal((2, d)))
    g, u = x @ wgu[:f].T, x @ wgu[f:].T
    h_ref = g / (1 + np.exp(-g)) * u
    h = oracle.dense_fc1(wgu, x)
    np.testing.assert_allclose(h, h_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(oracle.dense_fc2(wd, h), h @ wd.T, rtol=1e-12, atol=1e-14)


def test_combine_is_the_weighted_sum():
    rng = np.random.default_rng(4)
    yp = rng.standard_normal((2, 3, 5))
    w = rng.uniform(0.1, 1.0, (2, 3))
    np.testing.assert_allclose(oracle.combine(yp, w), np.einsum("bk,bkd->bd", w, yp), rtol=1e-14)


def test_rmsnorm_unit_rms_before_gamma():
    rng = np.random.default_rng(5)
    B, d, eps = 3, 512, 1e-6
    res = rng.standard_normal((B, d)) * 1.7
    yr = rng.standard_normal((B, d)) * 0.3
    ys = rng.standard_normal((B, d)) * 0.5
    z, out = oracle.tail(res, yr, ys, np.ones(d), eps)
    np.testing.assert_allclose(z, res + yr + ys, rtol=1e-15)
    ms = (z**2).mean(axis=1)
    rms_out = np.sqrt((out**2).mean(axis=1))
    np.testing.assert_allclose(rms_out, np.sqrt(ms / (ms + eps)), rtol=1e-12)
    # gamma scales elementwise
    gamma = rng.uniform(0.5, 1.5, d)
    _, out_g = oracle.tail(res, yr, ys, gamma, eps)
    np.testing.assert_allclose(out_g, out * gamma, rtol=1e-14)
    # eps matters only against tiny z
    z0, out0 = oracle.tail(np.zeros((1, d)), np.zeros((1, d)), np.zeros((1, d)), np.ones(d), eps)
    assert np.all(out0 == 0)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(6)
    v = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.uniform(-30, 30, 100000),
                        [1.0 + 2**-8, 1.0 + 3 * 2**-8, -(1.0 + 2**-8), 255.5, 256.5, 1e-40]])
    v = v.astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(v.astype(np.float64)), ref)
    # ties to even
    assert oracle.round_bf16(np.array([1.0 + 2**-8]))[0] == 1.0
    assert oracle.round_bf16(np.array([1.0 + 3 * 2**-8]))[0] == 1.0 + 2**-6
