"""Pins for the oracle's router: biased top-k selection and combine weights."""
import itertools
import math
import os

import numpy as np
import pytest

import gen
import oracle
from gen.configs import CONFIGS, T_ROUTER_W, T_ROUTER_BIAS, T_X


def _bf(a):
    return oracle.round_bf16(a)


def test_sigmoid_closed_forms():
    assert oracle.sigmoid(0.0) == 0.5
    for v in (0.3, 1.7, 5.0, 20.0):
        assert oracle.sigmoid(-v) == pytest.approx(1 - oracle.sigmoid(v), abs=1e-15)
        assert oracle.sigmoid(v) == pytest.approx(1 / (1 + math.exp(-v)), rel=1e-15)


def test_logits_one_hot_rows_pick_router_columns():
    rng = np.random.default_rng(0)
    E, d = 10, 64
    wr = _bf(rng.standard_normal((E, d)))
    x = np.zeros((3, d))
    x[0, 5] = 1.0
    x[1, 63] = 1.0
    x[2, 0] = -2.0
    logits, _, _, _ = oracle.router(x, wr, np.zeros(E, np.float32), 2, 2.5)
    assert np.array_equal(logits[0], wr[:, 5])
    assert np.array_equal(logits[1], wr[:, 63])
    assert np.array_equal(logits[2], -2.0 * wr[:, 0])


def test_logits_match_numpy_matmul():
    rng = np.random.default_rng(1)
    x = _bf(rng.standard_normal((4, 96)))
    wr = _bf(rng.standard_normal((12, 96)) / 10)
    logits, _, _, _ = oracle.router(x, wr, np.zeros(12, np.float32), 3, 1.0)
    np.testing.assert_allclose(logits, x @ wr.T, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("E,k", [(5, 1), (6, 2), (8, 3), (10, 4), (12, 4)])
def test_topk_matches_brute_force_subsets(E, k):
    rng = np.random.default_rng(E * 10 + k)
    for trial in range(20):
        d = 32
        x = _bf(rng.standard_normal((1, d)))
        wr = _bf(rng.standard_normal((E, d)) / math.sqrt(d))
        bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
        logits, idx, w, gap = oracle.router(x, wr, bias, k, 2.5)
        s = 1 / (1 + np.exp(-(x @ wr.T)[0]))
        biased = s + bias.astype(np.float64)
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(biased[list(c)]))
        assert set(idx[0]) == set(best)
        # listed in descending biased score
        assert all(biased[idx[0, j]] >= biased[idx[0, j + 1]] for j in range(k - 1))
        # weights: routed_scale * s / sum(s) over the selected, bias excluded
        sel = s[idx[0]]
        np.testing.assert_allclose(w[0], 2.5 * sel / sel.sum(), rtol=1e-14)
        assert w[0].sum() == pytest.approx(2.5, abs=1e-12) and np.all(w[0] > 0)


def test_ties_go_to_the_lower_index():
    E, d = 8, 32
    x = np.zeros((1, d))
    wr = np.zeros((E, d))          # every logit 0, every score 0.5
    bias = np.zeros(E, np.float32)
    bias[[2, 5, 6]] = 0.25         # three equal biased scores above the rest
    _, idx, w, gap = oracle.router(x, wr, bias, 2, 2.5)
    assert list(idx[0]) == [2, 5]
    assert gap[0] == 0.0
    assert np.allclose(w, 2.5 / 2)
    _, idx, w3, _ = oracle.router(x, wr, np.zeros(E, np.float32), 3, 2.5)
    assert list(idx[0]) == [0, 1, 2]
    assert np.allclose(w3, 2.5 / 3)


def test_bias_selects_but_does_not_weight():
    E, d = 6, 32
    x = np.zeros((1, d))
    x[0, 0] = 1.0
    wr = np.zeros((E, d))
    wr[:, 0] = [2.0, 1.0, 0.0, -1.0, -2.0, -3.0]
    bias = np.array([0, 0, 0, 0, 0, 10.0], np.float32)
    _, idx, w, _ = oracle.router(x, wr, bias, 2, 1.0)
    assert list(idx[0]) == [5, 0]
    s5, s0 = 1 / (1 + math.exp(3.0)), 1 / (1 + math.exp(-2.0))
    np.testing.assert_allclose(w[0], [s5 / (s5 + s0), s0 / (s5 + s0)], rtol=1e-14)


def test_routed_scale_is_linear():
    rng = np.random.default_rng(9)
    x = _bf(rng.standard_normal((3, 64)))
    wr = _bf(rng.standard_normal((16, 64)) / 8)
    bias = (rng.standard_normal(16) * 0.01).astype(np.float32)
    _, i1, w1, _ = oracle.router(x, wr, bias, 4, 1.0)
    _, i2, w2, _ = oracle.router(x, wr, bias, 4, 2.5)
    assert np.array_equal(i1, i2)
    np.testing.assert_allclose(w2, 2.5 * w1, rtol=1e-15)


def _expected_distinct(E, k, B):
    return E * (1 - ((E - k) / E) ** B)


def test_expected_union_formula_matches_page_figure():
    figs = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.txt")):
        if line.strip() and not line.startswith("#"):
            a, b = line.split()
            figs[a] = float(b)
    assert _expected_distinct(896, 16, 8) == pytest.approx(figs["expected_distinct_b8"], abs=0.05)


@pytest.mark.parametrize("B,tol", [(8, 4.0), (64, 15.0)])
def test_distinct_experts_statistics_full_router(B, tol):
    """Seeded full-size router: rows route nearly independently, so the mean
    number of distinct experts is close to E (1 - (1 - k/E)^B)."""
    c = CONFIGS["full_b1"]
    wr = _bf(gen.normal_host(1, T_ROUTER_W, 0, c.n_experts * c.d, 0.0,
                             c.std_router())).reshape(c.n_experts, c.d)
    bias = gen.normal_host(1, T_ROUTER_BIAS, 0, c.n_experts, 0.0, 0.01)
    counts = []
    for seed in range(100, 106):
        x = _bf(gen.normal_host(seed, T_X, 0, B * c.d, 0.0, 1.0)).reshape(B, c.d)
        _, idx, _, _ = oracle.router(x, wr, bias, c.top_k, 2.5)
        counts.append(len(set(idx.ravel().tolist())))
    want = _expected_distinct(896, 16, B)
    assert abs(np.mean(counts) - want) < tol, (counts, want)
