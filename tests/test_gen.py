"""Pins for the seeded input generator (Philox4x32-10 + Box-Muller)."""
import math
import os

import numpy as np
import pytest

import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kat():
    rows = []
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.strip() and not line.startswith("#"):
            v = [int(t, 16) for t in line.split()]
            rows.append((v[0:4], v[4:6], v[6:10]))
    return rows


@pytest.mark.parametrize("ctr,key,want", _kat())
def test_philox_known_answers(ctr, key, want):
    assert gen.philox4x32_10(ctr, key) == want


def test_ln_and_cos_against_libm():
    rng = np.random.default_rng(7)
    rs = [int(r) for r in rng.integers(0, 2**32, 20000)] + [0, 1, 511, 512, 2**31, 2**32 - 1]
    for r in rs:
        u = ((r >> 9) * 2 + 1) / 2**24
        ref = math.log(u)
        assert abs(gen.ln_u(r) - ref) <= 4e-7 * abs(ref) + 1e-7
        t = (r >> 30) / 4 + (((r >> 8) & 0x3FFFFF) * 2 + 1) / 2**23 / 4
        assert abs(gen.cos2pi_u(r) - math.cos(2 * math.pi * t)) <= 3e-7


def test_normal_moments_and_tails():
    n = 2_000_000
    a = gen.normal_host(5, 8, 1, n, 0.0, 1.0).astype(np.float64)
    se = 1 / math.sqrt(n)
    assert abs(a.mean()) < 5 * se
    assert abs(a.var() - 1) < 5 * math.sqrt(2) * se
    assert abs((a**3).mean()) < 5 * math.sqrt(15) * se
    assert abs((a**4).mean() - 3) < 5 * math.sqrt(96) * se
    # tail mass beyond 3 sigma: 0.0026998
    p3 = (np.abs(a) > 3).mean()
    assert abs(p3 - 0.0026998) < 5 * math.sqrt(0.0027 / n)
    assert np.abs(a).max() < 5.8   # radius bound sqrt(-2 ln 2^-24)


def test_mean_std_applied():
    a = gen.normal_host(3, 3, 0, 200_000, 1.0, 0.1).astype(np.float64)
    assert abs(a.mean() - 1.0) < 5 * 0.1 / math.sqrt(a.size)
    assert abs(a.std() - 0.1) < 0.002


def test_element_addressing_and_thread_invariance():
    full = gen.normal_host(11, 9, 4, 300_000, 0.0, 0.5, nthreads=1)
    part = gen.normal_host(11, 9, 4, 1000, 0.0, 0.5, start=123_456, nthreads=3)
    assert np.array_equal(full[123_456:124_456], part)
    many = gen.normal_host(11, 9, 4, 300_000, 0.0, 0.5, nthreads=8)
    assert np.array_equal(full, many)


def test_streams_differ():
    a = gen.normal_host(1, 8, 0, 1000, 0.0, 1.0)
    b = gen.normal_host(1, 8, 1, 1000, 0.0, 1.0)
    c = gen.normal_host(2, 8, 0, 1000, 0.0, 1.0)
    d = gen.normal_host(1, 9, 0, 1000, 0.0, 1.0)
    for o in (b, c, d):
        assert not np.array_equal(a, o)
        assert abs(np.corrcoef(a, o)[0, 1]) < 0.15


def test_uncorrelated_activation_rows_are_the_plain_stream():
    from gen.configs import CONFIGS, T_X
    cfg = CONFIGS["full_b8"]
    x = gen.activation_x(cfg, 2)
    n = gen.normal_host(2, T_X, 0, cfg.B * cfg.d, 0.0, 1.0).reshape(cfg.B, cfg.d)
    assert x.dtype == np.float32 and np.array_equal(x, n)


def test_verify_batch_rows_correlate_within_groups_only():
    """The correlated 16-row batch's recipe: rows of one group of 4 correlate
    by rho^2, rows of different groups not at all, and every row keeps unit
    variance."""
    from gen.configs import CONFIGS
    cfg = CONFIGS["verify_b16"]
    x = gen.activation_x(cfg, cfg.seeds[0]).astype(np.float64)
    assert x.shape == (16, cfg.d)
    c = np.corrcoef(x)
    g = np.arange(16) // (1 + cfg.drafts)
    same = (g[:, None] == g[None, :]) & ~np.eye(16, dtype=bool)
    diff = g[:, None] != g[None, :]
    assert abs(c[same].mean() - cfg.corr ** 2) < 0.01
    assert np.abs(c[diff]).max() < 0.06
    np.testing.assert_allclose(x.std(axis=1), 1.0, atol=0.03)


def test_verify_batch_rows_route_to_shared_experts():
    """What the correlation is for: the rows of a group pick mostly the same
    experts (exact routing by the oracle), so the batch touches far fewer
    distinct experts than 16 independent rows (about 225 of 896)."""
    import oracle
    from gen.configs import CONFIGS
    cfg = CONFIGS["verify_b16"]
    inp = oracle.LayerInputs(cfg)
    _, idx, _, _ = oracle.route(inp)
    sets = [set(r.tolist()) for r in idx]
    gsize = 1 + cfg.drafts
    within = [len(sets[a] & sets[b]) for a in range(16) for b in range(16)
              if a != b and a // gsize == b // gsize]
    across = [len(sets[a] & sets[b]) for a in range(16) for b in range(16)
              if a // gsize != b // gsize]
    assert np.mean(within) >= 8 and np.mean(across) <= 2
    assert len(set().union(*sets)) <= 140
