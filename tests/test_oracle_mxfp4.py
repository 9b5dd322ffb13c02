"""Pins for the oracle's MXFP4 encode/decode/pack (OCP MX v1.0 definitions)."""
import math
import os

import numpy as np
import pytest

import oracle
from gen.configs import CONFIGS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _spec_table():
    t = {}
    for line in open(os.path.join(GOLDEN, "e2m1_e8m0_spec.txt")):
        if line.strip() and not line.startswith("#"):
            c, v = line.split()
            t[int(c)] = float(v)
    return t


def test_e2m1_values_match_spec_table():
    table = _spec_table()
    assert len(table) == 16
    for code, v in table.items():
        got = oracle.e2m1_value(code)
        assert got == v and math.copysign(1, got) == math.copysign(1, v)


def test_e8m0_values():
    for b in range(255):
        assert oracle.e8m0_value(b) == math.ldexp(1.0, b - 127)
    assert math.isnan(oracle.e8m0_value(255))


def test_encode_round_trips_every_code():
    for code in range(16):
        v = oracle.e2m1_value(code)
        assert oracle.e2m1_encode(v) == code


@pytest.mark.parametrize("t,code", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
    (-0.25, 8), (-0.75, 10), (-1.25, 10), (-1.75, 12), (-2.5, 12), (-3.5, 14), (-5.0, 14),
    (6.9, 7), (7.9, 7), (100.0, 7), (-7.5, 15), (-0.1, 8), (0.1, 0), (-0.0, 8),
    (0.2500001, 1), (0.7499999, 1), (2.4999, 4), (2.5001, 5), (4.9999, 6), (5.0001, 7),
])
def test_encode_ties_to_even_and_saturation(t, code):
    assert oracle.e2m1_encode(t) == code


def test_encode_is_nearest_by_brute_force():
    rng = np.random.default_rng(1)
    table = _spec_table()
    for t in rng.uniform(-7.5, 7.5, 3000):
        dists = {c: abs(t - v) for c, v in table.items()}
        best = min(dists.values())
        code = oracle.e2m1_encode(t)
        assert dists[code] == best
        # the chosen code carries the sign of t
        assert (code >= 8) == (t < 0)


def test_block_exponent_definition():
    rng = np.random.default_rng(2)
    for _ in range(500):
        blk = (rng.standard_normal(32) * 10.0 ** rng.uniform(-6, 6)).astype(np.float32)
        amax = float(np.max(np.abs(blk)))
        e = oracle.block_exponent(blk)
        # amax / 2^e must lie in [4, 8)
        r = amax / 2.0**e
        assert 4.0 <= r < 8.0
    # exact powers of two: amax = 2^p gives e = p - 2
    for p in range(-100, 100, 7):
        blk = np.zeros(32, np.float32)
        blk[5] = -(2.0**p)
        assert oracle.block_exponent(blk) == p - 2
    assert oracle.block_exponent(np.zeros(32, np.float32)) == -127


def test_pack_dequant_error_bound_and_layout():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((6, 128)).astype(np.float32)
    q, s = oracle.mxfp4_pack(w)
    assert q.shape == (6, 64) and s.shape == (6, 4)
    wh = oracle.mxfp4_dequant(q, s)
    for r in range(6):
        for b in range(4):
            e = int(s[r, b]) - 127
            for i in range(32):
                t = float(w[r, b * 32 + i]) / 2.0**e
                a = abs(t)
                step = 0.5 if a <= 2 else (1.0 if a <= 4 else 2.0)
                bound = (step / 2 if a <= 6 else a - 6) * 2.0**e
                assert abs(w[r, b * 32 + i] - wh[r, b * 32 + i]) <= bound + 1e-30
    # nibble order: low nibble = even k
    for r in range(6):
        for j in range(0, 128, 2):
            byte = int(q[r, j // 2])
            e = int(s[r, j // 32]) - 127
            assert wh[r, j] == oracle.e2m1_value(byte & 15) * 2.0**e
            assert wh[r, j + 1] == oracle.e2m1_value(byte >> 4) * 2.0**e


def test_dequant_matches_numpy_table_lookup():
    rng = np.random.default_rng(4)
    q = rng.integers(0, 256, (5, 48), dtype=np.uint8)
    s = rng.integers(100, 150, (5, 3), dtype=np.uint8)
    table = np.array([v for _, v in sorted(_spec_table().items())])
    codes = np.stack([q & 15, q >> 4], axis=-1).reshape(5, 96)
    ref = table[codes] * np.exp2(np.repeat(s.astype(np.float64) - 127, 32, axis=1))
    assert np.array_equal(oracle.mxfp4_dequant(q, s), ref)


def test_exactly_representable_blocks_round_trip():
    rng = np.random.default_rng(5)
    table = _spec_table()
    vals = np.array([table[c] for c in range(16)])
    for _ in range(50):
        e = int(rng.integers(-20, 20))
        codes = rng.integers(0, 16, 32)
        codes[0] = 7      # amax = 6 * 2^e, so the block exponent is e
        w = (vals[codes] * 2.0**e).astype(np.float32)[None, :]
        q, s = oracle.mxfp4_pack(w)
        assert int(s[0, 0]) - 127 == e
        assert np.array_equal(oracle.mxfp4_dequant(q, s)[0], w[0].astype(np.float64))


def _page_figures():
    d = {}
    for line in open(os.path.join(GOLDEN, "page_figures.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            d[k] = float(v)
    return d


def test_expert_byte_count_closed_form():
    fig = _page_figures()
    c = CONFIGS["full_b1"]
    assert c.expert_bytes() == int(fig["expert_bytes_mxfp4"])
    # packed array sizes of one expert equal the closed form
    gu_q, gu_s = (2 * c.f * c.d // 2, 2 * c.f * c.d // 32)
    d_q, d_s = (c.d * c.f // 2, c.d * c.f // 32)
    assert gu_q + gu_s + d_q + d_s == int(fig["expert_bytes_mxfp4"])
    assert fig["experts_per_token"] * fig["expert_bytes_mxfp4"] / 1e9 == pytest.approx(
        fig["expert_bytes_per_token_gb"], abs=0.005)
    assert CONFIGS["tiny_b1"].expert_bytes() == 417792
    assert c.n_experts == fig["n_experts"] and c.top_k == fig["top_k"]


def test_pack_output_sizes_tiny_expert():
    c = CONFIGS["tiny_b1"]
    w = np.ones((2 * c.f, c.d), np.float32)
    q, s = oracle.mxfp4_pack(w)
    w2 = np.ones((c.d, c.f), np.float32)
    q2, s2 = oracle.mxfp4_pack(w2)
    assert q.nbytes + s.nbytes + q2.nbytes + s2.nbytes == c.expert_bytes()
