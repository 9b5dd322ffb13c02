"""Pins of the oracle's MXFP8 activation path (OCP MX v1.0: E4M3 elements, one
E8M0 scale per 32 elements), the FP4 x MXFP8 products of the pages' routed
experts ("Kimi K3 on GB300", "Why batch 1 on a rack is not only a bandwidth
problem"): the E4M3 table against the OFP8 specification and against torch's
float8_e4m3fn codec (an independent implementation), round-to-nearest-even at
midpoints, saturation, brute-force nearest, the block scale rule and its
error bound, and the layer's mxfp8 mode against the exact one."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gen.configs import CONFIGS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _spec():
    out = {}
    for line in open(os.path.join(GOLDEN, "e4m3_spec.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code, value = line.split()
        out[int(code, 16)] = float(value)
    return out


def test_e4m3_values_match_the_specification_table():
    for code, value in _spec().items():
        got = oracle.e4m3_value(code)
        if math.isnan(value):
            assert math.isnan(got), hex(code)
        else:
            assert got == value and math.copysign(1, got) == math.copysign(1, value), hex(code)


def test_e4m3_values_match_torch_float8_e4m3fn_for_every_code():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2   # S.1111.111 only
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_every_finite_code_round_trips():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c, hex(c)


@pytest.mark.parametrize("t, want", [
    (1.0625, 1.0),          # midpoint of 1.0 (mantissa 000) and 1.125 (001): even wins
    (1.1875, 1.25),         # midpoint of 1.125 (001) and 1.25 (010)
    (2.0 ** -10, 0.0),      # midpoint of 0 and the smallest subnormal 2^-9
    (3 * 2.0 ** -11, 2.0 ** -9),
    (464.0, 448.0),         # midpoint of 448 and the (non-finite) next step: saturates
    (500.0, 448.0),
    (1e9, 448.0),
    (-1e9, -448.0),
    (-2.0 ** -12, -0.0),    # a tiny negative value keeps its sign
])
def test_rounding_ties_and_saturation(t, want):
    got = oracle.e4m3_value(oracle.e4m3_encode(t))
    assert got == want and math.copysign(1, got) == math.copysign(1, want)


def test_encode_matches_torch_inside_the_finite_range():
    rng = np.random.default_rng(5)
    t = np.concatenate([rng.normal(0, 1, 4000) * 2.0 ** rng.integers(-12, 9, 4000),
                        rng.uniform(-460, 460, 1000)])
    t = t[np.abs(t) < 464]
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(oracle.e4m3_encode(v)) for v in t])
    assert np.array_equal(got, ref)


def test_encode_is_the_nearest_finite_value_by_brute_force():
    rng = np.random.default_rng(6)
    finite = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    for t in rng.normal(0, 1, 300) * 2.0 ** rng.integers(-10, 9, 300):
        q = oracle.e4m3_value(oracle.e4m3_encode(t))
        assert abs(abs(q) - abs(t)) <= np.min(np.abs(finite - abs(t))) + 0.0


def test_block_scale_rule():
    rng = np.random.default_rng(7)
    for _ in range(200):
        blk = rng.normal(0, 1, 32) * 2.0 ** rng.integers(-20, 20)
        e = oracle.block_exponent_e4m3(blk)
        assert 256 <= np.max(np.abs(blk)) / 2.0 ** e < 512
    assert oracle.block_exponent_e4m3(np.zeros(32)) == -127
    blk = np.zeros(32)
    blk[3] = 2.0 ** 5                       # an exact power of two: amax / scale = 256
    assert oracle.block_exponent_e4m3(blk) == 5 - 8


def test_quantisation_error_bound_and_idempotence():
    """Per element: |v_hat - v| <= 2^-4 |v| where v / scale is normal
    (>= 2^-6), <= 2^-10 scale in the subnormal range, and < 64 scale where
    v / scale saturates (v / scale < 512); rounding a rounded row changes
    nothing."""
    rng = np.random.default_rng(8)
    a = rng.normal(0, 1, (4, 256)) * np.exp(rng.normal(0, 2, (4, 256)))
    q, s = oracle.mxfp8_quant(a)
    v = oracle.mxfp8_dequant(q, s)
    scale = np.repeat(2.0 ** (s.astype(np.int64) - 127), 32, axis=1)
    r = np.abs(a) / scale
    err = np.abs(v - a)
    normal = (r >= 2.0 ** -6) & (r <= 448)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(a[normal]))
    assert np.all(err[r < 2.0 ** -6] <= 2.0 ** -10 * scale[r < 2.0 ** -6])
    assert np.all(err[r > 448] < 64 * scale[r > 448])
    assert np.array_equal(oracle.mxfp8_round(v), v)


def test_layer_mxfp8_mode():
    """The mxfp8 mode changes only the routed experts' activation operands:
    with x already MXFP8-exact its h equals the exact mode's bit for bit, and
    the shared expert is untouched.  Against the exact layer the outputs move
    by what E4M3's 4 significant bits imply: a relative rounding error of at
    most 2^-4 per element, about 2.5% RMS, so a few per cent on average and,
    over a row's 1024 outputs, up to a few times that."""
    cfg = CONFIGS["tiny_b1"]
    inp = oracle.clean_inputs(cfg)
    inp_r = oracle.LayerInputs(cfg, x_attempt=inp.attempt, x=oracle.mxfp8_round(inp.x))
    ex = oracle.forward(inp_r)
    f1 = oracle.forward(inp_r, act="mxfp8")
    assert np.array_equal(f1["h"], ex["h"])
    assert np.array_equal(f1["y_s"], ex["y_s"])
    # h itself is rounded before the down projection
    assert not np.array_equal(f1["y_pair"], ex["y_pair"])
    ex0 = oracle.forward(inp)
    f10 = oracle.forward(inp, act="mxfp8")
    rms = np.sqrt(np.mean(ex0["y_r"] ** 2))
    dev = np.abs(f10["y_r"] - ex0["y_r"])
    assert 1e-3 * rms < np.sqrt(np.mean(dev ** 2)) <= 0.06 * rms
    assert np.max(dev) <= 0.25 * rms
    assert np.abs(f10["out"] - ex0["out"]).sum() / np.abs(ex0["out"]).sum() <= 0.05
