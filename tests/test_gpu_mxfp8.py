"""GPU parity of the MXFP8-activation expert path (moe_set_act_format 1: x and
h rounded to E4M3 with one E8M0 scale per 32 elements before they meet the
MXFP4 weights) against the oracle's mxfp8 mode, element by element, at the
layer's stated tolerance: both sides round the same values the same way
(nearest E4M3, ties to even, saturation at 448), so they differ only by
summation order and by h's fp32 (GPU) against fp64 (oracle) values.  The
one-row mma.sync kernel and the tensor-core path (any B) take the format; the
mma.sync batch kernels refuse it."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import moe_decode_step_gb300 as M
from gen.configs import CONFIGS
from moe_decode_step_gb300 import synthetic

from _parity import assert_close
from test_gpu_layer import check_against_oracle, run_debug

pytestmark = pytest.mark.gpu


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _parity(cfg, rows=None, expert_path=0, max_batch=None):
    inp = oracle.clean_inputs(cfg)
    ref = oracle.forward(inp, rows=rows, act="mxfp8")
    ex = oracle.forward(inp, rows=rows)
    x, res = synthetic.make_activations(cfg, attempt=inp.attempt)
    layer = synthetic.make_layer(cfg, expert_path=expert_path, max_batch=max_batch)
    layer.set_act_format(1)
    idx, w = layer.router_topk(x)
    dbg = run_debug(layer, x, res)
    assert layer.status() == 0
    layer.close()
    check_against_oracle(ref, idx.cpu().numpy(), w.cpu().numpy().astype(np.float64), dbg,
                         _np(res), range(cfg.B) if rows is None else rows)
    # and it is the MXFP8 layer, not the exact one: y_routed sits a few per
    # cent of its RMS from the exact oracle's
    dev = np.abs(dbg["y_routed"][0] - ex["y_r"][0])
    assert np.sqrt(np.mean(dev ** 2)) > 5e-3 * np.sqrt(np.mean(ex["y_r"][0] ** 2))


def test_tiny_one_row_matches_oracle_mxfp8_mode():
    _parity(CONFIGS["tiny_b1"])


def test_full_size_one_row_matches_oracle_mxfp8_mode():
    _parity(CONFIGS["full_b1"])


@pytest.mark.parametrize("B", [1, 3, 8, 17, 64])
def test_tiny_tensor_core_path_matches_oracle_mxfp8_mode(B):
    """The tensor-core path's activation planes hold the MXFP8 roundings of x
    (built by the CUDA-core router below 25 rows, by the tensor-core router
    from 25) and of h (FC1's epilogue)."""
    _parity(dataclasses.replace(CONFIGS["tiny_b1"], name=f"tiny_b{B}", B=B), expert_path=2,
            max_batch=64)


@pytest.mark.parametrize("name,rows", [("full_b8", [0, 7]), ("verify_b16", [0, 5, 15]),
                                       ("full_b64", [0, 33, 63])])
def test_full_size_batches_match_oracle_mxfp8_mode(name, rows):
    """The batches the benchmark times, on their tensor-core path."""
    _parity(CONFIGS[name], rows=rows)


def test_mma_sync_batches_reject_the_format_and_it_switches_back():
    cfg = CONFIGS["tiny_b1"]
    layer = synthetic.make_layer(cfg, max_batch=4, expert_path=1)
    layer.set_act_format(1)
    x3, r3 = synthetic.make_activations(dataclasses.replace(cfg, name="tiny_b3", B=3))
    with pytest.raises(M.MoEError) as e:
        layer.forward(x3, r3.clone())
    assert e.value.code == M.MOE_ERR_UNSUPPORTED
    with pytest.raises(M.MoEError) as e:
        layer.set_act_format(2)
    assert e.value.code == M.MOE_ERR_INVALID_ARG
    # back to exact activations: the exact oracle's parity
    layer.set_act_format(0)
    inp = oracle.clean_inputs(cfg)
    ref = oracle.forward(inp)
    x, res = synthetic.make_activations(cfg, attempt=inp.attempt)
    idx, w = layer.router_topk(x)
    dbg = run_debug(layer, x, res)
    assert layer.status() == 0
    check_against_oracle(ref, idx.cpu().numpy(), w.cpu().numpy().astype(np.float64), dbg,
                         _np(res), [0])
    layer.close()




# ---------------------------------------------------------------------------
# Edge rows in the MXFP8 format: a row with max |x| >= 2^15 (its blocks' E8M0
# scales far above 1; on the one-row mma.sync kernel the f16 shift applies to
# the rounded values) and an all-zero row (every block's scale code is the
# smallest, every element rounds to 0, so h and the routed output are exact
# zeros).
from test_gpu_edge import _cfg, _check_rows, _edge_inputs, _run  # noqa: E402


def test_large_and_zero_rows_tensor_core_path_mxfp8():
    kinds = ["normal", "large", "zero"]
    cfg = _cfg(CONFIGS["tiny_b1"], len(kinds))
    x, res, inp = _edge_inputs(cfg, kinds)
    assert float(x[1].float().abs().max()) >= 2.0 ** 15
    ref = oracle.forward(inp, act="mxfp8")
    w = synthetic.make_weights(CONFIGS["tiny_b1"], layout=3)
    idx, wt, dbg, r = _run(cfg, w, x, res, 2, max_batch=len(kinds), act_format=1)
    _check_rows(ref, idx, wt, dbg, r, range(len(kinds)), zero_rows=(2,))


@pytest.mark.parametrize("kind", ["large", "zero"])
@pytest.mark.parametrize("path", [1, 2], ids=["mma_sync", "tcgen05"])
def test_one_edge_row_mxfp8(path, kind):
    cfg = _cfg(CONFIGS["tiny_b1"], 1)
    x, res, inp = _edge_inputs(cfg, [kind])
    ref = oracle.forward(inp, act="mxfp8")
    w = synthetic.make_weights(CONFIGS["tiny_b1"], layout=1 if path == 1 else 3)
    idx, wt, dbg, r = _run(cfg, w, x, res, path, max_batch=1, act_format=1)
    _check_rows(ref, idx, wt, dbg, r, [0], zero_rows=(0,) if kind == "zero" else ())
