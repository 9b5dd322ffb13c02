"""GPU parity at full size (d=7168, f=1536, 896 experts, top-16) in the launch
configuration the benchmark times.  Sampled rows are checked against the
oracle element by element; every row is checked for the RMSNorm property and
exact routing."""
import numpy as np
import pytest
import torch

import oracle
from gen.configs import CONFIGS
from moe_decode_step_gb300 import synthetic

from _parity import assert_close, bf16_ulp_distance
from test_gpu_layer import check_against_oracle, run_debug

pytestmark = pytest.mark.gpu


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name,rows,path", [("full_b1", [0], 0), ("full_b1", [0], 2),
                                            ("full_b8", [0, 7], 0), ("verify_b16", [0, 5, 15], 0),
                                            ("verify_b16", [3, 12], 1), ("full_b64", [0, 33, 63], 0)])
def test_full_layer_sampled_rows(name, rows, path):
    """path 0, the layer the benchmark times: mma.sync at B = 1, tcgen05 at
    B = 8, 16 and 64; path 2: tcgen05 at B = 1 as well; path 1: mma.sync on
    the verify batch, whose experts take several rows per pass."""
    cfg = CONFIGS[name]
    inp = oracle.clean_inputs(cfg)
    ref = oracle.forward(inp, rows=rows)
    layer = synthetic.make_layer(cfg, expert_path=path)
    x, res = synthetic.make_activations(cfg, attempt=inp.attempt)
    idx, w = layer.router_topk(x)
    dbg = run_debug(layer, x, res)
    assert layer.status() == 0
    idx = idx.cpu().numpy()
    # exact routing for every row, not only the sampled ones
    for b in range(cfg.B):
        assert sorted(idx[b].tolist()) == sorted(ref["idx"][b].tolist()), b
    assert len(set(idx.ravel().tolist())) == len(set(ref["idx"].ravel().tolist()))
    check_against_oracle(ref, idx, w.cpu().numpy().astype(np.float64), dbg, _np(res), rows)
    # every row: RMS of out / gamma is sqrt(ms / (ms + eps)) ~ 1 (fp32 values)
    o = dbg["out_f32"] / inp.gamma[None, :]
    np.testing.assert_allclose(np.sqrt((o ** 2).mean(axis=1)), 1.0, atol=1e-5)
    # dequant of one selected expert is bit-exact against the oracle's packing
    e = int(idx[rows[0], 0])
    q_gu, s_gu, q_d, s_d = inp.expert_packed(e)
    assert np.array_equal(_np(layer.debug_dequant(e, 1)), oracle.mxfp4_dequant(q_d, s_d))
    layer.close()


def test_chain_of_four_layers_teacher_forced():
    cfg = CONFIGS["chain4_b1"]
    layers = [synthetic.make_layer(cfg, layer=l) for l in range(cfg.n_layers)]
    for l in range(cfg.n_layers - 1):
        layers[l].set_prefetch_next(layers[l + 1])
    x, res = synthetic.make_activations(cfg, layer=0)
    x0 = x.clone()
    checked = 0
    for l in range(cfg.n_layers):
        inp = oracle.LayerInputs(cfg, layer=l, x=_np(x), residual=_np(res))
        _, _, _, gap = oracle.route(inp)
        idx, w = layers[l].router_topk(x)
        dbg_t = layers[l].forward_debug(x, res)
        torch.cuda.synchronize()
        dbg = {k: _np(v) for k, v in dbg_t.items()}
        assert layers[l].status() == 0
        if gap.min() >= 1e-5:
            ref = oracle.forward(inp)
            check_against_oracle(ref, idx.cpu().numpy(), w.cpu().numpy().astype(np.float64), dbg,
                                 _np(res), [0])
            checked += 1
        x = dbg_t["out"]
    assert checked >= 3
    for L in layers:
        L.close()
