"""GPU parity at the boundary dimensions moe_layer_create accepts: the largest
hidden size (d = 7680, with a small f and with the full-size f), the largest
expert intermediate size (f = 3072) with the largest shared one (f_shared =
4096), and the most experts with the most picks (E = 1024, k = 32), each with
the other dimensions small, at one row and a ragged batch of five, on every
expert path.  Rows are compared with the oracle element by element.  Where
the mma.sync kernels' stage rings do not fit the dims, that path must refuse
the layer (UNSUPPORTED) and the automatic one must run on the tensor cores.
Beyond the sizes themselves these reach code the full-size layer does not:
the routed down projection with up to 12 K blocks per warp, the tail's
second batch of 16 pair rows, a 32-pick selection."""
import dataclasses

import numpy as np
import pytest
import torch

import moe_decode_step_gb300 as M
import oracle
from gen.configs import LayerConfig
from moe_decode_step_gb300 import synthetic

from test_gpu_layer import check_against_oracle, run_debug

pytestmark = pytest.mark.gpu

LIMITS = {
    "d7680": LayerConfig("d7680", 1, 7680, 256, 64, 4, 256, (5,)),
    "f3072_fs4096": LayerConfig("f3072_fs4096", 1, 1024, 3072, 64, 4, 4096, (6,)),
    "f3072": LayerConfig("f3072", 1, 1024, 3072, 64, 4, 1536, (8,)),
    "d7680_f1536": LayerConfig("d7680_f1536", 1, 7680, 1536, 64, 4, 1536, (9,)),
    "e1024_k32": LayerConfig("e1024_k32", 1, 1024, 256, 1024, 32, 256, (7,)),
}


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("B", [1, 5])
@pytest.mark.parametrize("path", [0, 1, 2], ids=["auto", "mma_sync", "tcgen05"])
@pytest.mark.parametrize("name", sorted(LIMITS))
def test_boundary_dims_match_oracle(name, path, B):
    cfg = dataclasses.replace(LIMITS[name], B=B)
    inp = oracle.clean_inputs(cfg)
    ref = oracle.forward(inp)
    x, res = synthetic.make_activations(cfg, attempt=inp.attempt)
    try:
        layer = synthetic.make_layer(cfg, expert_path=path, max_batch=B)
    except M.MoEError as e:
        # only the mma.sync path may refuse a shape, and only as unsupported
        assert path == 1 and e.code == M.MOE_ERR_UNSUPPORTED, (name, path, e)
        print(f"{name}: the mma.sync path refuses these dims")
        return
    idx, w = layer.router_topk(x)
    dbg = run_debug(layer, x, res)
    assert layer.status() == 0
    layer.close()
    check_against_oracle(ref, idx.cpu().numpy(), w.cpu().numpy().astype(np.float64), dbg,
                         _np(res), range(B))
