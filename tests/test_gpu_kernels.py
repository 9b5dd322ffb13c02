"""GPU: seeded generator identity, MXFP4 packer and decode bit-exactness."""
import numpy as np
import pytest
import torch

import gen
import oracle
import moe_decode_step_gb300 as M
from gen.configs import CONFIGS, T_EXPERT_GU, T_X, T_ROUTER_W
from moe_decode_step_gb300 import synthetic

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed,tensor,sub,n,mean,std,start", [
    (0, T_X, 0, 100_003, 0.0, 1.0, 0),
    (1, T_EXPERT_GU, 895, 70_000, 0.0, float(np.float32(1 / np.sqrt(7168))), 11_000_000),
    (13, T_ROUTER_W, 0, 4096, 1.0, 0.1, 2**33 + 5),
])
def test_device_generator_bit_identical_to_host(seed, tensor, sub, n, mean, std, start):
    dev = torch.empty(n, dtype=torch.float32, device="cuda")
    gen.normal_device(seed, tensor, sub, dev, mean, std, start=start)
    host = gen.normal_host(seed, tensor, sub, n, mean, std, start=start)
    assert np.array_equal(dev.cpu().numpy().view(np.uint32), host.view(np.uint32))


def _edge_matrix():
    rng = np.random.default_rng(11)
    rows = list(rng.standard_normal((8, 64)).astype(np.float32))
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 4, np.float32)
    rows.append(np.concatenate([mids, -mids]))
    rows.append(np.zeros(64, np.float32))
    rows.append(np.concatenate([np.full(32, -0.0, np.float32), np.full(32, 1e-40, np.float32)]))
    rows.append((rng.standard_normal(64) * 1e30).astype(np.float32))
    rows.append((rng.standard_normal(64) * 1e-39).astype(np.float32))
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("which", ["edge", "random"])
def test_device_packer_matches_oracle_bytes(which):
    w = _edge_matrix() if which == "edge" else \
        np.random.default_rng(5).standard_normal((301, 2048)).astype(np.float32)
    q, s = M.mxfp4_pack_device(torch.from_numpy(w).cuda())
    qo, so = oracle.mxfp4_pack(w)
    assert np.array_equal(s.cpu().numpy(), so)
    assert np.array_equal(q.cpu().numpy(), qo)


def test_decode_of_all_256_bytes_matches_oracle_tables():
    """Every byte value through the kernels' cvt-based decode, at several scales."""
    cfg = CONFIGS["tiny_b1"]
    w = synthetic.make_weights(cfg, layout=0)   # canonical bytes, retiled by the layer
    rng = np.random.default_rng(0)
    q = w["w_gu_q"][0]
    s = w["w_gu_s"][0]
    pattern = np.tile(np.arange(256, dtype=np.uint8), q.numel() // 256 + 1)[:q.numel()]
    q.copy_(torch.from_numpy(pattern.reshape(q.shape)))
    # finite fp32 weights never get a scale byte above 252 (amax < 2^128 gives
    # floor(log2 amax) - 2 <= 125); 6 * 2^(253-127) would overflow fp32
    scales = rng.integers(0, 253, s.shape).astype(np.uint8)
    scales.flat[:5] = [0, 1, 127, 251, 252]
    s.copy_(torch.from_numpy(scales))
    layer = synthetic.make_layer(cfg, weights=w)
    got = layer.debug_dequant(0, 0).cpu().numpy().astype(np.float64)
    ref = oracle.mxfp4_dequant(q.cpu().numpy(), s.cpu().numpy())
    assert np.array_equal(got, ref)
    layer.close()


def test_layer_dequant_matches_oracle_packing_of_the_same_draws():
    cfg = CONFIGS["tiny_b1"]
    layer = synthetic.make_layer(cfg)
    inp = oracle.LayerInputs(cfg)
    for e in (0, 17, 63):
        q_gu, s_gu, q_d, s_d = inp.expert_packed(e)
        got0 = layer.debug_dequant(e, 0).cpu().numpy().astype(np.float64)
        got1 = layer.debug_dequant(e, 1).cpu().numpy().astype(np.float64)
        assert np.array_equal(got0, oracle.mxfp4_dequant(q_gu, s_gu))
        assert np.array_equal(got1, oracle.mxfp4_dequant(q_d, s_d))
    layer.close()


@pytest.mark.parametrize("layout", [1, 2, 3, 4])
def test_device_tiled_pack_and_retile_match_host_tiled_pack(layout):
    w = np.random.default_rng(layout).standard_normal((128, 512)).astype(np.float32)
    qh, sh = M.mxfp4_pack(torch.from_numpy(w), layout=layout)
    qd, sd = M.mxfp4_pack_device(torch.from_numpy(w).cuda(), layout=layout)
    assert torch.equal(qd.cpu(), qh) and torch.equal(sd.cpu(), sh)
    qc, sc = M.mxfp4_pack_device(torch.from_numpy(np.stack([w, -w])).cuda().view(256, 512))
    qr, sr = M.mxfp4_retile_device(qc.view(2, 128, 256), sc.view(2, 128, 16), layout)
    qh2, sh2 = M.mxfp4_pack(torch.from_numpy(-w), layout=layout)
    assert torch.equal(qr[0].cpu(), qh) and torch.equal(sr[0].cpu(), sh)
    assert torch.equal(qr[1].cpu(), qh2) and torch.equal(sr[1].cpu(), sh2)


@pytest.mark.parametrize("path", [0, 2, 1])
def test_layer_output_does_not_depend_on_the_weight_layout_given(path):
    """moe_layer_create with canonical, tiled or UMMA expert bytes (relaid into
    the handle's own copy unless already in the path's layouts) gives
    bit-identical outputs on either expert path."""
    cfg = CONFIGS["tiny_b1"]
    x, r = synthetic.make_activations(cfg, B=5)
    outs = []
    for layout in (0, 1, 3):
        w = synthetic.make_weights(cfg, layout=layout)
        layer = synthetic.make_layer(cfg, max_batch=5, weights=w, expert_path=path)
        res = r.clone()
        out = torch.empty_like(x)
        layer.forward(x, res, out)
        torch.cuda.synchronize()
        outs.append((out.cpu(), res.cpu()))
        layer.close()
    for o in outs[1:]:
        assert torch.equal(outs[0][0], o[0]) and torch.equal(outs[0][1], o[1])
