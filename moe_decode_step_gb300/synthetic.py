"""Seeded synthetic MoE layers on the GPU for tests and benchmarks.

Values come from the shared seeded generator (`gen`, device side), bf16
tensors are rounded by torch (round to nearest even), and the expert matrices
are packed to MXFP4 by this library's own device packer.  The CPU oracle
builds the same layer independently from the host side of `gen`.
"""
import torch

import gen
from gen.configs import (T_ROUTER_W, T_ROUTER_BIAS, T_GAMMA, T_SHARED_GU, T_SHARED_D, T_X,
                         T_RESIDUAL, T_EXPERT_GU, T_EXPERT_D, activation_seed)

from . import MoELayer, mxfp4_pack_device


def _normal(seed, tensor, sub, shape, mean, std, device, scratch=None):
    n = 1
    for s in shape:
        n *= s
    out = scratch[:n].view(*shape) if scratch is not None else torch.empty(
        shape, dtype=torch.float32, device=device)
    gen.normal_device(seed, tensor, sub, out, mean, std)
    return out


# weight layout -> (FC1 gate/up layout, FC2 layout)
_LAYOUTS = {0: (0, 0), 1: (2, 1), 3: (4, 3)}


def make_weights(cfg, layer=0, device="cuda", layout=3):
    """Device tensors of one seeded layer (dict in MoELayer's naming).  layout 3
    packs the experts straight into the tcgen05 path's UMMA layouts (FC1 gate/up
    pairs: layout 4, FC2: layout 3), layout 1 into the mma.sync path's tiled
    layouts (2 and 1); layout 0 keeps them canonical."""
    gu_layout, d_layout = _LAYOUTS[layout]
    c = cfg
    s = c.seeds[layer]
    dev = torch.device(device)
    E, d, f, fs = c.n_experts, c.d, c.f, c.f_shared
    w = {}
    w["router_w"] = _normal(s, T_ROUTER_W, 0, (E, d), 0.0, c.std_router(), dev).to(torch.bfloat16)
    w["router_bias"] = _normal(s, T_ROUTER_BIAS, 0, (E,), 0.0, 0.01, dev)
    w["rms_gamma"] = _normal(s, T_GAMMA, 0, (d,), 1.0, 0.1, dev).to(torch.bfloat16)
    w["shared_gu"] = _normal(s, T_SHARED_GU, 0, (2 * fs, d), 0.0, c.std_gu(), dev).to(torch.bfloat16)
    w["shared_d"] = _normal(s, T_SHARED_D, 0, (d, fs), 0.0, c.std_shared_down(),
                            dev).to(torch.bfloat16)
    w["w_gu_q"] = torch.empty((E, 2 * f, d // 2), dtype=torch.uint8, device=dev)
    w["w_gu_s"] = torch.empty((E, 2 * f, d // 32), dtype=torch.uint8, device=dev)
    w["w_d_q"] = torch.empty((E, d, f // 2), dtype=torch.uint8, device=dev)
    w["w_d_s"] = torch.empty((E, d, f // 32), dtype=torch.uint8, device=dev)
    scratch = torch.empty(2 * f * d, dtype=torch.float32, device=dev)
    for e in range(E):
        gu = _normal(s, T_EXPERT_GU, e, (2 * f, d), 0.0, c.std_gu(), dev, scratch)
        mxfp4_pack_device(gu, w["w_gu_q"][e], w["w_gu_s"][e], layout=gu_layout)
        dn = _normal(s, T_EXPERT_D, e, (d, f), 0.0, c.std_down(), dev, scratch)
        mxfp4_pack_device(dn, w["w_d_q"][e], w["w_d_s"][e], layout=d_layout)
    del scratch
    w["mxfp4_layout"] = layout
    return w


def make_activations(cfg, layer=0, attempt=0, device="cuda", B=None):
    """x, residual: device bf16 [B, d] for seed + 1000 * attempt."""
    c = cfg
    B = c.B if B is None else B
    s = activation_seed(c.seeds[layer], attempt)
    dev = torch.device(device)
    if c.drafts > 0 and c.corr != 0.0:
        # a verify batch: the rows mixed on the host (see gen.activation_x)
        x = torch.from_numpy(gen.activation_x(c, s, B)).to(dev).to(torch.bfloat16)
    else:
        x = _normal(s, T_X, 0, (B, c.d), 0.0, 1.0, dev).to(torch.bfloat16)
    r = _normal(s, T_RESIDUAL, 0, (B, c.d), 0.0, 1.0, dev).to(torch.bfloat16)
    return x, r


def make_layer(cfg, layer=0, device="cuda", max_batch=None, weights=None, expert_path=0):
    mb = max_batch if max_batch is not None else max(cfg.B, 1)
    # the layouts the layer reads in place: the tiled ones when it only runs
    # the mma.sync path (expert_path 1, or the default with max_batch 1)
    tiled = expert_path == 1 or (expert_path == 0 and mb == 1)
    w = weights if weights is not None else make_weights(
        cfg, layer, device, layout=1 if tiled else 3)
    return MoELayer(cfg.d, cfg.f, cfg.n_experts, cfg.top_k, cfg.f_shared, mb, w,
                    routed_scale=cfg.routed_scale, rms_eps=cfg.rms_eps,
                    expert_path=expert_path)
