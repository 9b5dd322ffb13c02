"""Seeded synthetic workloads for one MoE decode layer.

Shapes and value distributions follow the workload descriptions that go with
the Kimi K3 latency-specialised decode write-ups: a tiny layer (d=1024, f=256,
64 experts, top-4) for fast exact checks, and the full-size layer (d=7168,
f=1536, 896 experts, top-16; each MXFP4 expert 17,547,264 bytes, the figure
the teardown page gives in "What one decode step of Kimi K3 does") at B = 1,
8 and 64 rows, plus a chain of four full-size layers at B = 1.  The
teardown's verify steps (section "What DSpark adds": an anchor token and 7
drafts, 8 rows that route independently, about 120 distinct experts; at most
64 rows per verify batch) are the B = 8 and B = 64 layers.  verify_b16 adds a
case the pages do not model: 16 rows in groups of 4 with correlated hidden
states, so that several rows share an expert (runs of up to 4 rows per
expert at full size).

Every "N(a, b)" is read as mean a, standard deviation b.
"""
from dataclasses import dataclass, field
import math

import numpy as np

# Tensor ids in the Philox counter (word 2); word 3 carries the expert index.
T_ROUTER_W = 1
T_ROUTER_BIAS = 2
T_GAMMA = 3
T_SHARED_GU = 4
T_SHARED_D = 5
T_X = 6
T_RESIDUAL = 7
T_EXPERT_GU = 8
T_EXPERT_D = 9


def f32(v):
    """The float32 value both sides pass to the generator for a std/mean."""
    return float(np.float32(v))


@dataclass(frozen=True)
class LayerConfig:
    name: str
    B: int
    d: int
    f: int
    n_experts: int
    top_k: int
    f_shared: int
    seeds: tuple            # one weight seed per layer (chain: several)
    routed_scale: float = 2.5
    rms_eps: float = 1e-6
    drafts: int = 0         # verify batch: rows come in groups of 1 + drafts
    corr: float = 0.0       # correlation of x between the rows of a group

    @property
    def n_layers(self):
        return len(self.seeds)

    def std_router(self):
        return f32(1.0 / math.sqrt(self.d))

    def std_gu(self):
        return f32(1.0 / math.sqrt(self.d))

    def std_down(self):
        return f32(1.0 / math.sqrt(self.f))

    def std_shared_down(self):
        return f32(1.0 / math.sqrt(self.f_shared))

    def expert_bytes(self):
        """MXFP4 bytes per expert: 3*d*f nibbles/2 + 3*d*f/32 scale bytes."""
        n = 3 * self.d * self.f
        return n // 2 + n // 32


CONFIGS = {
    "tiny_b1": LayerConfig("tiny_b1", 1, 1024, 256, 64, 4, 256, (0,)),
    "full_b1": LayerConfig("full_b1", 1, 7168, 1536, 896, 16, 1536, (1,)),
    "full_b8": LayerConfig("full_b8", 8, 7168, 1536, 896, 16, 1536, (2,)),
    "full_b64": LayerConfig("full_b64", 64, 7168, 1536, 896, 16, 1536, (3,)),
    "chain4_b1": LayerConfig("chain4_b1", 1, 7168, 1536, 896, 16, 1536, (10, 11, 12, 13)),
    "verify_b16": LayerConfig("verify_b16", 16, 7168, 1536, 896, 16, 1536, (4,), drafts=3,
                              corr=0.95),
}


def activation_seed(seed, attempt):
    """x / residual redraw after a near-tie: seed + 1000 * attempt."""
    return seed + 1000 * attempt
