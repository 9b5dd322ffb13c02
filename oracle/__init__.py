"""ORACLE — test infrastructure only.

A plain, slow, fp64 CPU statement of one MoE decode layer (router with biased
top-k, MXFP4 SwiGLU routed experts with weighted combine, bf16 shared expert,
residual add + RMSNorm tail).  The arithmetic lives in oracle.c; this module
draws the seeded inputs through `gen`, packs the expert weights with the
oracle's own MXFP4 packer and sequences the steps.

Only `tests/`, `__graft_entry__.smoke()` and bench.py's CPU-baseline leg may
import this package.  It never imports the CUDA library and the CUDA library
never imports it.

Every function is pinned by the `-m "not gpu"` tests in tests/test_oracle_*.py
(spec tables, brute force, closed forms, invariants); none is "parity unpinned".
"""
import ctypes
import time

import numpy as np

import gen
from gen.configs import (T_ROUTER_W, T_ROUTER_BIAS, T_GAMMA, T_SHARED_GU, T_SHARED_D, T_X,
                         T_RESIDUAL, T_EXPERT_GU, T_EXPERT_D, activation_seed)
from . import build as _build

_lib = None
_P = ctypes.c_void_p


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(_build.build())
        L.oracle_set_threads.argtypes = [ctypes.c_int]
        L.oracle_e2m1_value.argtypes = [ctypes.c_int]
        L.oracle_e2m1_value.restype = ctypes.c_double
        L.oracle_e8m0_value.argtypes = [ctypes.c_int]
        L.oracle_e8m0_value.restype = ctypes.c_double
        L.oracle_e2m1_encode.argtypes = [ctypes.c_double]
        L.oracle_e2m1_encode.restype = ctypes.c_int
        L.oracle_block_exponent.argtypes = [_P]
        L.oracle_block_exponent.restype = ctypes.c_int
        L.oracle_mxfp4_pack.argtypes = [_P, ctypes.c_int64, ctypes.c_int64, _P, _P]
        L.oracle_mxfp4_dequant.argtypes = [_P, _P, ctypes.c_int64, ctypes.c_int64, _P]
        L.oracle_e4m3_value.argtypes = [ctypes.c_int]
        L.oracle_e4m3_value.restype = ctypes.c_double
        L.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        L.oracle_e4m3_encode.restype = ctypes.c_int
        L.oracle_block_exponent_e4m3.argtypes = [_P]
        L.oracle_block_exponent_e4m3.restype = ctypes.c_int
        L.oracle_mxfp8_quant_row.argtypes = [_P, ctypes.c_int64, _P, _P]
        L.oracle_mxfp8_dequant_row.argtypes = [_P, _P, ctypes.c_int64, _P]
        L.oracle_sigmoid.argtypes = [ctypes.c_double]
        L.oracle_sigmoid.restype = ctypes.c_double
        L.oracle_swiglu.argtypes = [ctypes.c_double, ctypes.c_double]
        L.oracle_swiglu.restype = ctypes.c_double
        L.oracle_round_bf16.argtypes = [ctypes.c_double]
        L.oracle_round_bf16.restype = ctypes.c_double
        L.oracle_round_bf16_array.argtypes = [_P, ctypes.c_int64, _P]
        L.oracle_router.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_double, _P, _P, _P, _P]
        for name in ("oracle_mxfp4_fc1", "oracle_mxfp4_fc2"):
            getattr(L, name).argtypes = [_P, _P, ctypes.c_int, ctypes.c_int, _P, ctypes.c_int, _P]
        for name in ("oracle_dense_fc1", "oracle_dense_fc2"):
            getattr(L, name).argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, ctypes.c_int, _P]
        L.oracle_combine.argtypes = [_P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
        L.oracle_tail.argtypes = [_P, _P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                  _P, _P]
        L.oracle_set_threads(gen.host_threads())
        _lib = L
    return _lib


def set_threads(n):
    lib().oracle_set_threads(int(n))


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# MXFP4 (OCP MX v1.0: E2M1 elements, E8M0 scale per 32 contiguous K elements)
# --------------------------------------------------------------------------
def e2m1_value(code):
    return lib().oracle_e2m1_value(int(code))


def e8m0_value(byte):
    return lib().oracle_e8m0_value(int(byte))


def e2m1_encode(t):
    return lib().oracle_e2m1_encode(float(t))


def block_exponent(block32):
    b = _c(block32, np.float32)
    assert b.size == 32
    return lib().oracle_block_exponent(_p(b))


def mxfp4_pack(w):
    """w float32 [rows, k] -> (q uint8 [rows, k/2], s uint8 [rows, k/32])."""
    w = _c(w, np.float32)
    rows, k = w.shape
    assert k % 32 == 0
    q = np.empty((rows, k // 2), np.uint8)
    s = np.empty((rows, k // 32), np.uint8)
    lib().oracle_mxfp4_pack(_p(w), rows, k, _p(q), _p(s))
    return q, s


def mxfp4_dequant(q, s):
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    rows, half = q.shape
    out = np.empty((rows, half * 2), np.float64)
    lib().oracle_mxfp4_dequant(_p(q), _p(s), rows, half * 2, _p(out))
    return out


# --------------------------------------------------------------------------
# MXFP8 activations (OCP MX v1.0: E4M3 elements, E8M0 scale per 32 elements)
# --------------------------------------------------------------------------
def e4m3_value(code):
    return lib().oracle_e4m3_value(int(code))


def e4m3_encode(t):
    return lib().oracle_e4m3_encode(float(t))


def block_exponent_e4m3(block32):
    b = _c(block32, np.float64)
    assert b.size == 32
    return lib().oracle_block_exponent_e4m3(_p(b))


def mxfp8_quant(a):
    """a [rows, k] (k a multiple of 32) -> (q uint8 [rows, k] E4M3 codes,
    s uint8 [rows, k/32] E8M0 scale bytes)."""
    a = _c(np.atleast_2d(a), np.float64)
    rows, k = a.shape
    assert k % 32 == 0
    q = np.empty((rows, k), np.uint8)
    s = np.empty((rows, k // 32), np.uint8)
    for r in range(rows):
        lib().oracle_mxfp8_quant_row(_p(a[r]), k, _p(q[r]), _p(s[r]))
    return q, s


def mxfp8_dequant(q, s):
    q = _c(np.atleast_2d(q), np.uint8)
    s = _c(np.atleast_2d(s), np.uint8)
    rows, k = q.shape
    out = np.empty((rows, k), np.float64)
    for r in range(rows):
        lib().oracle_mxfp8_dequant_row(_p(q[r]), _p(s[r]), k, _p(out[r]))
    return out


def mxfp8_round(a):
    """The values an MXFP8 activation operand carries for a (rows, k)."""
    return mxfp8_dequant(*mxfp8_quant(a))


def round_bf16(a):
    a = _c(a, np.float64)
    out = np.empty_like(a)
    lib().oracle_round_bf16_array(_p(a), a.size, _p(out))
    return out


def sigmoid(v):
    return lib().oracle_sigmoid(float(v))


def swiglu(g, u):
    return lib().oracle_swiglu(float(g), float(u))


# --------------------------------------------------------------------------
# Layer steps
# --------------------------------------------------------------------------
def router(x, wr, bias, top_k, routed_scale):
    """x [B,d], wr [E,d] (bf16 values), bias [E] float32 ->
    (logits [B,E], idx [B,k] int32, w [B,k], gap [B])."""
    x = _c(x, np.float64)
    wr = _c(wr, np.float64)
    bias = _c(bias, np.float32)
    B, d = x.shape
    E = wr.shape[0]
    logits = np.empty((B, E), np.float64)
    idx = np.empty((B, top_k), np.int32)
    w = np.empty((B, top_k), np.float64)
    gap = np.empty(B, np.float64)
    lib().oracle_router(_p(x), B, d, _p(wr), _p(bias), E, top_k, float(routed_scale),
                        _p(logits), _p(idx), _p(w), _p(gap))
    return logits, idx, w, gap


def mxfp4_fc1(q_gu, s_gu, x):
    """h [r,f] = silu(W_gate x) * (W_up x) for an MXFP4 expert; x [r,d]."""
    x = _c(x, np.float64)
    r, d = x.shape
    f = q_gu.shape[0] // 2
    h = np.empty((r, f), np.float64)
    lib().oracle_mxfp4_fc1(_p(_c(q_gu, np.uint8)), _p(_c(s_gu, np.uint8)), d, f, _p(x), r, _p(h))
    return h


def mxfp4_fc2(q_d, s_d, h):
    """y [r,d] = W_down h for an MXFP4 expert; h [r,f]."""
    h = _c(h, np.float64)
    r, f = h.shape
    d = q_d.shape[0]
    y = np.empty((r, d), np.float64)
    lib().oracle_mxfp4_fc2(_p(_c(q_d, np.uint8)), _p(_c(s_d, np.uint8)), d, f, _p(h), r, _p(y))
    return y


def dense_fc1(w_gu, x):
    x = _c(x, np.float64)
    w_gu = _c(w_gu, np.float64)
    r, d = x.shape
    f = w_gu.shape[0] // 2
    h = np.empty((r, f), np.float64)
    lib().oracle_dense_fc1(_p(w_gu), d, f, _p(x), r, _p(h))
    return h


def dense_fc2(w_d, h):
    h = _c(h, np.float64)
    w_d = _c(w_d, np.float64)
    r, f = h.shape
    d = w_d.shape[0]
    y = np.empty((r, d), np.float64)
    lib().oracle_dense_fc2(_p(w_d), d, f, _p(h), r, _p(y))
    return y


def combine(y_pair, w):
    """y_pair [B,k,d], w [B,k] -> y_r [B,d] = sum_j w[b,j] y_pair[b,j]."""
    y_pair = _c(y_pair, np.float64)
    w = _c(w, np.float64)
    B, k, d = y_pair.shape
    y = np.empty((B, d), np.float64)
    lib().oracle_combine(_p(y_pair), _p(w), B, k, d, _p(y))
    return y


def tail(residual, y_r, y_s, gamma, eps):
    """-> (z [B,d], out [B,d]) before any output rounding."""
    residual = _c(residual, np.float64)
    B, d = residual.shape
    z = np.empty((B, d), np.float64)
    out = np.empty((B, d), np.float64)
    lib().oracle_tail(_p(residual), _p(_c(y_r, np.float64)), _p(_c(y_s, np.float64)),
                      _p(_c(gamma, np.float64)), B, d, float(eps), _p(z), _p(out))
    return z, out


# --------------------------------------------------------------------------
# Seeded inputs (drawn through gen on the host, rounded to bf16 by the oracle)
# --------------------------------------------------------------------------
class LayerInputs:
    """Host copies of one seeded layer: dense tensors eagerly, experts lazily."""

    def __init__(self, cfg, layer=0, x_attempt=0, x=None, residual=None):
        self.cfg = cfg
        self.seed = cfg.seeds[layer]
        c = cfg
        s = self.seed
        bf = round_bf16
        self.wr = bf(gen.normal_host(s, T_ROUTER_W, 0, c.n_experts * c.d, 0.0,
                                     c.std_router())).reshape(c.n_experts, c.d)
        self.bias = gen.normal_host(s, T_ROUTER_BIAS, 0, c.n_experts, 0.0, 0.01)
        self.gamma = bf(gen.normal_host(s, T_GAMMA, 0, c.d, 1.0, 0.1))
        self.shared_gu = bf(gen.normal_host(s, T_SHARED_GU, 0, 2 * c.f_shared * c.d, 0.0,
                                            c.std_gu())).reshape(2 * c.f_shared, c.d)
        self.shared_d = bf(gen.normal_host(s, T_SHARED_D, 0, c.d * c.f_shared, 0.0,
                                           c.std_shared_down())).reshape(c.d, c.f_shared)
        self.x_seed = activation_seed(s, x_attempt)
        if x is None:
            x = bf(gen.activation_x(c, self.x_seed))
        if residual is None:
            residual = bf(gen.normal_host(self.x_seed, T_RESIDUAL, 0, c.B * c.d, 0.0,
                                          1.0)).reshape(c.B, c.d)
        self.x = np.asarray(x, np.float64)
        self.residual = np.asarray(residual, np.float64)
        self._experts = {}

    def expert_f32(self, e):
        c = self.cfg
        gu = gen.normal_host(self.seed, T_EXPERT_GU, e, 2 * c.f * c.d, 0.0,
                             c.std_gu()).reshape(2 * c.f, c.d)
        dn = gen.normal_host(self.seed, T_EXPERT_D, e, c.d * c.f, 0.0,
                             c.std_down()).reshape(c.d, c.f)
        return gu, dn

    def expert_packed(self, e):
        """(q_gu, s_gu, q_d, s_d) packed by the oracle's own MXFP4 packer."""
        if e not in self._experts:
            gu, dn = self.expert_f32(e)
            self._experts[e] = mxfp4_pack(gu) + mxfp4_pack(dn)
        return self._experts[e]


def route(inp):
    c = inp.cfg
    return router(inp.x, inp.wr, inp.bias, c.top_k, c.routed_scale)


def forward(inp, rows=None, timings=None, act="exact"):
    """Run the layer for the given rows (default all) of `inp`.

    act="exact": the routed experts multiply the MXFP4 weights by x and h as
    they are (bf16 x, fp64 h).  act="mxfp8": by their MXFP8 roundings (OCP MX
    v1.0 E4M3 elements with one E8M0 scale per 32 along K, mxfp8_round), the
    FP4 x MXFP8 products of the pages' routed-expert kernel; the shared
    expert, router and tail are the same in both.

    Returns a dict with idx, w, gap, logits, h [B,k,f], y_pair [B,k,d], y_r,
    h_s, y_s, z, out (all fp64, pre-rounding) and residual_bf16 / out_bf16.
    Rows outside `rows` are left as NaN in the per-row outputs.
    """
    assert act in ("exact", "mxfp8")
    c = inp.cfg
    B = c.B
    rows = list(range(B)) if rows is None else sorted(rows)
    t0 = time.perf_counter()
    logits, idx, w, gap = route(inp)
    # group the selected (row, slot) pairs by expert, experts ascending
    by_expert = {}
    for b in rows:
        for j in range(c.top_k):
            by_expert.setdefault(int(idx[b, j]), []).append((b, j))
    h = np.full((B, c.top_k, c.f), np.nan)
    y_pair = np.full((B, c.top_k, c.d), np.nan)
    t_route = time.perf_counter()
    t_pack = 0.0
    for e in sorted(by_expert):
        tp = time.perf_counter()
        q_gu, s_gu, q_d, s_d = inp.expert_packed(e)
        t_pack += time.perf_counter() - tp
        pairs = by_expert[e]
        xr = inp.x[[b for b, _ in pairs]]
        if act == "mxfp8":
            xr = mxfp8_round(xr)
        he = mxfp4_fc1(q_gu, s_gu, xr)
        ye = mxfp4_fc2(q_d, s_d, mxfp8_round(he) if act == "mxfp8" else he)
        for t, (b, j) in enumerate(pairs):
            h[b, j] = he[t]
            y_pair[b, j] = ye[t]
    xs = inp.x[rows]
    h_s_rows = dense_fc1(inp.shared_gu, xs)
    y_s_rows = dense_fc2(inp.shared_d, h_s_rows)
    y_r_rows = combine(y_pair[rows], w[rows])
    z_rows, out_rows = tail(inp.residual[rows], y_r_rows, y_s_rows, inp.gamma, c.rms_eps)
    t_end = time.perf_counter()

    def full(rows_arr, width):
        a = np.full((B, width), np.nan)
        a[rows] = rows_arr
        return a

    res = dict(idx=idx, w=w, gap=gap, logits=logits, h=h, y_pair=y_pair,
               y_r=full(y_r_rows, c.d), h_s=full(h_s_rows, c.f_shared), y_s=full(y_s_rows, c.d),
               z=full(z_rows, c.d), out=full(out_rows, c.d), rows=rows,
               n_distinct=len(set(int(e) for e in idx[rows].ravel())))
    res["residual_bf16"] = round_bf16(res["z"])
    res["out_bf16"] = round_bf16(res["out"])
    if timings is not None:
        timings["route_s"] = t_route - t0
        timings["pack_s"] = t_pack
        timings["compute_s"] = (t_end - t0) - t_pack
    return res


def clean_inputs(cfg, layer=0, tie_gap=1e-5, max_attempts=20):
    """Draw inputs, redrawing x / residual (seed + 1000*attempt) while any row's
    k-th vs (k+1)-th biased-score gap is below `tie_gap`."""
    for attempt in range(max_attempts):
        inp = LayerInputs(cfg, layer, attempt)
        _, _, _, gap = route(inp)
        if np.all(gap >= tie_gap):
            inp.attempt = attempt
            return inp
    raise RuntimeError(f"no tie-free draw for {cfg.name} in {max_attempts} attempts")
