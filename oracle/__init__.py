"""ctypes binding of liboracle.so -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.

The oracle is a plain fp64 CPU statement of one decode step (oracle.c).  Only
the tests, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py`
may import this package.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

import synth as synth_kinds  # tensor kind ids only

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liboracle.so")

c_int, c_double, c_float = ctypes.c_int, ctypes.c_double, ctypes.c_float
P_D = ctypes.POINTER(ctypes.c_double)
P_F = ctypes.POINTER(ctypes.c_float)
P_I = ctypes.POINTER(ctypes.c_int32)


class OrcConfig(ctypes.Structure):
    _fields_ = [(n, c_int) for n in ("n_layers", "hidden", "n_q", "n_kv", "head_dim",
                                     "n_experts", "top_k", "inter", "vocab", "page_size",
                                     "window", "full_period")] + \
               [(n, c_double) for n in ("rope_base", "eps", "weight_sigma", "kv_sigma")] + \
               [("expert_fp8", c_int), ("expert_fp4", c_int)]


class OrcMatrix(ctypes.Structure):
    _fields_ = [("row", ctypes.c_void_p), ("ctx", ctypes.c_void_p), ("rows", c_int),
                ("cols", c_int)]


class OrcDense(ctypes.Structure):
    _fields_ = [("data", P_D), ("cols", c_int)]


class OrcStepIn(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("batch", c_int), ("tokens", P_I), ("seq_lens", P_I),
                ("block_tables", P_I), ("max_pages", c_int), ("router_bias", P_F),
                ("force_ids", P_I), ("n_rows", c_int), ("rows", P_I), ("norm_gamma", P_D),
                ("final_gamma", P_D), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("num_pages", ctypes.c_int64)]


class OrcStepOut(ctypes.Structure):
    _fields_ = [("logits", P_D), ("ids", P_I), ("weights", P_D), ("own_ids", P_I),
                ("margin", P_F), ("router_logits", P_F), ("hidden", P_D), ("kv_new", P_D),
                ("attn", P_D)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            from .build import build
            build()
        L = ctypes.CDLL(LIB_PATH)
        L.orc_rmsnorm.argtypes = [c_int, P_D, P_D, c_double, P_D]
        L.orc_rope.argtypes = [c_int, P_D, ctypes.c_int64, c_double]
        L.orc_softmax.argtypes = [c_int, P_D, P_D]
        L.orc_synth_dense.argtypes = [ctypes.POINTER(OrcConfig), ctypes.c_uint64, c_int, c_int, c_int, P_D]
        L.orc_synth_dense.restype = ctypes.c_int64
        L.orc_e4m3_value.argtypes = [c_int]
        L.orc_e4m3_value.restype = c_double
        L.orc_e2m1_value.argtypes = [c_int]
        L.orc_e2m1_value.restype = c_double
        L.orc_silu.argtypes = [c_double]
        L.orc_silu.restype = c_double
        L.orc_matvec.argtypes = [ctypes.POINTER(OrcMatrix), P_D, P_D]
        L.orc_attend.argtypes = [c_int, c_int, P_D, P_D, P_D, c_double, P_D]
        L.orc_attend_partial.argtypes = [c_int, c_int, P_D, P_D, P_D, c_double, P_D, P_D, P_D]
        L.orc_attend_combine.argtypes = [c_int, c_int, P_D, P_D, P_D, P_D]
        L.orc_topk.argtypes = [c_int, c_int, P_F, P_I, P_F]
        L.orc_topk.restype = c_int
        L.orc_swiglu_expert.argtypes = [ctypes.POINTER(OrcMatrix)] * 3 + [P_D, P_D]
        L.orc_moe_routed.argtypes = [c_int, P_I, P_D] + [ctypes.POINTER(OrcMatrix)] * 3 + [P_D, P_D]
        L.orc_moe_dense_gated.argtypes = [c_int, P_D] + [ctypes.POINTER(OrcMatrix)] * 3 + [P_D, P_D]
        L.orc_kv_slot.argtypes = [ctypes.c_int64, c_int, P_I, c_int, P_I, P_I]
        L.orc_kv_slot.restype = c_int
        L.orc_pool_vec.argtypes = [ctypes.POINTER(OrcConfig), ctypes.c_uint64, c_int, c_int, c_int,
                                   c_int, c_int, P_D]
        L.orc_route_queue.argtypes = [c_int, c_int, c_int, P_I, P_I, P_I, P_I, P_I]
        L.orc_route_queue.restype = c_int
        L.orc_decode_step.argtypes = [ctypes.POINTER(OrcConfig), ctypes.POINTER(OrcStepIn),
                                      ctypes.POINTER(OrcStepOut)]
        L.orc_decode_step.restype = c_int
        _lib = L
    return _lib


def _d(a):
    return a.ctypes.data_as(P_D)


def _f(a):
    return a.ctypes.data_as(P_F)


def _i(a):
    return a.ctypes.data_as(P_I)


def _dbl(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def config_from_shape(shape) -> OrcConfig:
    return OrcConfig(shape.n_layers, shape.hidden, shape.n_q, shape.n_kv, shape.head_dim,
                     shape.n_experts, shape.top_k, shape.inter, shape.vocab, shape.page_size,
                     shape.window, shape.full_period, shape.rope_base, shape.eps,
                     shape.weight_sigma, shape.kv_sigma, int(getattr(shape, "expert_fp8", False)),
                     int(getattr(shape, "expert_fp4", False)))


# ----------------------------------------------------------- layer operations

def rmsnorm(x, gamma=None, eps=1e-5):
    x = _dbl(x)
    out = np.empty_like(x)
    g = _dbl(gamma) if gamma is not None else None
    lib().orc_rmsnorm(x.size, _d(x), _d(g) if g is not None else None, eps, _d(out))
    return out


def rope(v, pos, base=500000.0):
    v = _dbl(v).copy()
    lib().orc_rope(v.size, _d(v), int(pos), base)
    return v


def softmax(s):
    s = _dbl(s)
    p = np.empty_like(s)
    lib().orc_softmax(s.size, _d(s), _d(p))
    return p


def silu(x):
    return lib().orc_silu(float(x))


def synth_matrix(shape, seed: int, kind: int, layer: int = 0, expert: int = 0) -> np.ndarray:
    """A weight matrix exactly as the oracle reads it (FP8 / FP4 experts dequantized)."""
    rows, cols = {synth_kinds.WG: (shape.inter, shape.hidden), synth_kinds.WU: (shape.inter, shape.hidden),
                  synth_kinds.WD: (shape.hidden, shape.inter)}[kind]
    cfg = config_from_shape(shape)
    out = np.empty((rows, cols), np.float64)
    n = lib().orc_synth_dense(ctypes.byref(cfg), seed, kind, layer, expert, _d(out))
    assert n == rows * cols
    return out


def e2m1_value(code: int) -> float:
    """The value of an FP4 E2M1 code (the oracle's own decoding)."""
    return lib().orc_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    """The value of an OCP FP8 E4M3 code (the oracle's own decoding)."""
    return lib().orc_e4m3_value(int(code))


class Dense:
    """A dense matrix as an oracle row source (keeps its buffers alive)."""

    def __init__(self, W):
        self.W = _dbl(W)
        self.dense = OrcDense(_d(self.W), self.W.shape[1])
        fn = ctypes.cast(lib().orc_dense_row, ctypes.c_void_p).value
        self.m = OrcMatrix(fn, ctypes.cast(ctypes.pointer(self.dense), ctypes.c_void_p).value,
                           self.W.shape[0], self.W.shape[1])


def matvec(W, x):
    D = Dense(W)
    x = _dbl(x)
    y = np.empty(D.W.shape[0])
    lib().orc_matvec(ctypes.byref(D.m), _d(x), _d(y))
    return y


def attend(q, K, V, scale):
    q, K, V = _dbl(q), _dbl(K), _dbl(V)
    out = np.empty(q.size)
    lib().orc_attend(q.size, K.shape[0], _d(q), _d(K), _d(V), scale, _d(out))
    return out


def attend_partial(q, K, V, scale):
    q, K, V = _dbl(q), _dbl(K), _dbl(V)
    m, l_, o = c_double(), c_double(), np.empty(q.size)
    lib().orc_attend_partial(q.size, K.shape[0], _d(q), _d(K), _d(V), scale, ctypes.byref(m),
                             ctypes.byref(l_), _d(o))
    return m.value, l_.value, o


def attend_combine(m, l_, o):
    m, l_, o = _dbl(m), _dbl(l_), _dbl(o)
    out = np.empty(o.shape[1])
    lib().orc_attend_combine(o.shape[1], o.shape[0], _d(m), _d(l_), _d(o), _d(out))
    return out


def topk(logits, k):
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    ids = np.empty(k, dtype=np.int32)
    margin = c_float()
    rc = lib().orc_topk(lg.size, k, _f(lg), _i(ids), ctypes.byref(margin))
    if rc != 0:
        raise ValueError("bad k")
    return ids, margin.value


def swiglu_expert(Wg, Wu, Wd, x):
    g, u, dn = Dense(Wg), Dense(Wu), Dense(Wd)
    x = _dbl(x)
    out = np.empty(dn.W.shape[0])
    lib().orc_swiglu_expert(ctypes.byref(g.m), ctypes.byref(u.m), ctypes.byref(dn.m), _d(x),
                            _d(out))
    return out


def _experts(Wgs, Wus, Wds):
    keep = [[Dense(w) for w in ws] for ws in (Wgs, Wus, Wds)]
    arrs = [(OrcMatrix * len(ds))(*[d.m for d in ds]) for ds in keep]
    return keep, arrs


def moe_routed(ids, w, Wgs, Wus, Wds, x):
    keep, (ag, au, ad) = _experts(Wgs, Wus, Wds)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w, x = _dbl(w), _dbl(x)
    out = np.empty(keep[2][0].W.shape[0])
    lib().orc_moe_routed(ids.size, _i(ids), _d(w), ag, au, ad, _d(x), _d(out))
    return out


def moe_dense_gated(gate, Wgs, Wus, Wds, x):
    keep, (ag, au, ad) = _experts(Wgs, Wus, Wds)
    gate, x = _dbl(gate), _dbl(x)
    out = np.empty(keep[2][0].W.shape[0])
    lib().orc_moe_dense_gated(gate.size, _d(gate), ag, au, ad, _d(x), _d(out))
    return out


def kv_slot(pos, page_size, block_row):
    br = np.ascontiguousarray(block_row, dtype=np.int32)
    page, off = ctypes.c_int32(), ctypes.c_int32()
    rc = lib().orc_kv_slot(int(pos), page_size, _i(br), br.size, ctypes.byref(page),
                           ctypes.byref(off))
    return (page.value, off.value) if rc == 0 else None


def pool_vec(shape, seed, is_v, layer, page, head, slot):
    cfg = config_from_shape(shape)
    out = np.empty(shape.head_dim)
    lib().orc_pool_vec(ctypes.byref(cfg), seed, int(is_v), layer, page, head, slot, _d(out))
    return out


@dataclass
class RouteQueue:
    counts: np.ndarray   # [E] rows routed to each expert
    offsets: np.ndarray  # [E + 1] exclusive prefix sum
    rows: np.ndarray     # [B * k] expert-ordered list of b * k + j
    active: np.ndarray   # [n_active, 3] {expert, offset, count}, experts ascending


def route_queue(ids, n_experts: int) -> RouteQueue:
    """The canonical MoE work queue of one layer from its routing ids [B][k]."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    B, k = ids.shape
    counts = np.empty(n_experts, np.int32)
    offsets = np.empty(n_experts + 1, np.int32)
    rows = np.empty(B * k, np.int32)
    active = np.empty((n_experts, 3), np.int32)
    n = lib().orc_route_queue(B, k, n_experts, _i(ids), _i(counts), _i(offsets), _i(rows), _i(active))
    if n < 0:
        raise ValueError("expert id out of range")
    return RouteQueue(counts, offsets, rows, active[:n].copy())


# ------------------------------------------------------------- the full step

@dataclass
class StepResult:
    logits: np.ndarray        # [R, V] float64
    ids: np.ndarray           # [L, R, k] experts used
    weights: np.ndarray       # [L, R, k]
    own_ids: np.ndarray       # [L, R, k]
    margin: np.ndarray        # [L, R]
    router_logits: np.ndarray  # [L, R, E] float32
    hidden: np.ndarray | None
    kv_new: np.ndarray | None
    attn: np.ndarray | None
    rows: np.ndarray


def decode_step(shape, seed, tokens, seq_lens, block_tables, router_bias=None, rows=None,
                force_ids=None, want_hidden=False, want_kv=False, want_attn=False, gains=None,
                pools=None) -> StepResult:
    """One decode step of the given rows.  gains: (layer gains [L][H], final
    gain [H]) or None for ones.  pools: (K pool, V pool) as writable uint16
    arrays [L][pages][n_kv][P][d] of BF16 bits, read through the block table
    and updated with the new K/V, or None for the generator's pool."""
    cfg = config_from_shape(shape)
    ng = fg = kp = vp = None
    if gains is not None:
        ng = np.ascontiguousarray(gains[0], np.float64)
        fg = np.ascontiguousarray(gains[1], np.float64)
        assert ng.shape == (shape.n_layers, shape.hidden) and fg.shape == (shape.hidden,)
    if pools is not None:
        kp, vp = pools
        for a in (kp, vp):
            assert a.dtype == np.uint16 and a.flags.c_contiguous and a.flags.writeable
            assert a.shape[0] == shape.n_layers and a.shape[2:] == (shape.n_kv, shape.page_size,
                                                                    shape.head_dim)
        assert kp.shape == vp.shape
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    B = tokens.size
    rows = np.arange(B, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    R, L, H, V = rows.size, shape.n_layers, shape.hidden, shape.vocab
    k, E = shape.top_k, shape.n_experts
    bias = np.ascontiguousarray(router_bias, np.float32) if router_bias is not None else None
    force = np.ascontiguousarray(force_ids, np.int32) if force_ids is not None else None
    res = StepResult(np.empty((R, V)), np.empty((L, R, k), np.int32), np.empty((L, R, k)),
                     np.empty((L, R, k), np.int32), np.empty((L, R), np.float32),
                     np.empty((L, R, E), np.float32),
                     np.empty((L + 1, R, H)) if want_hidden else None,
                     np.empty((L, R, 2, shape.n_kv, shape.head_dim)) if want_kv else None,
                     np.empty((L, R, shape.n_q * shape.head_dim)) if want_attn else None, rows)
    sin = OrcStepIn(seed, B, _i(tokens), _i(seq_lens), _i(bt), bt.shape[1],
                    _f(bias) if bias is not None else None,
                    _i(force) if force is not None else None, R, _i(rows),
                    _d(ng) if ng is not None else None, _d(fg) if fg is not None else None,
                    kp.ctypes.data if kp is not None else None, vp.ctypes.data if vp is not None else None,
                    kp.shape[1] if kp is not None else 0)
    sout = OrcStepOut(_d(res.logits), _i(res.ids), _d(res.weights), _i(res.own_ids),
                      _f(res.margin), _f(res.router_logits),
                      _d(res.hidden) if want_hidden else None,
                      _d(res.kv_new) if want_kv else None,
                      _d(res.attn) if want_attn else None)
    rc = lib().orc_decode_step(ctypes.byref(cfg), ctypes.byref(sin), ctypes.byref(sout))
    if rc != 0:
        raise ValueError("orc_decode_step rejected its arguments")
    return res
