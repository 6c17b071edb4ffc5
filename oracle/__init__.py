"""Python handle on the CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this module.  It is a plain, slow, f64
implementation of one MoE layer forward written from the pages; the GPU path
shares no code with it.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(_HERE, "_lib", "liboracle.so")

SHARED_BF16 = 0
SHARED_KQUANT = 1


class Cfg(ctypes.Structure):
    _fields_ = [("dim", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_routed", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("gate_temp", ctypes.c_float), ("norm_topk_prob", ctypes.c_int32),
                ("route_scale", ctypes.c_float), ("swiglu_limit", ctypes.c_float), ("score_func", ctypes.c_int32)]


SCORE_SQRTSOFTPLUS, SCORE_SIGMOID, SCORE_SOFTMAX = 0, 1, 2


class Layer(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("router_w", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("given_logits", ctypes.c_void_p), ("experts", ctypes.c_void_p), ("shared_kind", ctypes.c_int32),
                ("sh1", ctypes.c_void_p), ("sh3", ctypes.c_void_p), ("sh2", ctypes.c_void_p),
                ("bias_vl", ctypes.c_void_p), ("image_mask", ctypes.c_void_p)]


class Stats(ctypes.Structure):
    _fields_ = [("nan_keys", ctypes.c_int32), ("clipped", ctypes.c_int32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(SO):
            raise RuntimeError(f"{SO} is missing: run __graft_entry__.build() first")
        L = ctypes.CDLL(SO)
        vp, i32, f32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double
        L.orc_bf16_value.restype = dbl
        L.orc_bf16_value.argtypes = [ctypes.c_uint16]
        L.orc_bf16_from_f32.restype = ctypes.c_uint16
        L.orc_bf16_from_f32.argtypes = [f32]
        L.orc_f16_value.restype = dbl
        L.orc_f16_value.argtypes = [ctypes.c_uint16]
        L.orc_f16_from_f32.restype = ctypes.c_uint16
        L.orc_f16_from_f32.argtypes = [f32]
        L.orc_dequant_q2k.argtypes = [vp, vp]
        L.orc_dequant_q3k.argtypes = [vp, vp]
        L.orc_q3k_scale_code.restype = i32
        L.orc_q3k_scale_code.argtypes = [vp, i32]
        L.orc_dequant_matrix.argtypes = [i32, vp, i32, i32, vp]
        L.orc_quantize_q8_1.argtypes = [vp, i32, vp]
        L.orc_dequant_q8_1.argtypes = [vp, i32, vp]
        L.orc_router_logits.argtypes = [vp, i32, vp, i32, i32, vp]
        L.orc_score.restype = f32
        L.orc_score.argtypes = [f32, f32]
        L.orc_route_from_logits.restype = i32
        L.orc_route_from_logits.argtypes = [ctypes.POINTER(Cfg), vp, i32, vp, vp, vp]
        L.orc_route_from_logits_vl.restype = i32
        L.orc_route_from_logits_vl.argtypes = [ctypes.POINTER(Cfg), vp, i32, vp, vp, vp, vp, vp]
        L.orc_scores.argtypes = [ctypes.POINTER(Cfg), vp, vp]
        L.orc_swiglu.restype = dbl
        L.orc_swiglu.argtypes = [dbl, dbl, dbl, vp]
        L.orc_expert_kquant.argtypes = [ctypes.POINTER(Cfg), vp, vp, vp, vp, vp, vp]
        L.orc_shared_bf16.argtypes = [ctypes.POINTER(Cfg), vp, vp, vp, vp, vp, vp]
        L.orc_moe_layer.restype = i32
        L.orc_moe_layer.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Layer), vp, i32, vp, vp, vp, i32,
                                    ctypes.POINTER(Stats)]
        L.orc_flip_candidates.restype = i32
        L.orc_flip_candidates.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Layer), i32, vp, vp, dbl, dbl, i32, vp,
                                          vp]
        L.orc_moe_layer_dense.restype = i32
        L.orc_moe_layer_dense.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Layer), i32, vp, vp, vp]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def make_cfg(dim, inter, n_routed, topk, gate_temp=1.0, norm_topk_prob=True, route_scale=1.5, swiglu_limit=10.0,
             score_func=SCORE_SQRTSOFTPLUS):
    return Cfg(dim, inter, n_routed, topk, gate_temp, int(bool(norm_topk_prob)), route_scale, swiglu_limit,
               int(score_func))


def cfg_of(w) -> Cfg:
    """oracle config of a synth.workloads.Workload"""
    return make_cfg(w.dim, w.inter, w.n_routed, w.topk, w.gate_temp, w.norm_topk_prob, w.route_scale,
                    w.swiglu_limit, getattr(w, "score_func", SCORE_SQRTSOFTPLUS))


# ----------------------------------------------------------------- formats

def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(bits)


def bf16_from_f32(v: float) -> int:
    return lib().orc_bf16_from_f32(v)


def f16_value(bits: int) -> float:
    return lib().orc_f16_value(bits)


def f16_from_f32(v: float) -> int:
    return lib().orc_f16_from_f32(v)


def dequant_q2k(block: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(block, dtype=np.uint8)
    assert b.size == 84
    out = np.empty(256, dtype=np.float64)
    lib().orc_dequant_q2k(_p(b), _p(out))
    return out


def dequant_q3k(block: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(block, dtype=np.uint8)
    assert b.size == 110
    out = np.empty(256, dtype=np.float64)
    lib().orc_dequant_q3k(_p(b), _p(out))
    return out


def q3k_scale_code(scales12: np.ndarray, b: int) -> int:
    s = np.ascontiguousarray(scales12, dtype=np.uint8)
    return lib().orc_q3k_scale_code(_p(s), b)


def dequant_matrix(kind: int, mat: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """kind 2 = Q2_K, 3 = Q3_K; [rows][cols/256] blocks -> f64 [rows, cols]"""
    m = np.ascontiguousarray(mat, dtype=np.uint8)
    out = np.empty((rows, cols), dtype=np.float64)
    lib().orc_dequant_matrix(kind, _p(m), rows, cols, _p(out))
    return out


def quantize_q8_1(x: np.ndarray) -> np.ndarray:
    """q8_1 blocks (uint8 [..., n/32*36]) of f32 rows x [..., n]"""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.shape[-1]
    rows = x.reshape(-1, n)
    out = np.empty((rows.shape[0], n // 32 * 36), dtype=np.uint8)
    for r in range(rows.shape[0]):
        lib().orc_quantize_q8_1(_p(rows[r]), n, _p(out[r]))
    return out.reshape(x.shape[:-1] + (n // 32 * 36,))


def dequant_q8_1(q8: np.ndarray, n: int) -> np.ndarray:
    q = np.ascontiguousarray(q8, dtype=np.uint8)
    out = np.empty(n, dtype=np.float64)
    lib().orc_dequant_q8_1(_p(q), n, _p(out))
    return out


def router_logits(x_bf16: np.ndarray, router_bf16: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    W = np.ascontiguousarray(router_bf16, dtype=np.uint16)
    m, D = x.shape
    N = W.shape[0]
    z = np.empty((m, N), dtype=np.float32)
    lib().orc_router_logits(_p(x), m, _p(W), D, N, _p(z))
    return z


def score(z: float, gate_temp: float = 1.0) -> float:
    return lib().orc_score(z, gate_temp)


def route_from_logits(cfg: Cfg, logits: np.ndarray, bias: np.ndarray, bias_vl=None, image_mask=None):
    """(weights f32 [m, k], indices i32 [m, k], nan_keys); tokens with a nonzero
    image_mask entry pick with bias_vl"""
    z = np.ascontiguousarray(logits, dtype=np.float32)
    b = np.ascontiguousarray(bias, dtype=np.float32)
    bv = None if bias_vl is None else np.ascontiguousarray(bias_vl, dtype=np.float32)
    im = None if image_mask is None else np.ascontiguousarray(image_mask, dtype=np.uint8)
    m = z.shape[0]
    w = np.empty((m, cfg.topk), dtype=np.float32)
    idx = np.empty((m, cfg.topk), dtype=np.int32)
    nan = lib().orc_route_from_logits_vl(ctypes.byref(cfg), _p(z), m, _p(b), _p(bv), _p(im), _p(w), _p(idx))
    return w, idx, nan


def scores(cfg: Cfg, logits_row: np.ndarray) -> np.ndarray:
    """f32 scores of one token's logits by the configuration's score function"""
    z = np.ascontiguousarray(logits_row, dtype=np.float32)
    s = np.empty(cfg.n_routed, dtype=np.float32)
    lib().orc_scores(ctypes.byref(cfg), _p(z), _p(s))
    return s


def swiglu(g: float, u: float, limit: float) -> float:
    return lib().orc_swiglu(g, u, limit, None)


def expert_kquant(cfg: Cfg, xq8: np.ndarray, w1, w3, w2):
    xq8 = np.ascontiguousarray(xq8, dtype=np.uint8)
    E = np.empty(cfg.dim, dtype=np.float64)
    clipped = ctypes.c_int(0)
    lib().orc_expert_kquant(ctypes.byref(cfg), _p(xq8), _p(w1), _p(w3), _p(w2), _p(E), ctypes.addressof(clipped))
    return E, clipped.value


def shared_bf16(cfg: Cfg, x_row: np.ndarray, w1, w3, w2):
    x = np.ascontiguousarray(x_row, dtype=np.uint16)
    S = np.empty(cfg.dim, dtype=np.float64)
    clipped = ctypes.c_int(0)
    lib().orc_shared_bf16(ctypes.byref(cfg), _p(x), _p(w1), _p(w3), _p(w2), _p(S), ctypes.addressof(clipped))
    return S, clipped.value


@dataclass
class LayerResult:
    out: np.ndarray        # f64 [n_tok, dim]
    topk_w: np.ndarray     # f32 [n_tok, k]
    topk_idx: np.ndarray   # i32 [n_tok, k]
    nan_keys: int
    clipped: int


def moe_layer(cfg: Cfg, x, router_w, bias, experts, shared_kind, sh1, sh3, sh2, tokens=None, given_logits=None,
              nthreads=None, bias_vl=None, image_mask=None) -> LayerResult:
    """One MoE layer on the CPU.

    experts: list of n_routed entries, each None or a (w1, w3, w2) tuple of uint8
    arrays.  tokens: optional list of token rows to compute (default: all).
    given_logits: optional f32 [m, n_routed] to route from instead of the router.
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    router_w = np.ascontiguousarray(router_w, dtype=np.uint16)
    bias = np.ascontiguousarray(bias, dtype=np.float32)
    m = x.shape[0]
    keep = []
    table = (ctypes.c_void_p * (3 * cfg.n_routed))()
    for e in range(cfg.n_routed):
        ent = experts[e] if e < len(experts) else None
        if ent is None:
            continue
        for j in range(3):
            a = np.ascontiguousarray(ent[j], dtype=np.uint8)
            keep.append(a)
            table[3 * e + j] = a.ctypes.data
    sh = [np.ascontiguousarray(s) for s in (sh1, sh3, sh2)]
    gl = None if given_logits is None else np.ascontiguousarray(given_logits, dtype=np.float32)
    bv = None if bias_vl is None else np.ascontiguousarray(bias_vl, dtype=np.float32)
    im = None if image_mask is None else np.ascontiguousarray(image_mask, dtype=np.uint8)
    L = Layer(_p(x), _p(router_w), _p(bias), _p(gl), ctypes.cast(table, ctypes.c_void_p), shared_kind,
              _p(sh[0]), _p(sh[1]), _p(sh[2]), _p(bv), _p(im))
    if tokens is None:
        tok = None
        n_tok = m
    else:
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        n_tok = tok.size
    out = np.empty((n_tok, cfg.dim), dtype=np.float64)
    w = np.empty((n_tok, cfg.topk), dtype=np.float32)
    idx = np.empty((n_tok, cfg.topk), dtype=np.int32)
    st = Stats()
    nthreads = nthreads or max(1, os.cpu_count() or 1)
    rc = lib().orc_moe_layer(ctypes.byref(cfg), ctypes.byref(L), _p(tok), n_tok, _p(out), _p(w), _p(idx), nthreads,
                             ctypes.byref(st))
    if rc != 0:
        raise RuntimeError(f"oracle layer failed with status {rc}")
    return LayerResult(out, w, idx, st.nan_keys, st.clipped)


def moe_layer_dense(cfg: Cfg, x, router_w, bias, experts, shared_kind, sh1, sh3, sh2, given_logits=None,
                    bias_vl=None, image_mask=None) -> LayerResult:
    """The brute-force mode: every matrix dequantised to dense f64 up front,
    textbook loops over all tokens.  Small inputs only (every expert must be
    given).  clipped and nan_keys are not counted here (0)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    router_w = np.ascontiguousarray(router_w, dtype=np.uint16)
    bias = np.ascontiguousarray(bias, dtype=np.float32)
    m = x.shape[0]
    keep = []
    table = (ctypes.c_void_p * (3 * cfg.n_routed))()
    for e in range(cfg.n_routed):
        for j in range(3):
            a = np.ascontiguousarray(experts[e][j], dtype=np.uint8)
            keep.append(a)
            table[3 * e + j] = a.ctypes.data
    sh = [np.ascontiguousarray(s) for s in (sh1, sh3, sh2)]
    gl = None if given_logits is None else np.ascontiguousarray(given_logits, dtype=np.float32)
    bv = None if bias_vl is None else np.ascontiguousarray(bias_vl, dtype=np.float32)
    im = None if image_mask is None else np.ascontiguousarray(image_mask, dtype=np.uint8)
    L = Layer(_p(x), _p(router_w), _p(bias), _p(gl), ctypes.cast(table, ctypes.c_void_p), shared_kind,
              _p(sh[0]), _p(sh[1]), _p(sh[2]), _p(bv), _p(im))
    out = np.empty((m, cfg.dim), dtype=np.float64)
    w = np.empty((m, cfg.topk), dtype=np.float32)
    idx = np.empty((m, cfg.topk), dtype=np.int32)
    rc = lib().orc_moe_layer_dense(ctypes.byref(cfg), ctypes.byref(L), m, _p(out), _p(w), _p(idx))
    if rc != 0:
        raise RuntimeError(f"dense oracle layer failed with status {rc}")
    return LayerResult(out, w, idx, 0, 0)


@dataclass
class Flips:
    meta: np.ndarray       # i32 [n, 4]: slot (k = shared expert), kind, element or block, alternative
    delta: np.ndarray      # f64 [n, dim]: the change each makes to the token's output
    total: int             # candidates found (only the first max_c are held)


FLIP_Q8_CODE, FLIP_Q8_SCALE, FLIP_BF16 = 0, 1, 2


def flip_candidates(cfg: Cfg, x, t: int, topk_w, topk_idx, experts, shared_kind, sh1, sh3, sh2, kappa: float,
                    min_change: float = 0.0, max_c: int = 4096) -> Flips:
    """The requantisations of h that g and u known to within kappa * sum|terms|
    can change, for token t of x routed to topk_idx with weights topk_w
    (reading C-F1 of moe_oracle.c); those changing no output element by
    min_change or more are left out."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    keep = []
    table = (ctypes.c_void_p * (3 * cfg.n_routed))()
    for e in range(cfg.n_routed):
        ent = experts[e] if e < len(experts) else None
        if ent is None:
            continue
        for j in range(3):
            a = np.ascontiguousarray(ent[j], dtype=np.uint8)
            keep.append(a)
            table[3 * e + j] = a.ctypes.data
    sh = [np.ascontiguousarray(s) for s in (sh1, sh3, sh2)]
    L = Layer(_p(x), None, None, None, ctypes.cast(table, ctypes.c_void_p), shared_kind,
              _p(sh[0]), _p(sh[1]), _p(sh[2]), None, None)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    meta = np.zeros((max_c, 4), dtype=np.int32)
    delta = np.zeros((max_c, cfg.dim), dtype=np.float64)
    n = lib().orc_flip_candidates(ctypes.byref(cfg), ctypes.byref(L), int(t), _p(w), _p(idx), float(kappa),
                                  float(min_change), max_c, _p(meta), _p(delta))
    if n < 0:
        raise RuntimeError(f"oracle flip candidates failed with status {-n}")
    k = min(n, max_c)
    return Flips(meta[:k].copy(), delta[:k].copy(), n)
