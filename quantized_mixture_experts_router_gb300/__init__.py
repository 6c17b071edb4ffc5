"""Python binding of libmoe_v41 (include/moe_v41.h): argument marshalling only.

Every step of the MoE layer runs in the library's sm_103a kernels; this
module converts torch tensors (device memory) and streams into the C-ABI's
plain pointers and raises on a non-zero return code.  There is no fallback:
if the compiled library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(_HERE, "_lib", "libmoe_v41.so")

MOE_PATH_AUTO, MOE_PATH_DECODE, MOE_PATH_PREFILL = 0, 1, 2
MOE_SCORE_SQRTSOFTPLUS, MOE_SCORE_SIGMOID, MOE_SCORE_SOFTMAX = 0, 1, 2
MOE_SHARED_BF16, MOE_SHARED_KQUANT = 0, 1
MOE_OK, MOE_ERR_ARG, MOE_ERR_ALIGN, MOE_ERR_WORKSPACE, MOE_ERR_CUDA = 0, 1, 2, 3, 4
MOE_STATUS_NAN_KEY, MOE_STATUS_MISSING_EXPERT, MOE_STATUS_TIMEOUT = 1, 2, 4


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: moe_v41 error {code} ({strerror(code)})")
        self.code = code


class moe_v41_cfg(ctypes.Structure):
    _fields_ = [("dim", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_routed", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("gate_temp", ctypes.c_float), ("norm_topk_prob", ctypes.c_int32),
                ("route_scale", ctypes.c_float), ("swiglu_limit", ctypes.c_float), ("max_tokens", ctypes.c_int32),
                ("path", ctypes.c_int32), ("wait_timeout_us", ctypes.c_uint32), ("score_func", ctypes.c_int32)]


class moe_v41_cache_cfg(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_routed", ctypes.c_int32), ("n_slots", ctypes.c_int32),
                ("slot_bytes", ctypes.c_uint64), ("off_w1", ctypes.c_uint64), ("off_w3", ctypes.c_uint64),
                ("off_w2", ctypes.c_uint64), ("arena", ctypes.c_void_p), ("slots", ctypes.c_void_p),
                ("tables", ctypes.c_void_p)]


class moe_v41_cache_stats(ctypes.Structure):
    _fields_ = [("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64), ("evictions", ctypes.c_uint64),
                ("bytes_copied", ctypes.c_uint64), ("prefetched", ctypes.c_uint64),
                ("prefetch_hits", ctypes.c_uint64)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(SO):
            raise RuntimeError(f"{SO} is missing: the CUDA library must be built (__graft_entry__.build())")
        L = ctypes.CDLL(SO)
        vp, i32, sz, cfgp = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(moe_v41_cfg)
        L.moe_v41_workspace_bytes.restype = sz
        L.moe_v41_workspace_bytes.argtypes = [cfgp]
        L.moe_v41_workspace_init.argtypes = [vp, sz, vp]
        L.moe_v41_quantize_q8_1.argtypes = [vp, i32, i32, i32, vp, vp]
        L.moe_v41_select_from_logits.argtypes = [cfgp, vp, i32, vp, vp, vp, vp, sz, vp]
        L.moe_v41_route.argtypes = [cfgp, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_v41_forward.argtypes = [cfgp, vp, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_v41_select_from_logits_vl.argtypes = [cfgp, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_v41_route_vl.argtypes = [cfgp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_v41_forward_vl.argtypes = [cfgp, vp, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                         vp]
        L.moe_v41_read_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32), i32]
        L.moe_v41_forward_noalloc.argtypes = [cfgp, vp, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.moe_v41_kernel_launches.argtypes = [cfgp, i32, i32]
        L.moe_v41_kernel_launches.restype = i32
        L.moe_v41_strerror.restype = ctypes.c_char_p
        L.moe_v41_strerror.argtypes = [i32]
        cp = ctypes.c_void_p
        L.moe_v41_cache_create.argtypes = [ctypes.POINTER(moe_v41_cache_cfg), vp, ctypes.POINTER(cp)]
        L.moe_v41_cache_destroy.argtypes = [cp]
        L.moe_v41_cache_fetch.argtypes = [cp, i32, vp, i32, i32, vp]
        L.moe_v41_cache_wait.argtypes = [cp, i32, vp]
        L.moe_v41_cache_reads.argtypes = [cp, i32, vp, i32, vp]
        L.moe_v41_cache_slot_of.argtypes = [cp, i32, i32]
        L.moe_v41_cache_get_stats.argtypes = [cp, ctypes.POINTER(moe_v41_cache_stats)]
        L.moe_v41_forward_streamed.argtypes = [cfgp, cp, i32, vp, i32, vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp,
                                               vp, vp, sz, vp, vp, vp]
        for f in ("moe_v41_workspace_init", "moe_v41_quantize_q8_1", "moe_v41_select_from_logits", "moe_v41_route",
                  "moe_v41_forward", "moe_v41_read_status", "moe_v41_forward_noalloc",
                  "moe_v41_select_from_logits_vl", "moe_v41_route_vl", "moe_v41_forward_vl", "moe_v41_cache_create",
                  "moe_v41_cache_destroy", "moe_v41_cache_fetch", "moe_v41_cache_wait", "moe_v41_cache_reads",
                  "moe_v41_cache_slot_of", "moe_v41_cache_get_stats", "moe_v41_forward_streamed"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().moe_v41_strerror(code).decode()


def _p(t):
    """device address of a tensor, or an int address, or None"""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(t):
    return t.numel() * t.element_size()


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def make_cfg(dim, inter, n_routed, topk, gate_temp=1.0, norm_topk_prob=True, route_scale=1.5, swiglu_limit=10.0,
             max_tokens=1, path=MOE_PATH_AUTO, wait_timeout_us=0, score_func=MOE_SCORE_SQRTSOFTPLUS) -> moe_v41_cfg:
    return moe_v41_cfg(dim, inter, n_routed, topk, gate_temp, int(bool(norm_topk_prob)), route_scale, swiglu_limit,
                       max_tokens, path, wait_timeout_us, score_func)


def moe_v41_workspace_bytes(cfg: moe_v41_cfg) -> int:
    return int(lib().moe_v41_workspace_bytes(ctypes.byref(cfg)))


def moe_v41_workspace_init(ws, stream=None):
    _check(lib().moe_v41_workspace_init(_p(ws), _nbytes(ws), _s(stream)), "moe_v41_workspace_init")


def moe_v41_quantize_q8_1(x, x_is_f32: bool, rows: int, cols: int, q8_out, stream=None):
    _check(lib().moe_v41_quantize_q8_1(_p(x), int(x_is_f32), rows, cols, _p(q8_out), _s(stream)),
           "moe_v41_quantize_q8_1")


def moe_v41_select_from_logits(cfg, logits, m, bias, topk_w, topk_idx, ws, stream=None):
    _check(lib().moe_v41_select_from_logits(ctypes.byref(cfg), _p(logits), m, _p(bias), _p(topk_w), _p(topk_idx),
                                            _p(ws), _nbytes(ws), _s(stream)), "moe_v41_select_from_logits")


def moe_v41_select_from_logits_vl(cfg, logits, m, bias, bias_vl, image_mask, topk_w, topk_idx, ws, stream=None):
    _check(lib().moe_v41_select_from_logits_vl(ctypes.byref(cfg), _p(logits), m, _p(bias), _p(bias_vl),
                                               _p(image_mask), _p(topk_w), _p(topk_idx), _p(ws), _nbytes(ws),
                                               _s(stream)), "moe_v41_select_from_logits_vl")


def moe_v41_route_vl(cfg, x, m, router_w, bias, bias_vl, image_mask, logits_out, topk_w, topk_idx, ws, stream=None):
    _check(lib().moe_v41_route_vl(ctypes.byref(cfg), _p(x), m, _p(router_w), _p(bias), _p(bias_vl), _p(image_mask),
                                  _p(logits_out), _p(topk_w), _p(topk_idx), _p(ws), _nbytes(ws), _s(stream)),
           "moe_v41_route_vl")


def moe_v41_route(cfg, x, m, router_w, bias, logits_out, topk_w, topk_idx, ws, stream=None):
    _check(lib().moe_v41_route(ctypes.byref(cfg), _p(x), m, _p(router_w), _p(bias), _p(logits_out), _p(topk_w),
                               _p(topk_idx), _p(ws), _nbytes(ws), _s(stream)), "moe_v41_route")


def moe_v41_forward(cfg, x, m, router_w, bias, expert_ptrs, shared_kind, sh_w1, sh_w3, sh_w2, out, topk_w, topk_idx,
                    logits_out, ws, stream=None):
    _check(lib().moe_v41_forward(ctypes.byref(cfg), _p(x), m, _p(router_w), _p(bias), _p(expert_ptrs), shared_kind,
                                 _p(sh_w1), _p(sh_w3), _p(sh_w2), _p(out), _p(topk_w), _p(topk_idx), _p(logits_out),
                                 _p(ws), _nbytes(ws), _s(stream)), "moe_v41_forward")


def moe_v41_forward_vl(cfg, x, m, router_w, bias, bias_vl, image_mask, expert_ptrs, shared_kind, sh_w1, sh_w3, sh_w2,
                       out, topk_w, topk_idx, logits_out, ws, stream=None):
    _check(lib().moe_v41_forward_vl(ctypes.byref(cfg), _p(x), m, _p(router_w), _p(bias), _p(bias_vl), _p(image_mask),
                                    _p(expert_ptrs), shared_kind, _p(sh_w1), _p(sh_w3), _p(sh_w2), _p(out),
                                    _p(topk_w), _p(topk_idx), _p(logits_out), _p(ws), _nbytes(ws), _s(stream)),
           "moe_v41_forward_vl")


NOALLOC_SCRATCH_BYTES = 512 << 10


def moe_v41_forward_noalloc(cfg, x, m, router_w, bias, expert_ptrs, shared_kind, sh_w1, sh_w3, sh_w2, out, topk_w,
                            topk_idx, logits_out=None, status_out=None, stream=None):
    """moe_v41_forward without a workspace: the library's own fixed scratch
    array (512 KiB per device) is used.  For callers that cannot allocate device
    memory when they call; see include/moe_v41.h for the limits."""
    _check(lib().moe_v41_forward_noalloc(ctypes.byref(cfg), _p(x), m, _p(router_w), _p(bias), _p(expert_ptrs),
                                         shared_kind, _p(sh_w1), _p(sh_w3), _p(sh_w2), _p(out), _p(topk_w),
                                         _p(topk_idx), _p(logits_out), _p(status_out), _s(stream)),
           "moe_v41_forward_noalloc")


def moe_v41_kernel_launches(cfg, m: int, shared_kind: int) -> int:
    return int(lib().moe_v41_kernel_launches(ctypes.byref(cfg), int(m), int(shared_kind)))


def moe_v41_read_status(ws, stream=None, clear: bool = False) -> int:
    v = ctypes.c_uint32(0)
    _check(lib().moe_v41_read_status(_p(ws), _s(stream), ctypes.byref(v), int(clear)), "moe_v41_read_status")
    return v.value


# ------------------------------------------------------------ expert cache

def _ids(experts):
    a = [int(e) for e in experts]
    return (ctypes.c_int32 * max(1, len(a)))(*a), len(a)


class ExpertCache:
    """include/moe_v41_cache.h: routed experts of a host arena held in a
    least-recently-used set of HBM slots, with the per-layer slot pointer
    tables moe_v41_forward reads.  arena: page-locked host tensor (or address)
    of [n_layers, n_routed, slot_bytes]; slots: device [n_slots, slot_bytes];
    tables: device int64 [n_layers, n_routed, 3].  With slots and tables None
    the cache only simulates the replacement policy (no CUDA call)."""

    def __init__(self, n_layers, n_routed, n_slots, slot_bytes, off_w1, off_w3, off_w2, arena=None, slots=None,
                 tables=None, stream=None):
        self.sim = slots is None and tables is None
        self.cfg = moe_v41_cache_cfg(n_layers, n_routed, n_slots, slot_bytes, off_w1, off_w3, off_w2, _p(arena),
                                     _p(slots), _p(tables))
        self._keep = (arena, slots, tables)
        self._h = ctypes.c_void_p()
        _check(lib().moe_v41_cache_create(ctypes.byref(self.cfg), None if self.sim else _s(stream),
                                          ctypes.byref(self._h)), "moe_v41_cache_create")
        self.tables = tables

    def _st(self, stream):
        return None if self.sim else _s(stream)

    def fetch(self, layer, experts, prefetch=False, copy_stream=None):
        a, n = _ids(experts)
        _check(lib().moe_v41_cache_fetch(self._h, layer, a, n, int(bool(prefetch)), self._st(copy_stream)),
               "moe_v41_cache_fetch")

    def wait(self, layer, stream=None):
        _check(lib().moe_v41_cache_wait(self._h, layer, self._st(stream)), "moe_v41_cache_wait")

    def reads(self, layer, experts=None, stream=None):
        if experts is None:
            _check(lib().moe_v41_cache_reads(self._h, layer, None, 0, self._st(stream)), "moe_v41_cache_reads")
        else:
            a, n = _ids(experts)
            _check(lib().moe_v41_cache_reads(self._h, layer, a, n, self._st(stream)), "moe_v41_cache_reads")

    def slot_of(self, layer, expert) -> int:
        return int(lib().moe_v41_cache_slot_of(self._h, layer, expert))

    def stats(self) -> dict:
        st = moe_v41_cache_stats()
        _check(lib().moe_v41_cache_get_stats(self._h, ctypes.byref(st)), "moe_v41_cache_get_stats")
        return {f: int(getattr(st, f)) for f, _ in moe_v41_cache_stats._fields_}

    def table(self, layer):
        """the device slot pointer table of one layer ([n_routed, 3] int64 view)"""
        return self.tables[layer]

    def close(self):
        if self._h:
            lib().moe_v41_cache_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_v41_forward_streamed(cfg, cache: ExpertCache, layer, x, m, router_w, bias, next_router_w, next_bias,
                             prefetch_k, shared_kind, sh_w1, sh_w3, sh_w2, out, topk_w, topk_idx, ws, host_picks,
                             stream=None, copy_stream=None):
    _check(lib().moe_v41_forward_streamed(ctypes.byref(cfg), cache._h, layer, _p(x), m, _p(router_w), _p(bias),
                                          _p(next_router_w), _p(next_bias), prefetch_k, shared_kind, _p(sh_w1),
                                          _p(sh_w3), _p(sh_w2), _p(out), _p(topk_w), _p(topk_idx), _p(ws),
                                          _nbytes(ws), _p(host_picks), _s(stream), _s(copy_stream)),
           "moe_v41_forward_streamed")
