"""Argument checks of the C-ABI on the host, without a GPU.

Every call here is rejected by the checks include/moe_v41.h states before any
CUDA call is made, so the addresses passed are fake and never dereferenced:
A is 256-byte aligned, A + 4 only 4-byte aligned."""
import ctypes
import glob
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
A = 1 << 20


@pytest.fixture(scope="module")
def Q():
    import quantized_mixture_experts_router_gb300 as Q
    import quantized_mixture_experts_router_gb300.build as qb
    srcs = glob.glob(os.path.join(ROOT, "quantized_mixture_experts_router_gb300", "csrc", "*"))
    srcs += glob.glob(os.path.join(ROOT, "include", "*.h"))
    if not os.path.exists(Q.SO) or max(os.path.getmtime(f) for f in srcs) > os.path.getmtime(Q.SO):
        qb.build()
    return Q


def _cfg(Q, **kw):
    base = dict(dim=512, inter=256, n_routed=16, topk=2, max_tokens=8)
    base.update(kw)
    return Q.make_cfg(base.pop("dim"), base.pop("inter"), base.pop("n_routed"), base.pop("topk"), **base)


def _forward(Q, cfg, **kw):
    a = dict(x=A, m=1, router_w=A, bias=A, ep=A, shared=0, sh1=A, sh3=A, sh2=A, out=A, tw=A, ti=A, lg=None, ws=A,
             ws_bytes=1 << 40)
    a.update(kw)
    return Q.lib().moe_v41_forward(ctypes.byref(cfg), a["x"], a["m"], a["router_w"], a["bias"], a["ep"], a["shared"],
                                   a["sh1"], a["sh3"], a["sh2"], a["out"], a["tw"], a["ti"], a["lg"], a["ws"],
                                   a["ws_bytes"], None)


def test_forward_rejects_a_bad_configuration(Q):
    for bad in (dict(dim=300), dict(dim=7936), dict(inter=128), dict(topk=0), dict(topk=17), dict(n_routed=1025),
                dict(gate_temp=0.0), dict(gate_temp=float("nan")), dict(max_tokens=0), dict(path=3),
                dict(score_func=3)):
        assert _forward(Q, _cfg(Q, **bad)) == Q.MOE_ERR_ARG, bad


def test_forward_rejects_missing_or_out_of_range_arguments(Q):
    cfg = _cfg(Q)
    for name in ("x", "router_w", "bias", "ep", "sh1", "sh3", "sh2", "out", "tw", "ti"):
        assert _forward(Q, cfg, **{name: None}) == Q.MOE_ERR_ARG, name
    assert _forward(Q, cfg, m=0) == Q.MOE_ERR_ARG
    assert _forward(Q, cfg, m=9) == Q.MOE_ERR_ARG          # above max_tokens
    assert _forward(Q, cfg, shared=2) == Q.MOE_ERR_ARG


def test_forward_rejects_misaligned_pointers(Q):
    cfg = _cfg(Q)
    for name, off in (("x", 8), ("router_w", 8), ("ep", 4), ("sh1", 128), ("sh3", 16), ("sh2", 64)):
        assert _forward(Q, cfg, **{name: A + off}) == Q.MOE_ERR_ALIGN, name


def test_forward_checks_the_workspace(Q):
    cfg = _cfg(Q)
    need = Q.moe_v41_workspace_bytes(cfg)
    assert need > 0
    assert _forward(Q, cfg, ws=None) == Q.MOE_ERR_WORKSPACE
    assert _forward(Q, cfg, ws=A + 128) == Q.MOE_ERR_ALIGN
    assert _forward(Q, cfg, ws_bytes=need - 1) == Q.MOE_ERR_WORKSPACE


def test_out_needs_no_more_than_f32_alignment(Q):
    # out, topk_w and topk_idx are not alignment-checked: a bad configuration
    # is still the first error reported with them one float off
    assert _forward(Q, _cfg(Q, dim=300), out=A + 4, tw=A + 4, ti=A + 4) == Q.MOE_ERR_ARG
    assert _forward(Q, _cfg(Q), out=A + 4, ws=None) == Q.MOE_ERR_WORKSPACE


def test_error_strings(Q):
    for code in (Q.MOE_ERR_ARG, Q.MOE_ERR_ALIGN, Q.MOE_ERR_WORKSPACE, Q.MOE_ERR_CUDA):
        assert Q.strerror(code) and Q.strerror(code) != Q.strerror(Q.MOE_OK)


def _noalloc(Q, cfg, **kw):
    a = dict(x=A, m=1, router_w=A, bias=A, ep=A, shared=0, sh1=A, sh3=A, sh2=A, out=A, tw=A, ti=A, lg=None, st=None)
    a.update(kw)
    return Q.lib().moe_v41_forward_noalloc(ctypes.byref(cfg), a["x"], a["m"], a["router_w"], a["bias"], a["ep"],
                                           a["shared"], a["sh1"], a["sh3"], a["sh2"], a["out"], a["tw"], a["ti"],
                                           a["lg"], a["st"], None)


def test_noalloc_rejects_what_the_plain_forward_rejects(Q):
    """The allocation-free forward checks the configuration exactly like
    moe_v41_forward, plus its own limits (decode kernels only: at most eight
    tokens, never the prefill path), before any CUDA call."""
    for bad in (dict(dim=300), dict(topk=0), dict(n_routed=1025), dict(gate_temp=0.0), dict(max_tokens=0),
                dict(path=3), dict(path=-1), dict(score_func=3)):
        assert _noalloc(Q, _cfg(Q, **bad)) == Q.MOE_ERR_ARG, bad
        assert _forward(Q, _cfg(Q, **bad)) == Q.MOE_ERR_ARG, bad
    assert _noalloc(Q, _cfg(Q, max_tokens=9)) == Q.MOE_ERR_ARG
    assert _noalloc(Q, _cfg(Q, path=Q.MOE_PATH_PREFILL)) == Q.MOE_ERR_ARG
    cfg = _cfg(Q, max_tokens=4)
    assert _noalloc(Q, cfg, m=0) == Q.MOE_ERR_ARG
    assert _noalloc(Q, cfg, m=5) == Q.MOE_ERR_ARG
    for name in ("x", "router_w", "bias", "ep", "sh1", "sh3", "sh2", "out", "tw", "ti"):
        assert _noalloc(Q, cfg, **{name: None}) == Q.MOE_ERR_ARG, name
    assert _noalloc(Q, cfg, shared=2) == Q.MOE_ERR_ARG
    for name, off in (("x", 8), ("router_w", 8), ("ep", 4), ("sh1", 128)):
        assert _noalloc(Q, cfg, **{name: A + off}) == Q.MOE_ERR_ALIGN, name


def test_noalloc_scratch_figure_of_the_header(Q):
    """include/moe_v41.h states the scratch the DeepSeek-V4.1 shape needs at
    eight tokens; it must fit the fixed array, and a shape that needs more is
    refused before any CUDA call."""
    ds = _cfg(Q, dim=5120, inter=2304, n_routed=384, topk=6, max_tokens=8)
    assert Q.moe_v41_workspace_bytes(ds) == 381952 <= Q.NOALLOC_SCRATCH_BYTES
    big = _cfg(Q, dim=5120, inter=2560, n_routed=1024, topk=16, max_tokens=8)
    assert Q.moe_v41_workspace_bytes(big) > Q.NOALLOC_SCRATCH_BYTES
    assert _noalloc(Q, big) == Q.MOE_ERR_WORKSPACE
