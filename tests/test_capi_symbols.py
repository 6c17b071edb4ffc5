"""The C-ABI library builds for sm_103a, loads without a GPU, and exports
every function include/*.h declares (no compute calls)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_v41_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    import quantized_mixture_experts_router_gb300 as Q
    import quantized_mixture_experts_router_gb300.build as qb
    srcs = glob.glob(os.path.join(ROOT, "quantized_mixture_experts_router_gb300", "csrc", "*"))
    srcs += glob.glob(os.path.join(ROOT, "include", "*.h"))
    if not os.path.exists(Q.SO) or max(os.path.getmtime(f) for f in srcs) > os.path.getmtime(Q.SO):
        qb.build()
    return ctypes.CDLL(Q.SO)


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("moe_v41_route", "moe_v41_forward", "moe_v41_workspace_bytes", "moe_v41_read_status",
              "moe_v41_forward_vl", "moe_v41_route_vl", "moe_v41_select_from_logits_vl"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_workspace_sizing_is_host_only(lib):
    import quantized_mixture_experts_router_gb300 as Q
    cfg = Q.make_cfg(5120, 2304, 384, 6, max_tokens=8)
    n = Q.moe_v41_workspace_bytes(cfg)
    assert n > 0 and n % 256 == 0
    assert Q.moe_v41_workspace_bytes(Q.make_cfg(5000, 2304, 384, 6)) == 0      # dim not a multiple of 256
    assert Q.moe_v41_workspace_bytes(Q.make_cfg(5120, 2304, 384, 17)) == 0     # topk above 16
    assert Q.moe_v41_workspace_bytes(Q.make_cfg(5120, 2304, 4, 6)) == 0        # topk above n_routed
    assert Q.moe_v41_workspace_bytes(Q.make_cfg(5120, 2304, 384, 6, gate_temp=0.0)) == 0
    for sf in (Q.MOE_SCORE_SIGMOID, Q.MOE_SCORE_SOFTMAX):                     # the Gate's other score functions
        assert Q.moe_v41_workspace_bytes(Q.make_cfg(5120, 2304, 384, 6, max_tokens=8, score_func=sf)) == n
    assert Q.moe_v41_workspace_bytes(Q.make_cfg(5120, 2304, 384, 6, score_func=3)) == 0
    assert Q.moe_v41_workspace_bytes(Q.make_cfg(5120, 2304, 384, 6, score_func=-1)) == 0
    assert Q.strerror(Q.MOE_ERR_WORKSPACE).startswith("workspace")


def test_workspace_holds_prefill_buffers_only_when_prefill_can_run(lib):
    import quantized_mixture_experts_router_gb300 as Q
    dec = Q.moe_v41_workspace_bytes(Q.make_cfg(5120, 2304, 384, 6, max_tokens=8))
    auto = Q.moe_v41_workspace_bytes(Q.make_cfg(5120, 2304, 384, 6, max_tokens=4096))
    pre8 = Q.moe_v41_workspace_bytes(Q.make_cfg(5120, 2304, 384, 6, max_tokens=8, path=Q.MOE_PATH_PREFILL))
    # 4096 tokens: at least the fp16 high/low activations, h and the per-pair expert outputs
    assert auto > 4096 * 5120 * 4 + 4096 * 7 * (2304 * 2 + 5120 * 4)
    assert pre8 > dec


def test_kernel_launch_counts(lib):
    import quantized_mixture_experts_router_gb300 as Q
    auto = Q.make_cfg(5120, 2304, 384, 6, max_tokens=4096)
    assert Q.moe_v41_kernel_launches(auto, 1, Q.MOE_SHARED_BF16) == 1       # one persistent decode kernel
    assert Q.moe_v41_kernel_launches(auto, 8, Q.MOE_SHARED_KQUANT) == 1
    assert Q.moe_v41_kernel_launches(auto, 9, Q.MOE_SHARED_BF16) == 11      # prefill, bf16 shared expert
    assert Q.moe_v41_kernel_launches(auto, 4096, Q.MOE_SHARED_KQUANT) == 9  # shared expert as one more expert
    assert Q.moe_v41_kernel_launches(auto, 4097, Q.MOE_SHARED_BF16) == -1
    dec = Q.make_cfg(5120, 2304, 384, 6, max_tokens=16, path=Q.MOE_PATH_DECODE)
    assert Q.moe_v41_kernel_launches(dec, 9, Q.MOE_SHARED_BF16) == -1
    # widths one decode stage does not hold: AUTO runs even a single token on the prefill kernels, and the
    # workspace of such a configuration holds the prefill buffers although max_tokens <= 8
    wide = Q.make_cfg(7680, 4096, 384, 6, max_tokens=1)
    assert Q.moe_v41_kernel_launches(wide, 1, Q.MOE_SHARED_BF16) == 11
    assert Q.moe_v41_workspace_bytes(wide) > Q.moe_v41_workspace_bytes(Q.make_cfg(5120, 2304, 384, 6, max_tokens=1))
    wide_dec = Q.make_cfg(7680, 4096, 384, 6, max_tokens=1, path=Q.MOE_PATH_DECODE)
    assert Q.moe_v41_kernel_launches(wide_dec, 1, Q.MOE_SHARED_BF16) == -1  # the forward refuses it too
