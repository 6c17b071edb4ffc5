"""moe_v41_forward_noalloc: the forward for callers that cannot hand the
library any device memory when they call (a plugin inside an engine that
owns the whole GPU memory pool, a loop that must not call cudaMalloc).  Its
scratch is a fixed array the library keeps on each GPU.  It runs the same
deterministic decode kernel as moe_v41_forward, so its results must equal
that call's bit for bit on the same inputs, call after call, and stay within
the parity bars of the oracle.

This file is collected last on purpose, and must pass both on its own in a
fresh process and after every other test."""
import numpy as np
import pytest

import synth.workloads as W
from _helpers import assert_close, assert_output, gpu_forward, lib_cfg, oracle_for

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import quantized_mixture_experts_router_gb300 as Q  # noqa: E402
from synth.device import stage_layer  # noqa: E402


def _noalloc(dl, cfg, m):
    w = dl.w
    out = torch.empty((m, w.dim), dtype=torch.float32, device="cuda")
    tw = torch.empty((m, w.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((m, w.topk), dtype=torch.int32, device="cuda")
    lg = torch.empty((m, w.n_routed), dtype=torch.float32, device="cuda")
    st = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    Q.moe_v41_forward_noalloc(cfg, dl.x, m, dl.router_w, dl.bias, dl.expert_ptrs, w.shared_kind, dl.sh1, dl.sh3,
                              dl.sh2, out, tw, ti, lg, st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), tw.cpu().numpy(), ti.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("name,m", [("tiny", 4), ("decode_m1_40layer", 1), ("decode_m8_kquant_shared", 8)])
def test_noalloc_matches_workspace_forward_twice(name, m):
    w = W.WORKLOADS[name].with_(m=m)
    dl = stage_layer(w, 0, experts_on_gpu=True)
    ref = gpu_forward(dl)
    cfg = lib_cfg(w, max_tokens=m)
    for _ in range(2):
        out, tw, ti, status = _noalloc(dl, cfg, m)
        assert status == 0
        np.testing.assert_array_equal(ti, ref["topk_idx"])
        np.testing.assert_array_equal(tw.view(np.int32), ref["topk_w"].view(np.int32))
        np.testing.assert_array_equal(out.view(np.int32), ref["out"].view(np.int32))
    # and the oracle, on the same logits
    r = oracle_for(w, 0, given_logits=ref["logits"], picked=np.unique(ti))
    np.testing.assert_array_equal(ti, r.topk_idx)
    assert_close(tw, r.topk_w, "routing weights")
    assert_output(out, r)


def test_noalloc_rejects_what_does_not_fit():
    w = W.WORKLOADS["tiny"]
    dl = stage_layer(w, 0, experts_on_gpu=True)
    big = Q.make_cfg(5120, 2560, 1024, 16, max_tokens=8)  # needs ~700 KB of scratch
    assert Q.moe_v41_workspace_bytes(big) > Q.NOALLOC_SCRATCH_BYTES
    out = torch.empty((8, 5120), device="cuda")
    tw = torch.empty((8, 16), device="cuda")
    ti = torch.empty((8, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(Q.MoeError) as e:
        Q.moe_v41_forward_noalloc(big, dl.x, 1, dl.router_w, dl.bias, dl.expert_ptrs, 0, dl.sh1, dl.sh3, dl.sh2,
                                  out, tw, ti)
    assert e.value.code == Q.MOE_ERR_WORKSPACE
    with pytest.raises(Q.MoeError) as e:  # more than eight tokens: the decode kernels only
        Q.moe_v41_forward_noalloc(lib_cfg(w, max_tokens=9), dl.x, 9, dl.router_w, dl.bias, dl.expert_ptrs, 0,
                                  dl.sh1, dl.sh3, dl.sh2, out, tw, ti)
    assert e.value.code == Q.MOE_ERR_ARG
