"""Shared helpers of the parity tests: run the CUDA path through the C-ABI,
run the oracle on the same seeded inputs, compare at the stated tolerances."""
from __future__ import annotations

import numpy as np

import oracle
import synth.workloads as W

# tolerances: relative L2 of the whole compared output, and the largest
# element error relative to the oracle output's RMS
REL_L2 = 2e-3
MAX_ABS_REL = 1e-2


def rel_errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = got - ref
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.linalg.norm(err) / np.linalg.norm(ref)), float(np.abs(err).max() / rms)


def assert_close(got, ref, what=""):
    l2, mx = rel_errors(got, ref)
    assert l2 <= REL_L2 and mx <= MAX_ABS_REL, f"{what}: rel L2 {l2:.3e} (<= {REL_L2}), max-abs/RMS {mx:.3e} (<= {MAX_ABS_REL})"
    return l2, mx


def lib_cfg(w: W.Workload, max_tokens=None, path=0, timeout_us=0):
    import quantized_mixture_experts_router_gb300 as Q
    return Q.make_cfg(w.dim, w.inter, w.n_routed, w.topk, w.gate_temp, w.norm_topk_prob, w.route_scale,
                      w.swiglu_limit, max_tokens or w.m, path, timeout_us, w.score_func)


def gpu_forward(dl, path=0, m=None, ws=None, cfg=None):
    """One moe_v41_forward through the C-ABI; returns host numpy results."""
    import torch
    import quantized_mixture_experts_router_gb300 as Q
    w = dl.w
    m = m or w.m
    cfg = cfg or lib_cfg(w, max_tokens=max(m, w.m), path=path)
    if ws is None:
        ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
        Q.moe_v41_workspace_init(ws)
    out = torch.empty((m, w.dim), dtype=torch.float32, device="cuda")
    tw = torch.empty((m, w.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((m, w.topk), dtype=torch.int32, device="cuda")
    lg = torch.empty((m, w.n_routed), dtype=torch.float32, device="cuda")
    if dl.image_mask is None:
        Q.moe_v41_forward(cfg, dl.x, m, dl.router_w, dl.bias, dl.expert_ptrs, w.shared_kind, dl.sh1, dl.sh3, dl.sh2,
                          out, tw, ti, lg, ws)
    else:
        Q.moe_v41_forward_vl(cfg, dl.x, m, dl.router_w, dl.bias, dl.bias_vl, dl.image_mask, dl.expert_ptrs,
                             w.shared_kind, dl.sh1, dl.sh3, dl.sh2, out, tw, ti, lg, ws)
    status = Q.moe_v41_read_status(ws, clear=True)
    return dict(out=out.cpu().numpy(), topk_w=tw.cpu().numpy(), topk_idx=ti.cpu().numpy(),
                logits=lg.cpu().numpy(), status=status, ws=ws)


def oracle_for(w: W.Workload, layer: int, given_logits=None, tokens=None, picked=None):
    """The oracle on the workload's seeded inputs.  With `picked` (expert ids)
    only those experts are drawn on the host (the full-size layers hold 384)."""
    x = W.x_bf16(w, layer)
    R = W.router_bf16(w, layer)
    b = W.bias_f32(w, layer)
    need = range(w.n_routed) if picked is None else sorted(set(int(e) for e in picked))
    experts = [None] * w.n_routed
    for e in need:
        experts[e] = W.expert_blocks(w, layer, e)
    sh = W.shared_weights(w, layer)
    im = W.image_mask(w, layer)
    bv = None if im is None else W.bias_vl_f32(w, layer)
    return oracle.moe_layer(oracle.cfg_of(w), x, R, b, experts, w.shared_kind, *sh, tokens=tokens,
                            given_logits=given_logits, bias_vl=bv, image_mask=im)
