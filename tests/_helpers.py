"""Shared helpers of the parity tests: run the CUDA path through the C-ABI,
run the oracle on the same seeded inputs, compare at the stated tolerances."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from types import SimpleNamespace

import numpy as np

import oracle
import synth.workloads as W

# tolerances: relative L2 of the whole compared output, and the largest
# element error relative to the oracle output's RMS
REL_L2 = 2e-3
MAX_ABS_REL = 1e-2

# Layer outputs: the largest element error relative to the oracle output's
# RMS once the requantisation flips of h are accounted for (reading C-F1 of
# the oracle: a q8_1 code, q8_1 block scale or bf16 value of h whose exact
# value lies within the f32 accumulation error of g and u of a rounding
# boundary may come out either way).  FLIP_KAPPA bounds that error relative
# to sum |terms| of the dot products: about 2^-24 sqrt(K) for K ~ 5000 terms
# in f32 with random rounding errors.  Tokens whose error passes
# FLIP_LOOK x the bar are looked at, with the candidates that move some
# output element by FLIP_MIN x the bar or more (smaller ones cannot take an
# element past it); a candidate counts as taken when the token's remaining
# error projects onto its output change by FLIP_TAKE[0] to FLIP_TAKE[1] times
# its own squared length (a flip's change is a W2 column, and the changes of
# different h elements are nearly orthogonal).
OUT_MAX_ABS_REL = 2e-3
FLIP_KAPPA = 2.0 ** -18
FLIP_LOOK = 0.5
FLIP_MIN = 0.1
FLIP_TAKE = (0.75, 1.5)
FLIP_MAX = 2048


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


def oracle_run(cfg, x, R, b, experts, shared_kind, sh, tokens=None, given_logits=None, bias_vl=None,
               image_mask=None):
    """oracle.moe_layer, its result carrying what assert_output needs to
    look for requantisation flips (the inputs and the rows' token ids)."""
    r = oracle.moe_layer(cfg, x, R, b, experts, shared_kind, *sh, tokens=tokens, given_logits=given_logits,
                         bias_vl=bias_vl, image_mask=image_mask)
    ids = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    r.inputs = SimpleNamespace(cfg=cfg, x=x, experts=experts, shared_kind=shared_kind, sh=sh, token_ids=ids)
    return r


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
    return oracle_run(oracle.cfg_of(w), x, R, b, experts, w.shared_kind, sh, tokens=tokens,
                      given_logits=given_logits, bias_vl=bv, image_mask=im)


def take_flips(resid: np.ndarray, delta: np.ndarray, take=FLIP_TAKE):
    """Greedy choice of requantisation flips explaining a token's error
    `resid` (GPU minus oracle): repeatedly the candidate whose output change
    lowers |resid|^2 the most, among those onto whose change the remaining
    error projects by take[0] to take[1] times its squared length.  Returns
    the remaining error and the indices taken."""
    resid = np.array(resid, dtype=np.float64)
    if len(delta) == 0:
        return resid, []
    nd = np.einsum("ij,ij->i", delta, delta)
    b = delta @ resid
    # a change the error does not line up with cannot be taken (the others'
    # changes are nearly orthogonal to it)
    keep = np.nonzero((nd > 0) & (b > 0.25 * nd))[0]
    if keep.size == 0:
        return resid, []
    D = delta[keep]
    G = D @ D.T
    nd, b = nd[keep], b[keep]
    avail = np.ones(keep.size, dtype=bool)
    used = []
    while True:
        gain = np.where(avail & (b >= take[0] * nd) & (b <= take[1] * nd), 2 * b - nd, -np.inf)
        k = int(np.argmax(gain))
        if not np.isfinite(gain[k]):
            break
        used.append(int(keep[k]))
        avail[k] = False
        resid -= D[k]
        b -= G[:, k]
    return resid, used


def assert_output(got, r, what="output", rows=None):
    """A layer output against the oracle result r (from oracle_run /
    oracle_for), optionally on some of its rows: relative L2 <= REL_L2 as it
    stands, and every element within OUT_MAX_ABS_REL x RMS once the tokens
    past FLIP_LOOK of that bar have had their requantisation flips taken (the
    oracle lists the candidates; a token with more than FLIP_MAX fails).  Returns (rel L2, raw max/RMS, max/RMS after the
    flips, tokens looked at, flips taken)."""
    ref = r.out if rows is None else r.out[rows]
    inp = r.inputs
    ids = inp.token_ids if rows is None else inp.token_ids[rows]
    tw = r.topk_w if rows is None else r.topk_w[rows]
    ti = r.topk_idx if rows is None else r.topk_idx[rows]
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    l2, raw = rel_errors(got, ref)
    assert l2 <= REL_L2, f"{what}: rel L2 {l2:.3e} (<= {REL_L2})"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    resid = got - ref
    todo = np.nonzero(np.abs(resid).max(axis=1) > FLIP_LOOK * OUT_MAX_ABS_REL * rms)[0]

    def one(i):
        F = oracle.flip_candidates(inp.cfg, inp.x, int(ids[i]), tw[i], ti[i], inp.experts, inp.shared_kind, *inp.sh,
                                   FLIP_KAPPA, min_change=FLIP_MIN * OUT_MAX_ABS_REL * rms, max_c=FLIP_MAX)
        assert F.total <= FLIP_MAX, f"{what}: token {ids[i]} has {F.total} flip candidates (> {FLIP_MAX})"
        rest, used = take_flips(resid[i], F.delta)
        return i, rest, len(used)

    n_flips = 0
    if todo.size:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1, todo.size)) as ex:
            for i, rest, n in ex.map(one, todo):
                resid[i] = rest
                n_flips += n
    mx = float(np.abs(resid).max() / rms)
    assert mx <= OUT_MAX_ABS_REL, (f"{what}: max-abs/RMS {mx:.3e} (<= {OUT_MAX_ABS_REL}) after {n_flips} flips "
                                   f"over {todo.size} tokens (raw {raw:.3e})")
    return l2, raw, mx, int(todo.size), n_flips
