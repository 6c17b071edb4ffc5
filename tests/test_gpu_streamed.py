"""GPU tests of the expert cache and the streamed forward
(include/moe_v41_cache.h), through the C-ABI.

The streamed forward runs the same kernels as the resident forward on the
same bytes (copied from a page-locked host arena into HBM slots), so its
outputs must equal the resident forward's bit for bit; its cache counters
must equal an independent model of the replacement policy fed with the
same picks; and every streamed output is checked against the oracle on the
same inputs.  The router of moe_v41_route and the fused decode kernel's
router share one accumulation order: their logits are compared bit for bit."""
import numpy as np
import pytest

import oracle
import synth.workloads as W
from _helpers import assert_close, assert_output, lib_cfg, oracle_run
from test_cache_policy import ModelLRU

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import quantized_mixture_experts_router_gb300 as Q  # noqa: E402
from synth.device import fill_experts_host, slot_layout, stage_layer  # noqa: E402


def _ws(cfg):
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    Q.moe_v41_workspace_init(ws)
    return ws


@pytest.mark.parametrize("name,m", [("tiny", 1), ("tiny", 8), ("decode_m1_40layer", 1), ("decode_m1_40layer", 5),
                                    ("decode_m1_40layer", 8)])
def test_route_logits_equal_the_forward_router_bitwise(name, m):
    w = W.WORKLOADS[name].with_(m=m)
    dl = stage_layer(w, 0, slots=min(16, w.n_routed), bulk_on_gpu=True)
    cfg = lib_cfg(w, path=Q.MOE_PATH_DECODE)
    ws = _ws(cfg)
    lg_r = torch.empty((m, w.n_routed), dtype=torch.float32, device="cuda")
    lg_f = torch.empty_like(lg_r)
    tw = torch.empty((m, w.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((m, w.topk), dtype=torch.int32, device="cuda")
    tw2, ti2 = torch.empty_like(tw), torch.empty_like(ti)
    out = torch.empty((m, w.dim), dtype=torch.float32, device="cuda")
    Q.moe_v41_route(cfg, dl.x, m, dl.router_w, dl.bias, lg_r, tw, ti, ws)
    Q.moe_v41_forward(cfg, dl.x, m, dl.router_w, dl.bias, dl.expert_ptrs, w.shared_kind, dl.sh1, dl.sh3, dl.sh2, out,
                      tw2, ti2, lg_f, ws)
    assert Q.moe_v41_read_status(ws, clear=True) == 0
    assert torch.equal(lg_r.view(torch.int32), lg_f.view(torch.int32))
    assert torch.equal(ti, ti2)
    assert torch.equal(tw.view(torch.int32), tw2.view(torch.int32))


class Arena:
    """A workload's layers: resident copies (the reference) and a page-locked
    host arena with the same expert bytes, plus HBM slots and tables."""

    def __init__(self, w, layers, n_slots):
        self.w = w
        self.layers = [stage_layer(w, l, experts_on_gpu=False) for l in range(layers)]
        o1, o3, o2, slot = slot_layout(w)
        self.arena = torch.empty((layers, w.n_routed, slot), dtype=torch.uint8, pin_memory=True)
        for l in range(layers):
            fill_experts_host(w, l, self.arena[l])
        self.slots = torch.empty((n_slots, slot), dtype=torch.uint8, device="cuda")
        self.tables = torch.empty((layers, w.n_routed, 3), dtype=torch.int64, device="cuda")
        self.cache = Q.ExpertCache(layers, w.n_routed, n_slots, slot, o1, o3, o2, self.arena, self.slots,
                                   self.tables)
        self.copy_stream = torch.cuda.Stream()


def _resident(cfg, dl, x, m, logits=None):
    w = dl.w
    ws = _ws(cfg)
    out = torch.empty((m, w.dim), dtype=torch.float32, device="cuda")
    tw = torch.empty((m, w.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((m, w.topk), dtype=torch.int32, device="cuda")
    Q.moe_v41_forward(cfg, x, m, dl.router_w, dl.bias, dl.expert_ptrs, w.shared_kind, dl.sh1, dl.sh3, dl.sh2, out,
                      tw, ti, logits, ws)
    assert Q.moe_v41_read_status(ws, clear=True) == 0
    return out, tw, ti


def _oracle_check(w, layer, x_host, logits, out, tw, ti):
    """The streamed call against the oracle: the layer's own seeded router,
    bias, experts and shared expert, the step's x, the call's logits."""
    experts = [W.expert_blocks(w, layer, e) for e in range(w.n_routed)]
    r = oracle_run(oracle.cfg_of(w), x_host, W.router_bf16(w, layer), W.bias_f32(w, layer), experts,
                   w.shared_kind, W.shared_weights(w, layer), given_logits=logits)
    np.testing.assert_array_equal(ti, r.topk_idx)
    assert_close(tw, r.topk_w, "routing weights")
    assert_output(out, r)


@pytest.mark.parametrize("m,prefetch_k,n_slots", [(1, 0, 2), (1, 2, 4), (1, 2, 9), (3, 0, 7), (20, 0, 16)])
def test_streamed_forward_equals_resident(m, prefetch_k, n_slots):
    """Tokens stepped through 5 layers with the experts streamed through few
    slots (many evictions); every layer of a token takes the same x, so the
    next layer's prediction is its true routing and every prefetch is used."""
    layers, steps = 5, 4
    w = W.WORKLOADS["tiny"].with_(m=m)
    A = Arena(w, layers, n_slots)
    cfg = lib_cfg(w)
    ws = _ws(cfg)
    model = ModelLRU(n_slots, slot_layout(w)[3])
    P = prefetch_k
    host = torch.empty(m * w.topk + P, dtype=torch.int32, pin_memory=True)
    stream = torch.cuda.current_stream()
    xs = [stage_layer(w.with_(seed=w.seed + 100 + s), 0, experts_on_gpu=False).x for s in range(steps)]
    xs_host = [W.x_bf16(w.with_(seed=w.seed + 100 + s), 0) for s in range(steps)]
    lg = torch.empty((m, w.n_routed), dtype=torch.float32, device="cuda")
    for s in range(steps):
        x = xs[s]
        for l in range(layers):
            dl = A.layers[l]
            nxt = A.layers[l + 1] if l + 1 < layers else None
            out = torch.empty((m, w.dim), dtype=torch.float32, device="cuda")
            tw = torch.empty((m, w.topk), dtype=torch.float32, device="cuda")
            ti = torch.empty((m, w.topk), dtype=torch.int32, device="cuda")
            Q.moe_v41_forward_streamed(cfg, A.cache, l, x, m, dl.router_w, dl.bias,
                                       None if nxt is None else nxt.router_w, None if nxt is None else nxt.bias, P,
                                       w.shared_kind, dl.sh1, dl.sh3, dl.sh2, out, tw, ti, ws, host, stream,
                                       A.copy_stream)
            assert Q.moe_v41_read_status(ws, clear=True) == 0
            ro, rw, ri = _resident(cfg, dl, x, m, logits=lg)
            assert torch.equal(ti, ri)
            assert torch.equal(tw.view(torch.int32), rw.view(torch.int32))
            assert torch.equal(out.view(torch.int32), ro.view(torch.int32)), f"step {s} layer {l}"
            _oracle_check(w, l, xs_host[s], lg.cpu().numpy(), out.cpu().numpy(), tw.cpu().numpy(),
                          ti.cpu().numpy())
            picks = ti.cpu().numpy().reshape(-1)
            model.fetch(l, picks)
            if P and m == 1 and nxt is not None:
                pred = host.numpy()[m * w.topk:m * w.topk + P]
                _, _, ri_next = _resident(cfg, nxt, x, m)
                assert sorted(pred.tolist()) == sorted(ri_next.cpu().numpy().reshape(-1)[:P].tolist()) or P != w.topk
                model.fetch(l + 1, pred, prefetch=True)
    torch.cuda.synchronize()
    st = A.cache.stats()
    assert st == model.st
    if P:
        assert st["prefetch_hits"] > 0
    assert st["evictions"] > 0 or n_slots >= layers * w.n_routed


def test_unfetched_expert_is_reported_missing():
    w = W.WORKLOADS["tiny"].with_(m=1)
    A = Arena(w, 2, 4)
    cfg = lib_cfg(w)
    ws = _ws(cfg)
    dl = A.layers[0]
    out = torch.empty((1, w.dim), dtype=torch.float32, device="cuda")
    tw = torch.empty((1, w.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((1, w.topk), dtype=torch.int32, device="cuda")
    Q.moe_v41_forward(cfg, dl.x, 1, dl.router_w, dl.bias, A.cache.table(0), w.shared_kind, dl.sh1, dl.sh3, dl.sh2,
                      out, tw, ti, None, ws)
    assert Q.moe_v41_read_status(ws, clear=True) & Q.MOE_STATUS_MISSING_EXPERT
    # fetched by hand, the same call is complete and equals the resident one
    A.cache.fetch(0, ti.cpu().numpy().reshape(-1), copy_stream=A.copy_stream)
    A.cache.wait(0)
    Q.moe_v41_forward(cfg, dl.x, 1, dl.router_w, dl.bias, A.cache.table(0), w.shared_kind, dl.sh1, dl.sh3, dl.sh2,
                      out, tw, ti, None, ws)
    A.cache.reads(0, ti.cpu().numpy().reshape(-1))
    assert Q.moe_v41_read_status(ws, clear=True) == 0
    ro, _, _ = _resident(cfg, dl, dl.x, 1)
    assert torch.equal(out.view(torch.int32), ro.view(torch.int32))
