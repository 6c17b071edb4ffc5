"""GPU parity of the decode path (m <= 8) against the oracle, through the C-ABI.

Bars: q8_1(x) bit-exact; top-k indices bit-exact on identical f32 logits
(both directions); outputs and routing weights within 2e-3 relative L2 and
max-abs <= 1e-2 x RMS of the oracle output."""
import time

import numpy as np
import pytest

import oracle
import synth
import synth.workloads as W
from _helpers import assert_close, assert_output, gpu_forward, lib_cfg, oracle_for, rel_errors

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import quantized_mixture_experts_router_gb300 as Q  # noqa: E402
from synth.device import stage_layer  # noqa: E402


def _f32_to_bf16_bits(a):
    return np.array([oracle.bf16_from_f32(float(v)) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)


# ------------------------------------------------------------------- q8_1

@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 512), (5, 5120), (64, 2304)])
def test_q8_1_bitexact_f32(rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    x = (rng.standard_normal((rows, cols)) * np.repeat(rng.uniform(1e-3, 80, (rows, cols // 32)), 32, axis=1))
    x = x.astype(np.float32)
    x[0, :32] = 0.0                                   # an all-zero block
    if cols >= 64:
        x[0, 32:64] = np.arange(32, dtype=np.float32) - 15.5  # halfway values after scaling
        x[0, 32] = 127.0
    if rows > 1:
        x[1, :32] = np.float32(2.0 ** -20) * (np.arange(32) - 16)  # fp16-subnormal scale
    q8 = torch.empty(rows * cols // 32 * 36, dtype=torch.uint8, device="cuda")
    Q.moe_v41_quantize_q8_1(torch.from_numpy(x).cuda(), True, rows, cols, q8)
    ref = oracle.quantize_q8_1(x).reshape(-1)
    np.testing.assert_array_equal(q8.cpu().numpy(), ref)


def test_q8_1_bitexact_bf16_with_outliers():
    w = W.WORKLOADS["prefill_m4096_outliers"].with_(m=256)
    x = W.x_bf16(w, 0)  # rows scaled by 50 included
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    q8 = torch.empty(x.shape[0] * x.shape[1] // 32 * 36, dtype=torch.uint8, device="cuda")
    Q.moe_v41_quantize_q8_1(torch.from_numpy(x.view(np.int16)).cuda(), False, x.shape[0], x.shape[1], q8)
    np.testing.assert_array_equal(q8.cpu().numpy(), oracle.quantize_q8_1(xf).reshape(-1))


# -------------------------------------------------------------- selection

def _select_gpu(w, logits, bias):
    cfg = lib_cfg(w, max_tokens=logits.shape[0])
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    Q.moe_v41_workspace_init(ws)
    m = logits.shape[0]
    tw = torch.empty((m, w.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((m, w.topk), dtype=torch.int32, device="cuda")
    Q.moe_v41_select_from_logits(cfg, torch.from_numpy(logits).cuda(), m, torch.from_numpy(bias).cuda(), tw, ti, ws)
    status = Q.moe_v41_read_status(ws, clear=True)
    return tw.cpu().numpy(), ti.cpu().numpy(), status


@pytest.mark.parametrize("name", ["decode_m1_40layer", "prefill_m512_hot", "tiny"])
def test_selection_bitexact(name):
    w = W.WORKLOADS[name]
    rng = np.random.default_rng(11)
    m = 300
    logits = (rng.standard_normal((m, w.n_routed)) * 2).astype(np.float32)
    logits[0] = 25.0                                  # all scores equal: ties by id
    logits[1, ::3] = 40.0                             # above the softplus threshold
    logits[2, :] = logits[2, 0]
    bias = W.bias_f32(w.with_(m=1), 0)
    tw, ti, status = _select_gpu(w, logits, bias)
    rw, ri, _ = oracle.route_from_logits(oracle.cfg_of(w), logits, bias)
    np.testing.assert_array_equal(ti, ri)
    np.testing.assert_allclose(tw, rw, rtol=2e-6, atol=0)
    assert status == 0


def test_selection_config_variants():
    base = W.WORKLOADS["prefill_m512_hot"]
    rng = np.random.default_rng(5)
    logits = (rng.standard_normal((64, base.n_routed)) * 3).astype(np.float32)
    bias = W.bias_f32(base.with_(m=1), 0)
    for w in (base.with_(topk=1), base.with_(norm_topk_prob=False), base.with_(gate_temp=0.5, route_scale=2.5),
              base.with_(topk=16)):
        tw, ti, _ = _select_gpu(w, logits, bias)
        rw, ri, _ = oracle.route_from_logits(oracle.cfg_of(w), logits, bias)
        np.testing.assert_array_equal(ti, ri)
        np.testing.assert_allclose(tw, rw, rtol=2e-6)
    # the largest routing: 1024 experts, 16 picks
    big = base.with_(n_routed=1024, topk=16)
    logits = (rng.standard_normal((64, 1024)) * 3).astype(np.float32)
    bias = W.bias_f32(big.with_(m=1), 0)
    for w in (big, big.with_(score_func=1), big.with_(score_func=2)):
        tw, ti, _ = _select_gpu(w, logits, bias)
        rw, ri, _ = oracle.route_from_logits(oracle.cfg_of(w), logits, bias)
        np.testing.assert_array_equal(ti, ri)
        np.testing.assert_allclose(tw, rw, rtol=2e-6)


def test_selection_nan_key_sets_status():
    w = W.WORKLOADS["tiny"]
    logits = np.arange(w.n_routed, dtype=np.float32)[None, :].repeat(2, 0)
    logits[1, 3] = np.nan
    bias = np.zeros(w.n_routed, np.float32)
    tw, ti, status = _select_gpu(w, logits, bias)
    _, ri, nan = oracle.route_from_logits(oracle.cfg_of(w), logits, bias)
    np.testing.assert_array_equal(ti, ri)
    assert nan == 1 and status & Q.MOE_STATUS_NAN_KEY


def _select_gpu_vl(w, logits, bias, bias_vl, mask):
    cfg = lib_cfg(w, max_tokens=logits.shape[0])
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    Q.moe_v41_workspace_init(ws)
    m = logits.shape[0]
    tw = torch.empty((m, w.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((m, w.topk), dtype=torch.int32, device="cuda")
    Q.moe_v41_select_from_logits_vl(cfg, torch.from_numpy(logits).cuda(), m, torch.from_numpy(bias).cuda(),
                                    torch.from_numpy(bias_vl).cuda(), torch.from_numpy(mask).cuda(), tw, ti, ws)
    status = Q.moe_v41_read_status(ws, clear=True)
    return tw.cpu().numpy(), ti.cpu().numpy(), status


def _near_tie_logits(w, bias, c=0.5):
    """logits whose sigmoid keys s + bias all land within a few f32 ulps of c,
    so that the fast keys cannot separate the picks and the exact re-scoring
    decides (ties between equal exact keys go to the lower id)"""
    s = np.clip(c - bias.astype(np.float64), 1e-6, 1 - 1e-6)
    return (w.gate_temp * np.log(s / (1.0 - s))).astype(np.float32)


@pytest.mark.parametrize("sf", [1, 2])
@pytest.mark.parametrize("name", ["decode_m1_40layer", "tiny"])
def test_selection_score_funcs_bitexact(sf, name):
    """Sigmoid and softmax scores (DeepSeek V4.1 model.py Gate.forward) with
    image tokens picking on bias_vl: indices bit-exact, weights within f32
    rounding of the oracle's."""
    w = W.WORKLOADS[name].with_(score_func=sf)
    rng = np.random.default_rng(23 + sf)
    m = 200
    logits = (rng.standard_normal((m, w.n_routed)) * 2).astype(np.float32)
    bias = W.bias_f32(w.with_(m=1), 0)
    bias_vl = W.bias_vl_f32(w.with_(m=1), 0)
    logits[0] = 25.0                                  # equal logits
    logits[1, ::3] = 40.0                             # saturated sigmoid / dominant softmax terms
    logits[2, :5] = -200.0                            # exp underflow
    logits[3] = _near_tie_logits(w, bias)             # near-ties on the token's keys
    logits[4] = _near_tie_logits(w, bias_vl)          # the same for an image token
    mask = (np.arange(m) % 3 == 1).astype(np.uint8)
    mask[3], mask[4] = 0, 1
    for b, bv in ((bias, bias_vl), (np.zeros_like(bias), np.full_like(bias, 0.01))):
        tw, ti, status = _select_gpu_vl(w, logits, b, bv, mask)
        rw, ri, nan = oracle.route_from_logits(oracle.cfg_of(w), logits, b, bv, mask)
        np.testing.assert_array_equal(ti, ri)
        np.testing.assert_allclose(tw, rw, rtol=2e-6, atol=0)
        assert status == 0 and nan == 0


def test_selection_softmax_nan_logit_makes_every_score_nan():
    w = W.WORKLOADS["tiny"].with_(score_func=2)
    logits = np.tile(np.arange(w.n_routed, dtype=np.float32), (2, 1))
    logits[1, 5] = np.nan
    bias = np.zeros(w.n_routed, np.float32)
    tw, ti, status = _select_gpu_vl(w, logits, bias, bias, np.zeros(2, np.uint8))
    rw, ri, nan = oracle.route_from_logits(oracle.cfg_of(w), logits, bias)
    np.testing.assert_array_equal(ti, ri)
    assert list(ti[1]) == list(range(w.topk)) and np.all(np.isnan(tw[1])) and np.all(np.isnan(rw[1]))
    np.testing.assert_allclose(tw[0], rw[0], rtol=2e-6)
    assert nan == w.n_routed and status & Q.MOE_STATUS_NAN_KEY


# ----------------------------------------------------------------- layers

def _check_layer(w, layer, res, tokens=None, picked_experts=True):
    """Oracle on the GPU's logits, then compare out / weights / indices."""
    lg = res["logits"]
    ref_idx_set = None
    picked = np.unique(res["topk_idx"]) if picked_experts else None
    r = oracle_for(w, layer, given_logits=lg, tokens=tokens, picked=picked)
    sel = slice(None) if tokens is None else tokens
    np.testing.assert_array_equal(res["topk_idx"][sel], r.topk_idx)
    assert_close(res["topk_w"][sel], r.topk_w, "routing weights")
    l2, _, mx, _, _ = assert_output(res["out"][sel], r)
    # the router logits themselves, against the oracle's f64 dot
    zr = oracle.router_logits(W.x_bf16(w, layer)[sel] if tokens is not None else W.x_bf16(w, layer),
                              W.router_bf16(w, layer))
    np.testing.assert_allclose(lg[sel], zr, rtol=1e-4, atol=1e-4)
    # picks from the oracle's own logits: expected identical
    im = W.image_mask(w, layer)
    bv = None if im is None else W.bias_vl_f32(w, layer)
    if im is not None and tokens is not None:
        im = im[sel]
    rw, ri, _ = oracle.route_from_logits(oracle.cfg_of(w), zr, W.bias_f32(w, layer), bv, im)
    repicked = int(np.sum(np.any(np.sort(ri, 1) != np.sort(r.topk_idx, 1), axis=1)))
    return l2, mx, repicked


@pytest.mark.parametrize("m", [1, 2, 4, 7, 8])
def test_tiny_decode(m):
    w = W.WORKLOADS["tiny"].with_(m=m)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    res = gpu_forward(dl, path=Q.MOE_PATH_DECODE)
    assert res["status"] == 0
    _, _, repicked = _check_layer(w, 0, res)
    assert repicked == 0


@pytest.mark.parametrize("variant", ["topk1", "no_norm", "no_clip", "kquant_shared", "temp"])
def test_tiny_decode_variants(variant):
    base = W.WORKLOADS["tiny"]
    w = {"topk1": base.with_(topk=1), "no_norm": base.with_(norm_topk_prob=False),
         "no_clip": base.with_(swiglu_limit=0.0), "kquant_shared": base.with_(shared_kind=W.SHARED_KQUANT),
         "temp": base.with_(gate_temp=0.7, route_scale=2.0)}[variant]
    dl = stage_layer(w, 0, experts_on_gpu=False)
    res = gpu_forward(dl, path=Q.MOE_PATH_DECODE)
    assert res["status"] == 0
    _check_layer(w, 0, res)


@pytest.mark.parametrize("sf,vl,n_routed", [(1, False, 16), (2, False, 16), (0, True, 16), (0, True, 384),
                                             (1, True, 384), (2, True, 384)])
@pytest.mark.parametrize("m", [1, 8])
def test_tiny_decode_score_funcs_and_image_tokens(sf, vl, n_routed, m):
    """The Gate's score functions and the image-token bias through the fused
    decode kernel (384 experts: the register-resident selection path)."""
    w = W.WORKLOADS["tiny"].with_(m=m, score_func=sf, n_routed=n_routed, topk=2 if n_routed == 16 else 6,
                                  image_frac=(1.0 if m == 1 else 0.5) if vl else 0.0)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    assert (dl.image_mask is not None) == vl
    res = gpu_forward(dl, path=Q.MOE_PATH_DECODE)
    assert res["status"] == 0
    _, _, repicked = _check_layer(w, 0, res)
    assert repicked == 0


@pytest.mark.parametrize("sf", [0, 1, 2])
def test_decode_largest_routing(sf):
    """1024 experts, 16 picks per token, 8 tokens: 128 token/expert pairs,
    the largest decode plan; every score function."""
    w = W.WORKLOADS["tiny"].with_(n_routed=1024, topk=16, m=8, score_func=sf)
    dl = stage_layer(w, 0, experts_on_gpu=True)
    res = gpu_forward(dl, path=Q.MOE_PATH_DECODE)
    assert res["status"] == 0
    _, _, repicked = _check_layer(w, 0, res)
    assert repicked == 0


def test_tiny_decode_outliers_clip():
    w = W.WORKLOADS["tiny"].with_(m=8, outlier_frac=0.25)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    res = gpu_forward(dl, path=Q.MOE_PATH_DECODE)
    _check_layer(w, 0, res)


def test_decode_deterministic():
    w = W.WORKLOADS["tiny"].with_(m=8)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    a = gpu_forward(dl, path=Q.MOE_PATH_DECODE)
    b = gpu_forward(dl, path=Q.MOE_PATH_DECODE, ws=a["ws"])
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["topk_w"], b["topk_w"])


def test_gpu_generator_matches_host():
    w = W.WORKLOADS["tiny"]
    dl = stage_layer(w, 3, experts_on_gpu=True)
    from synth.device import slot_layout
    o1, o3, o2, slot = slot_layout(w)
    got = dl.experts.cpu().numpy()
    for e in (0, 7, 15):
        w1, w3, w2 = W.expert_blocks(w, 3, e)
        np.testing.assert_array_equal(got[e, o1:o1 + w.w1_bytes], w1)
        np.testing.assert_array_equal(got[e, o3:o3 + w.w1_bytes], w3)
        np.testing.assert_array_equal(got[e, o2:o2 + w.w2_bytes], w2)


def test_missing_expert_status():
    w = W.WORKLOADS["tiny"].with_(m=4)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    first = gpu_forward(dl, path=Q.MOE_PATH_DECODE)
    victim = int(first["topk_idx"][0, 0])
    dl.expert_ptrs[victim] = 0
    res = gpu_forward(dl, path=Q.MOE_PATH_DECODE)
    assert res["status"] & Q.MOE_STATUS_MISSING_EXPERT
    # the other tokens that did not pick the victim are unchanged
    keep = [t for t in range(w.m) if victim not in first["topk_idx"][t]]
    if keep:
        np.testing.assert_allclose(res["out"][keep], first["out"][keep], rtol=1e-6, atol=1e-6)


def test_wait_timeout_sets_status_and_returns():
    """Every in-kernel wait is bounded.  A ticket counter pushed past every
    item leaves the router count unreachable: the planner, the producer and
    the consumers give up after wait_timeout_us, the call ends with
    MOE_STATUS_TIMEOUT, and the next call on the re-initialised workspace is
    correct (the context stays usable; no fault, no trap)."""
    w = W.WORKLOADS["tiny"].with_(m=2)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    cfg = lib_cfg(w, path=Q.MOE_PATH_DECODE, timeout_us=20000)
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    Q.moe_v41_workspace_init(ws)
    # control block: status, route_arrive, then the decode ticket counter (u32 at byte 8)
    ws[8:12].view(torch.int32).fill_(0x40000000)
    t0 = time.perf_counter()
    res = gpu_forward(dl, path=Q.MOE_PATH_DECODE, ws=ws, cfg=cfg)
    elapsed = time.perf_counter() - t0
    assert res["status"] & Q.MOE_STATUS_TIMEOUT
    assert elapsed < 5.0
    Q.moe_v41_workspace_init(ws)
    good = gpu_forward(dl, path=Q.MOE_PATH_DECODE, ws=ws, cfg=cfg)
    assert good["status"] == 0
    r = oracle_for(w, 0, given_logits=good["logits"])
    np.testing.assert_array_equal(good["topk_idx"], r.topk_idx)
    assert_output(good["out"], r, "output after a timed-out call")


def test_graph_replay_matches_eager_and_the_oracle():
    """A decode step (three layer calls) captured as a CUDA graph and replayed
    gives the eager launches' results bit for bit (the call has no host round
    trip, and the kernel resets its call-wide counters itself), and every
    replayed layer's output is within the parity bars of the oracle run on
    the replay's own logits."""
    w = W.WORKLOADS["tiny"].with_(m=3)
    layers = [stage_layer(w, l, experts_on_gpu=False) for l in range(3)]
    cfg = lib_cfg(w, path=Q.MOE_PATH_DECODE)
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    Q.moe_v41_workspace_init(ws)
    outs = [torch.empty((w.m, w.dim), device="cuda") for _ in layers]
    tws = [torch.empty((w.m, w.topk), device="cuda") for _ in layers]
    tis = [torch.empty((w.m, w.topk), dtype=torch.int32, device="cuda") for _ in layers]
    lgs = [torch.empty((w.m, w.n_routed), device="cuda") for _ in layers]

    def step():
        for l, d in enumerate(layers):
            Q.moe_v41_forward(cfg, d.x, w.m, d.router_w, d.bias, d.expert_ptrs, w.shared_kind, d.sh1, d.sh3, d.sh2,
                              outs[l], tws[l], tis[l], lgs[l], ws)

    step()
    torch.cuda.synchronize()
    eager = [(o.clone(), t.clone(), i.clone()) for o, t, i in zip(outs, tws, tis)]
    for o, t, i, g in zip(outs, tws, tis, lgs):
        o.zero_()
        t.zero_()
        i.zero_()
        g.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert Q.moe_v41_read_status(ws, clear=True) == 0
    for (eo, et, ei), o, t, i in zip(eager, outs, tws, tis):
        assert torch.equal(eo, o) and torch.equal(et, t) and torch.equal(ei, i)
    for l in range(len(layers)):
        res = dict(out=outs[l].cpu().numpy(), topk_w=tws[l].cpu().numpy(), topk_idx=tis[l].cpu().numpy(),
                   logits=lgs[l].cpu().numpy())
        _, _, repicked = _check_layer(w, l, res)
        assert repicked == 0


def test_graph_replay_full_shape_step_matches_the_oracle():
    """The 40-layer decode step as the bench runs it (one CUDA graph of the
    layer calls, all 40 layers' experts resident), replayed twice: every
    layer's replayed output, weights and picks are checked against the
    oracle on the replay's own logits."""
    w = W.WORKLOADS["decode_m1_40layer"]
    n_layers = 40
    free, _ = torch.cuda.mem_get_info()
    from synth.device import slot_layout
    need = n_layers * w.n_routed * slot_layout(w)[3] + (4 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB of free device memory")
    layers = [stage_layer(w, l, experts_on_gpu=True) for l in range(n_layers)]
    cfg = lib_cfg(w)
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    Q.moe_v41_workspace_init(ws)
    outs = [torch.empty((w.m, w.dim), device="cuda") for _ in layers]
    tws = [torch.empty((w.m, w.topk), device="cuda") for _ in layers]
    tis = [torch.empty((w.m, w.topk), dtype=torch.int32, device="cuda") for _ in layers]
    lgs = [torch.empty((w.m, w.n_routed), device="cuda") for _ in layers]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        Q.moe_v41_forward(cfg, layers[0].x, w.m, layers[0].router_w, layers[0].bias, layers[0].expert_ptrs,
                          w.shared_kind, layers[0].sh1, layers[0].sh3, layers[0].sh2, outs[0], tws[0], tis[0],
                          lgs[0], ws, stream=s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            for l, d in enumerate(layers):
                Q.moe_v41_forward(cfg, d.x, w.m, d.router_w, d.bias, d.expert_ptrs, w.shared_kind, d.sh1, d.sh3,
                                  d.sh2, outs[l], tws[l], tis[l], lgs[l], ws, stream=s)
    for o in outs:
        o.zero_()
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert Q.moe_v41_read_status(ws, clear=True) == 0
    for l in range(n_layers):
        res = dict(out=outs[l].cpu().numpy(), topk_w=tws[l].cpu().numpy(), topk_idx=tis[l].cpu().numpy(),
                   logits=lgs[l].cpu().numpy())
        _, _, repicked = _check_layer(w, l, res)
        assert repicked == 0
    del layers, g
    torch.cuda.empty_cache()


def test_argument_errors():
    w = W.WORKLOADS["tiny"]
    cfg = lib_cfg(w)
    with pytest.raises(Q.MoeError):
        Q.moe_v41_quantize_q8_1(torch.zeros(31, device="cuda"), True, 1, 31, torch.zeros(64, dtype=torch.uint8,
                                                                                         device="cuda"))
    bad = lib_cfg(w.with_(dim=500))
    assert Q.moe_v41_workspace_bytes(bad) == 0
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    dl = stage_layer(w, 0, experts_on_gpu=False)
    out = torch.empty((w.m, w.dim), device="cuda")
    tw = torch.empty((w.m, w.topk), device="cuda")
    ti = torch.empty((w.m, w.topk), dtype=torch.int32, device="cuda")
    with pytest.raises(Q.MoeError) as e:
        Q.moe_v41_forward(cfg, dl.x, w.m, dl.router_w, dl.bias, dl.expert_ptrs, 0, dl.sh1, dl.sh3, dl.sh2, out, tw,
                          ti, None, ws)
    assert e.value.code == Q.MOE_ERR_WORKSPACE


# ------------------------------------------------------ full-size decode

@pytest.mark.parametrize("layer", range(40))
def test_decode_m1_full_shape_layers(layer):
    """The 40-layer decode workload at full shape, every layer checked in full
    (each layer's own seeded x, router, bias, experts and shared expert)."""
    w = W.WORKLOADS["decode_m1_40layer"]
    dl = stage_layer(w, layer, experts_on_gpu=True)
    res = gpu_forward(dl)
    assert res["status"] == 0
    _, _, repicked = _check_layer(w, layer, res)
    assert repicked == 0
    del dl
    torch.cuda.empty_cache()


def test_decode_m8_kquant_shared_full_shape():
    w = W.WORKLOADS["decode_m8_kquant_shared"]
    dl = stage_layer(w, 0, experts_on_gpu=True)
    res = gpu_forward(dl)
    assert res["status"] == 0
    distinct = np.unique(res["topk_idx"]).size
    assert 30 <= distinct <= 48
    _, _, repicked = _check_layer(w, 0, res)
    assert repicked == 0
