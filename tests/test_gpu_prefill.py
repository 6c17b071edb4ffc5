"""GPU parity of the prefill path (tensor-core GEMMs over expert-grouped
tokens) against the oracle, through the C-ABI.

Same bars as the decode path: top-k indices bit-exact on identical f32
logits; outputs and routing weights within 2e-3 relative L2 and max-abs <=
1e-2 x RMS of the oracle output.  The tiny shapes are checked on every token;
the full-size prefill workloads (512 tokens with hot experts, 4096 tokens
with x50 outlier rows) on every token as well, plus properties of every
token."""
import numpy as np
import pytest

import oracle
import synth.workloads as W
from _helpers import assert_close, assert_output, gpu_forward, lib_cfg, oracle_for

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import quantized_mixture_experts_router_gb300 as Q  # noqa: E402
from synth.device import stage_layer  # noqa: E402


def _check(w, layer, res, tokens=None):
    """Oracle on the GPU's logits for the given tokens (all by default)."""
    sel = slice(None) if tokens is None else np.asarray(tokens)
    picked = np.unique(res["topk_idx"][sel])
    r = oracle_for(w, layer, given_logits=res["logits"], tokens=tokens, picked=picked)
    np.testing.assert_array_equal(res["topk_idx"][sel], r.topk_idx)
    ew = assert_close(res["topk_w"][sel], r.topk_w, "routing weights")
    eo = assert_output(res["out"][sel], r)
    print(f"\n{w.name} m={w.m}: weights rel L2 {ew[0]:.2e} max/RMS {ew[1]:.2e}; "
          f"output rel L2 {eo[0]:.2e} max/RMS {eo[1]:.2e}, {eo[2]:.2e} after {eo[4]} flips in {eo[3]} tokens")
    # router logits against the oracle's f64 dot.  The tensor cores' f32
    # accumulation is not a sequential IEEE sum: bound the error by
    # 2^-14 of sum_k |x_k w_k| (about 8x the largest error seen).
    x = W.x_bf16(w, layer)[sel]
    R = W.router_bf16(w, layer)
    zr = oracle.router_logits(x, R)
    bf = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    cond = np.abs(bf(x)) @ np.abs(bf(R)).T
    err = np.abs(res["logits"][sel] - zr)
    assert np.all(err <= 2.0 ** -14 * cond + 1e-6), float((err / (cond + 1e-30)).max())
    return r


@pytest.mark.parametrize("m", [1, 4, 9, 100, 700])
def test_tiny_prefill(m):
    w = W.WORKLOADS["tiny"].with_(m=m)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    res = gpu_forward(dl, path=Q.MOE_PATH_PREFILL)
    assert res["status"] == 0
    _check(w, 0, res)


@pytest.mark.parametrize("m", [5, 130])
def test_tiny_prefill_odd_superblock_counts(m):
    """dim 768 and inter 768: three super-blocks per row, so the gate/up
    rows are only 4-byte aligned and both GEMMs end on a lone super-block."""
    w = W.WORKLOADS["tiny"].with_(dim=768, inter=768, m=m)
    dl = stage_layer(w, 0, experts_on_gpu=True)
    res = gpu_forward(dl, path=Q.MOE_PATH_PREFILL)
    assert res["status"] == 0
    _check(w, 0, res)


@pytest.mark.parametrize("m", [40, 300])
def test_tiny_prefill_kquant_shared_and_variants(m):
    """The K-quant shared expert as the GEMMs' extra expert, and the
    unclipped, unnormalised variant, on the prefill kernels."""
    for w in (W.WORKLOADS["tiny"].with_(m=m, shared_kind=W.SHARED_KQUANT),
              W.WORKLOADS["tiny"].with_(m=m, swiglu_limit=0.0, norm_topk_prob=False)):
        dl = stage_layer(w, 0, experts_on_gpu=True)
        res = gpu_forward(dl, path=Q.MOE_PATH_PREFILL)
        assert res["status"] == 0
        _check(w, 0, res)


@pytest.mark.parametrize("path,m", [("prefill", 37), ("decode", 3)])
@pytest.mark.parametrize("shared", [W.SHARED_BF16, W.SHARED_KQUANT])
def test_tiny_unaligned_out(path, m, shared):
    """out needs only f32 alignment: one float past a 16-byte boundary the
    prefill's ordered combine takes its scalar form, with the same sums bit
    for bit (the decode kernel writes out by value)."""
    pth = Q.MOE_PATH_PREFILL if path == "prefill" else Q.MOE_PATH_DECODE
    w = W.WORKLOADS["tiny"].with_(m=m, shared_kind=shared)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    ref = gpu_forward(dl, path=pth)
    cfg = lib_cfg(w, path=pth)
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    Q.moe_v41_workspace_init(ws)
    buf = torch.full((w.m * w.dim + 4,), float("nan"), dtype=torch.float32, device="cuda")
    out = buf[1:1 + w.m * w.dim].view(w.m, w.dim)
    assert out.data_ptr() % 16 == 4
    tw = torch.empty((w.m, w.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((w.m, w.topk), dtype=torch.int32, device="cuda")
    Q.moe_v41_forward(cfg, dl.x, w.m, dl.router_w, dl.bias, dl.expert_ptrs, w.shared_kind, dl.sh1, dl.sh3, dl.sh2,
                      out, tw, ti, None, ws)
    assert Q.moe_v41_read_status(ws, clear=True) == 0
    np.testing.assert_array_equal(out.cpu().numpy(), ref["out"])
    np.testing.assert_array_equal(ti.cpu().numpy(), ref["topk_idx"])
    # nothing written outside out
    assert torch.isnan(buf[0]).item() and bool(torch.isnan(buf[1 + w.m * w.dim:]).all())
    if path == "prefill":
        _check(w, 0, ref)
    else:
        r = oracle_for(w, 0, given_logits=ref["logits"])
        np.testing.assert_array_equal(ref["topk_idx"], r.topk_idx)
        assert_output(ref["out"], r)


def test_tiny_prefill_auto_path_above_eight():
    w = W.WORKLOADS["tiny"].with_(m=33)
    dl = stage_layer(w, 1, experts_on_gpu=False)
    res = gpu_forward(dl)  # AUTO: 33 tokens take the prefill kernels
    assert res["status"] == 0
    _check(w, 1, res)


def test_tiny_prefill_many_column_tiles():
    """Two hot experts take nearly every token: several 256-pair column
    tiles per expert, the last one ragged."""
    w = W.WORKLOADS["tiny"].with_(m=1100, hot_experts=2, hot_bias=3.0)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    res = gpu_forward(dl, path=Q.MOE_PATH_PREFILL)
    counts = np.bincount(res["topk_idx"].ravel(), minlength=w.n_routed)
    assert counts.max() > 3 * 256
    _check(w, 0, res)


@pytest.mark.parametrize("variant", ["topk1", "no_norm", "no_clip", "kquant_shared", "temp", "outliers", "wide"])
def test_tiny_prefill_variants(variant):
    base = W.WORKLOADS["tiny"].with_(m=40)
    w = {"topk1": base.with_(topk=1), "no_norm": base.with_(norm_topk_prob=False),
         "no_clip": base.with_(swiglu_limit=0.0), "kquant_shared": base.with_(shared_kind=W.SHARED_KQUANT),
         "temp": base.with_(gate_temp=0.7, route_scale=2.0), "outliers": base.with_(outlier_frac=0.2),
         "wide": base.with_(dim=1024, inter=768, n_routed=200, topk=8)}[variant]
    dl = stage_layer(w, 0, experts_on_gpu=False)
    res = gpu_forward(dl, path=Q.MOE_PATH_PREFILL)
    assert res["status"] == 0
    r = _check(w, 0, res)
    if variant == "outliers":
        assert r.clipped > 0


def test_prefill_matches_decode_path():
    w = W.WORKLOADS["tiny"].with_(m=8, shared_kind=W.SHARED_KQUANT)
    dl = stage_layer(w, 2, experts_on_gpu=False)
    a = gpu_forward(dl, path=Q.MOE_PATH_PREFILL)
    b = gpu_forward(dl, path=Q.MOE_PATH_DECODE)
    np.testing.assert_array_equal(a["topk_idx"], b["topk_idx"])
    # each against the oracle on its own logits (the two paths may take a
    # requantisation of h on either side of a boundary independently)
    for res, what in ((a, "prefill path"), (b, "decode path")):
        assert_output(res["out"], oracle_for(w, 2, given_logits=res["logits"]), what)


def test_prefill_deterministic():
    w = W.WORKLOADS["tiny"].with_(m=300)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    a = gpu_forward(dl, path=Q.MOE_PATH_PREFILL)
    b = gpu_forward(dl, path=Q.MOE_PATH_PREFILL, ws=a["ws"])
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["topk_w"], b["topk_w"])
    np.testing.assert_array_equal(a["topk_idx"], b["topk_idx"])


def test_prefill_missing_expert():
    w = W.WORKLOADS["tiny"].with_(m=50)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    first = gpu_forward(dl, path=Q.MOE_PATH_PREFILL)
    victim = int(first["topk_idx"][0, 0])
    dl.expert_ptrs[victim] = 0
    res = gpu_forward(dl, path=Q.MOE_PATH_PREFILL)
    assert res["status"] & Q.MOE_STATUS_MISSING_EXPERT
    keep = [t for t in range(w.m) if victim not in first["topk_idx"][t]]
    assert keep
    np.testing.assert_array_equal(res["out"][keep], first["out"][keep])
    hit = [t for t in range(w.m) if victim in first["topk_idx"][t]]
    assert np.all(np.isfinite(res["out"][hit]))


def test_route_above_eight_tokens():
    w = W.WORKLOADS["tiny"].with_(m=77)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    cfg = lib_cfg(w)
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    Q.moe_v41_workspace_init(ws)
    lg = torch.empty((w.m, w.n_routed), dtype=torch.float32, device="cuda")
    tw = torch.empty((w.m, w.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((w.m, w.topk), dtype=torch.int32, device="cuda")
    Q.moe_v41_route(cfg, dl.x, w.m, dl.router_w, dl.bias, lg, tw, ti, ws)
    torch.cuda.synchronize()
    logits = lg.cpu().numpy()
    zr = oracle.router_logits(W.x_bf16(w, 0), W.router_bf16(w, 0))
    np.testing.assert_allclose(logits, zr, rtol=1e-4, atol=1e-4)
    rw, ri, _ = oracle.route_from_logits(oracle.cfg_of(w), logits, W.bias_f32(w, 0))
    np.testing.assert_array_equal(ti.cpu().numpy(), ri)
    np.testing.assert_allclose(tw.cpu().numpy(), rw, rtol=2e-6)


@pytest.mark.parametrize("sf,vl,n_routed,m", [(1, False, 16, 100), (2, False, 16, 100), (0, True, 16, 100),
                                               (1, True, 384, 64), (2, True, 384, 64)])
def test_tiny_prefill_score_funcs_and_image_tokens(sf, vl, n_routed, m):
    """The Gate's sigmoid and softmax scores and the image-token bias through
    the prefill kernels."""
    w = W.WORKLOADS["tiny"].with_(m=m, score_func=sf, n_routed=n_routed, topk=2 if n_routed == 16 else 6,
                                  image_frac=0.4 if vl else 0.0)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    res = gpu_forward(dl, path=Q.MOE_PATH_PREFILL)
    assert res["status"] == 0
    _check(w, 0, res)


@pytest.mark.parametrize("m,path", [(5, Q.MOE_PATH_AUTO), (77, Q.MOE_PATH_AUTO)])
def test_route_vl_softmax(m, path):
    """moe_v41_route_vl on both router paths (decode kernel for m <= 8,
    tensor-core GEMM plus selection above): softmax scores, image tokens."""
    w = W.WORKLOADS["tiny"].with_(m=m, score_func=2, image_frac=0.5)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    cfg = lib_cfg(w, path=path)
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    Q.moe_v41_workspace_init(ws)
    lg = torch.empty((w.m, w.n_routed), dtype=torch.float32, device="cuda")
    tw = torch.empty((w.m, w.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((w.m, w.topk), dtype=torch.int32, device="cuda")
    Q.moe_v41_route_vl(cfg, dl.x, w.m, dl.router_w, dl.bias, dl.bias_vl, dl.image_mask, lg, tw, ti, ws)
    assert Q.moe_v41_read_status(ws, clear=True) == 0
    logits = lg.cpu().numpy()
    rw, ri, _ = oracle.route_from_logits(oracle.cfg_of(w), logits, W.bias_f32(w, 0), W.bias_vl_f32(w, 0),
                                         W.image_mask(w, 0))
    np.testing.assert_array_equal(ti.cpu().numpy(), ri)
    np.testing.assert_allclose(tw.cpu().numpy(), rw, rtol=2e-6)
    # the image tokens really picked on bias_vl: their picks under the text bias differ somewhere
    _, ri_text, _ = oracle.route_from_logits(oracle.cfg_of(w), logits, W.bias_f32(w, 0))
    assert np.any(ri_text != ri)


@pytest.mark.parametrize("m", [1, 3])
def test_wide_shapes_take_the_prefill_kernels_at_few_tokens(m):
    """dim 7680 / inter 4096 (the largest widths the configuration allows):
    the decode kernel's stages do not hold them, so MOE_PATH_AUTO runs every
    call, even one token, on the prefill kernels."""
    w = W.WORKLOADS["tiny"].with_(dim=7680, inter=4096, m=m)
    cfg = lib_cfg(w)
    assert Q.moe_v41_kernel_launches(cfg, 1, w.shared_kind) == Q.moe_v41_kernel_launches(
        lib_cfg(w.with_(m=64)), 64, w.shared_kind) > 1
    dl = stage_layer(w, 0, experts_on_gpu=True)
    res = gpu_forward(dl)
    assert res["status"] == 0
    _check(w, 0, res)


# ------------------------------------------------------ full-size prefill

def _full_properties(w, layer, res):
    assert res["status"] == 0
    assert np.all(np.isfinite(res["out"]))
    # every token's selection from the GPU logits, on the host
    rw, ri, _ = oracle.route_from_logits(oracle.cfg_of(w), res["logits"], W.bias_f32(w, layer))
    np.testing.assert_array_equal(res["topk_idx"], ri)
    np.testing.assert_allclose(res["topk_w"], rw, rtol=2e-6)
    s = res["topk_w"].sum(axis=1)
    np.testing.assert_allclose(s, w.route_scale, rtol=1e-5)


def test_prefill_m512_hot_full_shape():
    """Every token of the 512-token hot-expert workload against the oracle."""
    w = W.WORKLOADS["prefill_m512_hot"]
    dl = stage_layer(w, 0, experts_on_gpu=True)
    res = gpu_forward(dl)
    _full_properties(w, 0, res)
    hot = W.hot_experts(w, 0)
    counts = np.bincount(res["topk_idx"].ravel(), minlength=w.n_routed)
    assert counts[hot].sum() > 0.5 * counts.sum()  # imbalanced routing
    _check(w, 0, res)


@pytest.mark.slow
def test_prefill_m4096_outliers_full_shape():
    """Every token of the 4096-token workload with x50 outlier rows against
    the oracle (a few minutes of oracle time on the host cores): every
    (expert, row tile, column tile) of the call is compared, each expert's
    last column tile included."""
    w = W.WORKLOADS["prefill_m4096_outliers"]
    dl = stage_layer(w, 0, experts_on_gpu=True)
    res = gpu_forward(dl)
    _full_properties(w, 0, res)
    r = _check(w, 0, res)
    assert r.clipped > 0
    # the outlier rows on their own (their errors would vanish in the whole)
    rows = W.outlier_rows(w, 0)
    assert_output(res["out"][rows], r, "outlier rows", rows=rows)


@pytest.mark.slow
def test_prefill_at_the_token_limit():
    """max_tokens = 65536, the configuration's limit: 458,752 pair rows, so the
    per-pair buffers hold more than 2^31 values (every index into them is
    64-bit).  Properties of every token, and the oracle on sampled tokens:
    the first and last, outlier rows and a seeded spread."""
    w = W.WORKLOADS["prefill_m4096_outliers"].with_(m=65536)
    dl = stage_layer(w, 0, experts_on_gpu=True)
    res = gpu_forward(dl)
    _full_properties(w, 0, res)
    rng = np.random.default_rng(11)
    out_rows = W.outlier_rows(w, 0)
    tokens = np.unique(np.concatenate([[0, w.m - 1], out_rows[:4], rng.choice(w.m, 10, replace=False)]))
    _check(w, 0, res, tokens=tokens)


@pytest.mark.parametrize("path,m", [("decode", 4), ("prefill", 40)])
@pytest.mark.parametrize("n", [1, 16])
def test_every_expert_picked(path, m, n):
    """The degenerate routings: one expert in all (k = N = 1, no
    renormalisation at k = 1) and every expert picked (k = N = 16, no
    (k+1)-th key to separate), on both paths."""
    w = W.WORKLOADS["tiny"].with_(m=m, n_routed=n, topk=n)
    dl = stage_layer(w, 0, experts_on_gpu=False)
    res = gpu_forward(dl, path=Q.MOE_PATH_DECODE if path == "decode" else Q.MOE_PATH_PREFILL)
    assert res["status"] == 0
    assert np.array_equal(np.sort(res["topk_idx"], axis=1), np.tile(np.arange(n), (m, 1)))
    _check(w, 0, res)
