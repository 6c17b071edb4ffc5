"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: IEEE
format facts, hand-worked blocks and routing cases (tests/golden), closed
forms, invariants stated on the pages, and reductions to library routines
(numpy sort / matmul).  The pages cited: metrale moe_v41 module docs and its
moe_v41.rs source page; the open-model-atlas page "DeepSeek V4.1 · Mixture of
experts" (its steps, Parameters table, model.py listings and config.json).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth
import synth.workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ number formats

def test_bf16_round_to_nearest_even():
    # bf16 keeps the top 16 bits of an f32; ties go to even (moe_v41.rs, fn bf16_bytes)
    f = lambda bits: np.array([bits], dtype=np.uint32).view(np.float32)[0]
    assert oracle.bf16_from_f32(1.0) == 0x3F80
    assert oracle.bf16_from_f32(f(0x3F808000)) == 0x3F80  # tie, even below
    assert oracle.bf16_from_f32(f(0x3F818000)) == 0x3F82  # tie, even above
    assert oracle.bf16_from_f32(f(0x3F808001)) == 0x3F81  # just above the tie
    assert oracle.bf16_from_f32(-2.5) == 0xC020
    assert oracle.bf16_value(0x3F80) == 1.0
    assert oracle.bf16_value(0xC020) == -2.5


def test_fp16_values():
    assert oracle.f16_value(0x3C00) == 1.0
    assert oracle.f16_value(0x0001) == 2.0 ** -24
    assert oracle.f16_value(0x7BFF) == 65504.0
    assert oracle.f16_value(0xC000) == -2.0
    assert oracle.f16_from_f32(1.0 / 3.0) == 0x3555
    assert oracle.f16_from_f32(2.0 ** -20) == 0x0010  # subnormal kept
    assert oracle.f16_from_f32(65520.0) == 0x7C00     # rounds to infinity


# ------------------------------------------------------------ K-quant blocks

def _block(nbytes, fills):
    b = np.zeros(nbytes, dtype=np.uint8)
    for off, ln, val in fills:
        b[off:off + ln] = val
    return b


def _check_golden(entry, values):
    if "expect_all" in entry:
        np.testing.assert_array_equal(values, np.full(256, entry["expect_all"]))
    for start, ln, v in entry.get("expect_runs", []):
        np.testing.assert_array_equal(values[start:start + ln], np.full(ln, v))


def test_kquant_golden_blocks():
    g = json.load(open(os.path.join(GOLDEN, "kquant_blocks.json")))
    for e in g["q2k"]:
        _check_golden(e, oracle.dequant_q2k(_block(84, e["fill"])))
    for e in g["q3k"]:
        _check_golden(e, oracle.dequant_q3k(_block(110, e["fill"])))


# elements touched by one quant byte: worked out by hand from the block layout
# (256 weights = two halves of 128; each half stores four 2-bit planes of 32)
QS_BYTE_ELEMENTS = {0: [0, 32, 64, 96], 5: [5, 37, 69, 101], 31: [31, 63, 95, 127],
                    32: [128, 160, 192, 224], 63: [159, 191, 223, 255], 40: [136, 168, 200, 232]}


@pytest.mark.parametrize("k", sorted(QS_BYTE_ELEMENTS))
def test_q2k_quant_byte_mapping(k):
    b = _block(84, [(0, 16, 1), (81, 1, 0x3C)])  # scale 1, min 0, d = 1
    b[16 + k] = 0xFF
    w = oracle.dequant_q2k(b)
    assert sorted(np.nonzero(w)[0].tolist()) == QS_BYTE_ELEMENTS[k]
    assert np.all(w[QS_BYTE_ELEMENTS[k]] == 3.0)


@pytest.mark.parametrize("sb", [0, 1, 7, 8, 15])
def test_q2k_scale_byte_covers_its_sub_block(sb):
    b = _block(84, [(16, 64, 0x55), (81, 1, 0x3C), (83, 1, 0x3C)])  # q = 1, d = dmin = 1
    b[sb] = 0x35  # scale 5, min 3
    w = oracle.dequant_q2k(b)
    expect = np.zeros(256)
    expect[16 * sb:16 * sb + 16] = 5.0 - 3.0
    np.testing.assert_array_equal(w, expect)


@pytest.mark.parametrize("l,bit,elem", [(0, 0, 0), (3, 5, 163), (17, 2, 81), (31, 7, 255), (16, 4, 144)])
def test_q3k_hmask_bit_mapping(l, bit, elem):
    # hmask byte l, bit p selects element 128*(p//4) + 32*(p%4) + l (worked out by hand)
    b = _block(110, [(96, 8, 0x11), (104, 4, 0xAA), (109, 1, 0x3C)])  # scale code 33, d = 1, q = -4
    b[l] = 1 << bit
    w = oracle.dequant_q3k(b)
    assert w[elem] == 0.0            # hb set: q = lo - 0 = 0
    assert np.sum(w == 0.0) == 1 and np.all(np.delete(w, elem) == -4.0)


def test_q3k_scale_codes_each_sub_block():
    # code_b = b + 20: low nibbles in bytes 0..7 (b < 8) / high nibbles (b >= 8),
    # two high bits of sub-block b at bits 2*(b//4) of byte 8 + b%4
    codes = [b + 20 for b in range(16)]
    sc = np.zeros(12, dtype=np.uint8)
    for b, c in enumerate(codes):
        lo, hi = c & 15, c >> 4
        if b < 8:
            sc[b] |= lo
        else:
            sc[b - 8] |= lo << 4
        sc[8 + b % 4] |= hi << (2 * (b // 4))
    assert [oracle.q3k_scale_code(sc, b) for b in range(16)] == codes
    blk = _block(110, [(0, 32, 0xFF), (32, 64, 0x55), (109, 1, 0x3C)])
    blk[96:108] = sc
    w = oracle.dequant_q3k(blk)
    np.testing.assert_array_equal(w, np.repeat(np.array(codes, dtype=np.float64) - 32.0, 16))


def test_q3k_every_scale_code_decodes():
    for c in range(64):
        sc = np.zeros(12, dtype=np.uint8)
        sc[0] = c & 15
        sc[8] = c >> 4
        assert oracle.q3k_scale_code(sc, 0) == c


def test_dequant_is_linear_in_d():
    k = synth.key(7, 0, synth.T_W1, 0)
    blk = synth.q2k_blocks(1, k)
    w = oracle.dequant_q2k(blk)
    b2 = blk.copy()
    d = oracle.f16_value(int(blk[80]) | (int(blk[81]) << 8))
    dm = oracle.f16_value(int(blk[82]) | (int(blk[83]) << 8))
    b2[80:82] = np.array([synth.half_bits(2 * d)], dtype=np.uint16).view(np.uint8)
    b2[82:84] = np.array([synth.half_bits(2 * dm)], dtype=np.uint16).view(np.uint8)
    np.testing.assert_array_equal(oracle.dequant_q2k(b2), 2 * w)


# --------------------------------------------------------------------- q8_1

def test_q8_1_exact_integers():
    k = np.arange(-127, 129, dtype=np.float32)[:256]
    k = np.clip(k, -127, 127)
    rng = np.random.default_rng(0)
    k = rng.permutation(k)
    k[::32] = np.where(np.arange(8) % 2 == 0, 127.0, -127.0)  # amax 127 in every block
    for p in (-6, 0, 3):
        x = k * np.float32(2.0 ** p)
        q8 = oracle.quantize_q8_1(x)
        for blk in range(8):
            b = q8[36 * blk:36 * blk + 36]
            xb = x[32 * blk:32 * blk + 32]
            d = np.float32(2.0 ** p)  # amax = 127 * 2^p
            assert oracle.f16_value(int(b[0]) | (int(b[1]) << 8)) == d
            np.testing.assert_array_equal(b[4:].view(np.int8).astype(np.float32) * np.float32(d), xb)


def test_q8_1_half_rounds_away_from_zero():
    x = np.zeros(32, dtype=np.float32)
    x[:6] = [127.0, 0.5, -0.5, 1.5, -2.5, 126.5]
    q = oracle.quantize_q8_1(x)[4:].view(np.int8)
    assert q[:6].tolist() == [127, 1, -1, 2, -3, 127]
    assert np.all(q[6:] == 0)


def test_q8_1_zero_block_and_sum_field():
    z = oracle.quantize_q8_1(np.zeros(32, dtype=np.float32))
    assert np.all(z == 0)
    x = np.zeros(32, dtype=np.float32)
    x[0], x[1], x[2] = 127.0, 64.0, -3.0
    q = oracle.quantize_q8_1(x)
    assert oracle.f16_value(int(q[2]) | (int(q[3]) << 8)) == 188.0  # s = d * sum q, d = 1
    q = oracle.quantize_q8_1(x * np.float32(0.125))
    assert oracle.f16_value(int(q[0]) | (int(q[1]) << 8)) == 0.125
    assert oracle.f16_value(int(q[2]) | (int(q[3]) << 8)) == 23.5  # the same codes, s = 188 / 8


def test_q8_1_subnormal_scale():
    x = np.zeros(32, dtype=np.float32)
    x[0] = np.float32(127.0 * 2.0 ** -20)
    q = oracle.quantize_q8_1(x)
    assert int(q[0]) | (int(q[1]) << 8) == 0x0010
    assert q[4:].view(np.int8)[0] == 127


def test_q8_1_error_bound():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(4096) * np.repeat(rng.uniform(0.01, 50, 128), 32)).astype(np.float32)
    q8 = oracle.quantize_q8_1(x)
    xh = oracle.dequant_q8_1(q8, 4096)
    for blk in range(128):
        xb = x[32 * blk:32 * blk + 32].astype(np.float64)
        d = np.float32(np.abs(x[32 * blk:32 * blk + 32]).max() / np.float32(127))
        d16 = oracle.f16_value(int(q8[36 * blk]) | (int(q8[36 * blk + 1]) << 8))
        bound = d / 2 * (1 + 1e-6) + abs(d - d16) * 127
        assert np.max(np.abs(xb - xh[32 * blk:32 * blk + 32])) <= bound


# -------------------------------------------------------------------- scores

def test_score_closed_forms():
    assert abs(oracle.score(0.0) - math.sqrt(math.log(2.0))) <= 1e-7  # softplus(0) = ln 2
    assert oracle.score(25.0) == 5.0       # softplus(t) = t above 20
    assert oracle.score(400.0) == 20.0
    assert oracle.score(50.0, 2.0) == 5.0  # the temperature divides first
    # softplus(t) ~ e^t for t -> -inf, so s ~ e^(t/2)
    assert abs(oracle.score(-30.0) / math.exp(-15.0) - 1) < 1e-6
    # softplus(t) = t + ln(1 + e^-t): at t = 10 within 5e-5 of t
    assert abs(oracle.score(10.0) ** 2 - 10.0 - math.exp(-10.0)) < 5e-6


def test_score_monotone():
    z = np.linspace(-40, 40, 4001, dtype=np.float32)
    s = np.array([oracle.score(float(v)) for v in z])
    assert np.all(np.diff(s) >= 0)


# ------------------------------------------------------------------- routing

def test_routing_golden_cases():
    g = json.load(open(os.path.join(GOLDEN, "routing_cases.json")))
    for c in g["cases"]:
        n = len(c["logits"])
        cfg = oracle.make_cfg(256, 256, n, c["topk"], c["gate_temp"], c["norm_topk_prob"], c["route_scale"])
        w, idx, nan = oracle.route_from_logits(cfg, np.array([c["logits"]], np.float32), np.array(c["bias"], np.float32))
        assert nan == 0
        assert idx[0].tolist() == c["indices"], c["name"]
        expect = np.array(c["weights_num"]) / c["weights_den"]
        np.testing.assert_allclose(w[0], expect, rtol=3e-7, err_msg=c["name"])


def _random_cfg(n, k, norm=True):
    return oracle.make_cfg(256, 256, n, k, 1.0, norm, 1.5)


def test_routing_matches_brute_force_sort():
    rng = np.random.default_rng(2)
    n, k, m = 384, 6, 64
    z = rng.standard_normal((m, n)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, n).astype(np.float32)
    # force some exact ties of the keys
    z[:, 10] = z[:, 20]
    bias[10] = bias[20]
    w, idx, _ = oracle.route_from_logits(_random_cfg(n, k), z, bias)
    for t in range(m):
        s = np.array([oracle.score(float(v)) for v in z[t]], dtype=np.float32)
        key = (s + bias).astype(np.float32)
        order = np.lexsort((np.arange(n), -key.astype(np.float64)))  # key desc, then id asc
        assert idx[t].tolist() == order[:k].tolist()


def test_routing_weights_sum_to_route_scale_and_ignore_bias():
    rng = np.random.default_rng(3)
    n, k = 384, 6
    z = rng.standard_normal((32, n)).astype(np.float32) * 3
    bias = rng.uniform(-0.1, 0.1, n).astype(np.float32)
    cfg = _random_cfg(n, k)
    w, idx, _ = oracle.route_from_logits(cfg, z, bias)
    np.testing.assert_allclose(w.sum(axis=1), 1.5, rtol=2e-6)
    # a bias shift common to all experts keeps the picks and the weights
    w2, idx2, _ = oracle.route_from_logits(cfg, z, bias + np.float32(0.25))
    assert np.array_equal(idx, idx2)
    np.testing.assert_allclose(w, w2, rtol=0, atol=0)
    # the weights are the unbiased scores: ratios equal score ratios
    s0 = np.array([oracle.score(float(z[0, e])) for e in idx[0]])
    np.testing.assert_allclose(w[0] / w[0][0], s0 / s0[0], rtol=1e-6)


@pytest.mark.parametrize("sf", [oracle.SCORE_SQRTSOFTPLUS, oracle.SCORE_SIGMOID])
def test_routing_zero_scores_give_zero_weights(sf):
    """Logits of -inf score 0 under sqrt-softplus and sigmoid: the keys are the
    bias alone, and the weights are 0 / (0 + 1e-20) = 0, not 0 / 0 (the
    renormalisation of metrale moe_v41.rs fn route_from_logits)."""
    n, k = 12, 3
    z = np.full((1, n), -np.inf, np.float32)
    bias = np.linspace(-0.5, 0.6, n).astype(np.float32)[::-1].copy()
    w, idx, nan = oracle.route_from_logits(_cfg_sf(n, k, sf), z, bias)
    assert nan == 0
    assert idx[0].tolist() == [0, 1, 2]
    assert np.all(w == 0.0)


def test_routing_nan_key_ranks_last():
    n = 8
    z = np.arange(n, dtype=np.float32)[None, :] * 3
    z[0, 7] = np.nan
    w, idx, nan = oracle.route_from_logits(_random_cfg(n, 3), z, np.zeros(n, np.float32))
    assert nan == 1
    assert idx[0].tolist() == [6, 5, 4]


# ------------------------------------------- score-function and image-bias variants
# model.py Gate.forward (the atlas page): scores = linear(x, W) / gate_temp, then
# softmax over the experts, sigmoid, or sqrt(softplus); image tokens pick with bias_vl.

def _cfg_sf(n, k, sf, temp=1.0, norm=True):
    return oracle.make_cfg(256, 256, n, k, temp, norm, 1.5, 10.0, sf)


def _f32_ulp(v):
    return np.spacing(np.float32(abs(v)))


def test_sigmoid_score_closed_forms():
    c = _cfg_sf(8, 2, oracle.SCORE_SIGMOID)
    z = np.array([0.0, 40.0, -40.0, 2.0, -2.0, 1.0, 4.0, 0.5], np.float32)
    s = oracle.scores(c, z)
    assert s[0] == 0.5                                      # logistic(0)
    assert s[1] == 1.0                                      # 1 - e^-40 rounds to 1 in f32
    assert abs(s[2] / math.exp(-40.0) - 1) < 1e-6            # e^-40 / (1 + e^-40)
    assert abs((s[3] + s[4]) - 1.0) <= 2 * _f32_ulp(1.0)     # logistic(t) + logistic(-t) = 1
    assert abs(s[5] - SIGMA1) <= _f32_ulp(SIGMA1)
    # the temperature divides first: z / 2 = 0.5 at z = 1
    c2 = _cfg_sf(8, 2, oracle.SCORE_SIGMOID, temp=2.0)
    assert oracle.scores(c2, z)[5] == s[7]


def test_softmax_score_closed_forms():
    n = 16
    c = _cfg_sf(n, 2, oracle.SCORE_SOFTMAX)
    assert np.all(oracle.scores(c, np.full(n, 3.25, np.float32)) == np.float32(1.0 / n))
    # equal logits far beyond exp's range are still 1/n each (softmax is shift invariant)
    assert np.all(oracle.scores(c, np.full(n, 1000.0, np.float32)) == np.float32(1.0 / n))
    # one raised logit: e^a / (e^a + n - 1)
    z = np.zeros(n, np.float32)
    z[5] = 2.0
    s = oracle.scores(c, z)
    top = math.exp(2.0) / (math.exp(2.0) + n - 1)
    assert abs(s[5] - top) <= _f32_ulp(top)
    assert abs(s[0] - 1.0 / (math.exp(2.0) + n - 1)) <= _f32_ulp(s[0])
    # shift invariance on integer logits (the shifted t are exact): same bits
    zi = np.arange(n, dtype=np.float32) - 7
    assert np.array_equal(oracle.scores(c, zi), oracle.scores(c, zi + 5))
    # a NaN logit makes every softmax score NaN; all keys rank last, by id
    zn = zi.copy()
    zn[3] = np.nan
    w, idx, nan = oracle.route_from_logits(c, zn[None, :], np.zeros(n, np.float32))
    assert nan == n and idx[0].tolist() == [0, 1]


@pytest.mark.parametrize("sf", [1, 2])
def test_variant_scores_match_a_numpy_restatement(sf):
    """The f64 formulas restated with numpy: within one f32 ulp (the two exp
    implementations may differ in the last f64 bit)."""
    rng = np.random.default_rng(11 + sf)
    n = 384
    c = _cfg_sf(n, 6, sf, temp=0.7)
    for _ in range(8):
        z = (rng.standard_normal(n) * 3).astype(np.float32)
        t = (z / np.float32(0.7)).astype(np.float32).astype(np.float64)
        ref = 1.0 / (1.0 + np.exp(-t)) if sf == 1 else np.exp(t - t.max()) / np.sum(np.exp(t - t.max()))
        s = oracle.scores(c, z).astype(np.float64)
        assert np.all(np.abs(s - ref) <= np.spacing(ref.astype(np.float32)).astype(np.float64) + 1e-45)


@pytest.mark.parametrize("sf", [1, 2])
def test_variant_routing_matches_brute_force_sort(sf):
    rng = np.random.default_rng(5 + sf)
    n, k, m = 384, 6, 32
    z = rng.standard_normal((m, n)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, n).astype(np.float32) * (0.01 if sf == 2 else 1)
    c = _cfg_sf(n, k, sf)
    w, idx, _ = oracle.route_from_logits(c, z, bias)
    for t in range(m):
        s = oracle.scores(c, z[t])
        key = (s + bias).astype(np.float32)
        order = np.lexsort((np.arange(n), -key.astype(np.float64)))
        assert idx[t].tolist() == order[:k].tolist()
        g = s[order[:k]].astype(np.float32)
        expect = (g / (np.float32(g.astype(np.float64).sum()) + np.float32(1e-20))) * np.float32(1.5)
        np.testing.assert_allclose(w[t], expect, rtol=3e-7)
    np.testing.assert_allclose(w.sum(axis=1), 1.5, rtol=2e-6)


def test_image_tokens_pick_with_bias_vl():
    rng = np.random.default_rng(21)
    n, k, m = 64, 4, 12
    c = _cfg_sf(n, k, oracle.SCORE_SQRTSOFTPLUS)
    z = rng.standard_normal((m, n)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, n).astype(np.float32)
    w0, i0, _ = oracle.route_from_logits(c, z, bias)
    # no image token, or bias_vl equal to bias: nothing changes
    w1, i1, _ = oracle.route_from_logits(c, z, bias, bias.copy(), np.ones(m, np.uint8))
    w2, i2, _ = oracle.route_from_logits(c, z, bias, bias + 1, np.zeros(m, np.uint8))
    assert np.array_equal(i0, i1) and np.array_equal(i0, i2)
    assert np.array_equal(w0, w1) and np.array_equal(w0, w2)
    # a bias_vl that lifts experts 3, 17, 40, 41 makes the image tokens pick exactly them;
    # their weights are the raw scores of those picks (the bias never scales)
    bvl = np.zeros(n, np.float32)
    bvl[[3, 17, 40, 41]] = 100.0
    mask = np.zeros(m, np.uint8)
    mask[4:9] = 1
    w3, i3, _ = oracle.route_from_logits(c, z, bias, bvl, mask)
    for t in range(m):
        if mask[t]:
            assert sorted(i3[t].tolist()) == [3, 17, 40, 41]
            s = oracle.scores(c, z[t])[i3[t]]
            np.testing.assert_allclose(w3[t] / w3[t].sum(), s / s.sum(), rtol=1e-6)
        else:
            assert np.array_equal(i3[t], i0[t]) and np.array_equal(w3[t], w0[t])


def test_layer_image_tokens_equal_the_layer_with_bias_vl():
    w = _tiny().with_(m=6, image_frac=0.5)
    L = _tiny_layer(w)
    cfg = oracle.cfg_of(w)
    bvl = W.bias_vl_f32(w, 0) * np.float32(20)  # strong enough to change picks
    mask = W.image_mask(w, 0)
    r = oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"], L["experts"], w.shared_kind, *L["shared"],
                         bias_vl=bvl, image_mask=mask)
    plain = oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"], L["experts"], w.shared_kind, *L["shared"])
    vl = oracle.moe_layer(cfg, L["x"], L["router_w"], bvl, L["experts"], w.shared_kind, *L["shared"])
    for t in range(w.m):
        ref = vl if mask[t] else plain
        assert np.array_equal(r.topk_idx[t], ref.topk_idx[t])
        np.testing.assert_array_equal(r.out[t], ref.out[t])
    assert np.any(vl.topk_idx[mask == 1] != plain.topk_idx[mask == 1])


# -------------------------------------------------------------------- SwiGLU

SIGMA1 = 0.7310585786300049   # logistic(1)
SIGMA10 = 0.9999546021312976  # logistic(10)


def test_swiglu_clamps():
    # gate clamped from above only, up clamped on both sides (model.py Expert.forward)
    assert oracle.swiglu(15.0, 1.0, 10.0) == pytest.approx(10.0 * SIGMA10, rel=1e-15)
    assert oracle.swiglu(1.0, 50.0, 10.0) == pytest.approx(SIGMA1 * 10.0, rel=1e-15)
    assert oracle.swiglu(1.0, -50.0, 10.0) == pytest.approx(-SIGMA1 * 10.0, rel=1e-15)
    assert oracle.swiglu(0.0, 7.0, 10.0) == 0.0
    # no lower clamp on the gate: a very negative gate drives h to 0, not to -10*sigma(-10)*u
    assert abs(oracle.swiglu(-100.0, 5.0, 10.0)) < 1e-40
    # limit <= 0 disables the clamps
    assert oracle.swiglu(15.0, 50.0, 0.0) == pytest.approx(15.0 / (1 + math.exp(-15.0)) * 50.0, rel=1e-15)
    assert oracle.swiglu(1.0, 1.0, 10.0) == pytest.approx(SIGMA1, rel=1e-15)


# ------------------------------------------------------------- expert / layer

def _tiny():
    return W.WORKLOADS["tiny"]


def test_expert_reduces_to_integer_matmul():
    """d = 1, scale 1, min 0 and integer activations with a 127 in each block
    make the gate/up projections plain integer matrix products."""
    D, I = 512, 256
    rng = np.random.default_rng(4)
    cfg = oracle.make_cfg(D, I, 2, 1, swiglu_limit=0.0)
    qs1 = rng.integers(0, 256, (I, D // 256, 64), dtype=np.uint8)
    qs1[:, :, 0] = 0   # zero weight on every 32nd column (the columns holding the 127s)
    qs1[:, :, 32] = 0
    w1 = np.zeros((I, D // 256, 84), dtype=np.uint8)
    w1[:, :, 0:16] = 1
    w1[:, :, 16:80] = qs1
    w1[:, :, 81] = 0x3C
    Wint = oracle.dequant_matrix(2, w1, I, D)
    assert set(np.unique(Wint)) <= {0.0, 1.0, 2.0, 3.0}
    x = rng.integers(-1, 2, D).astype(np.float32)  # small g keeps h inside the fp16 scale range
    x[::32] = 127
    xq8 = oracle.quantize_q8_1(x)
    np.testing.assert_array_equal(oracle.dequant_q8_1(xq8, D), x)
    # gate == up == integer matmul; with no clamps h = g sigma(g) g
    g = Wint.astype(np.int64) @ x.astype(np.int64)
    w2 = np.zeros((D, I // 256, 110), dtype=np.uint8)  # all-zero down -> E = 0
    E, _ = oracle.expert_kquant(cfg, xq8, w1, w1, w2)
    assert np.all(E == 0)
    # now read h back through a down matrix that copies h[0] (one weight = 1)
    w2[:, :, 0:32] = 0xFF      # hb = 1 -> q = lo
    w2[:, :, 96:104] = 0x11    # scale code 33 -> s = 1
    w2[:, :, 104:108] = 0xAA
    w2[:, :, 109] = 0x3C       # d = 1
    w2[0, 0, 32] = 0x01        # element 0 of row 0: lo = 1; everything else lo = 0
    E, _ = oracle.expert_kquant(cfg, xq8, w1, w1, w2)
    h0 = float(g[0]) / (1 + math.exp(-float(g[0]))) * float(g[0])
    hq = oracle.quantize_q8_1(np.array([h0] + [oracle.swiglu(float(v), float(v), 0.0) for v in g[1:32]],
                                       dtype=np.float32))
    expect = oracle.dequant_q8_1(hq, 32)[0]
    assert E[0] == pytest.approx(expect, rel=1e-12)
    assert np.all(E[1:] == 0)


def test_expert_matches_dense_library_matmul():
    """The per-row oracle loops equal numpy matmuls over the dequantised
    matrices (catches a transposed operand or a dropped term)."""
    w = _tiny()
    cfg = oracle.cfg_of(w)
    w1, w3, w2 = W.expert_blocks(w, 0, 5)
    x = W.x_bf16(w, 0)[1]
    xf = np.array([oracle.bf16_value(int(v)) for v in x], dtype=np.float32)
    xq8 = oracle.quantize_q8_1(xf)
    xh = oracle.dequant_q8_1(xq8, w.dim)
    A1 = oracle.dequant_matrix(2, w1, w.inter, w.dim)
    A3 = oracle.dequant_matrix(2, w3, w.inter, w.dim)
    A2 = oracle.dequant_matrix(3, w2, w.dim, w.inter)
    g, u = A1 @ xh, A3 @ xh
    h = np.array([oracle.swiglu(a, b, w.swiglu_limit) for a, b in zip(g, u)], dtype=np.float32)
    hh = oracle.dequant_q8_1(oracle.quantize_q8_1(h), w.inter)
    E, _ = oracle.expert_kquant(cfg, xq8, w1, w3, w2)
    np.testing.assert_allclose(E, A2 @ hh, rtol=1e-12, atol=1e-12 * np.abs(A2 @ hh).max())


def test_router_logits_match_a_library_matmul():
    """z = x W_R^T on the bf16 values (the router step of the atlas page and
    model.py Gate.forward), against numpy's f64 matmul rounded to f32; the
    shapes differ in every dimension, so a transposed operand shows."""
    rng = np.random.default_rng(5)
    to_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x = to_bf16(rng.standard_normal((3, 256)))
    R = to_bf16(rng.standard_normal((7, 256)) / 16)
    f = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    z = oracle.router_logits(x, R)
    assert z.shape == (3, 7) and z.dtype == np.float32
    np.testing.assert_allclose(z, (f(x) @ f(R).T).astype(np.float32), rtol=2e-7, atol=0)


def test_shared_bf16_matches_dense_library_matmul():
    w = _tiny()
    cfg = oracle.cfg_of(w)
    s1, s3, s2 = W.shared_weights(w, 0)
    x = W.x_bf16(w, 0)[2]
    f = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    g, u = f(s1) @ f(x), f(s3) @ f(x)
    h = np.array([oracle.swiglu(a, b, w.swiglu_limit) for a, b in zip(g, u)], dtype=np.float32)
    hb = np.array([oracle.bf16_value(oracle.bf16_from_f32(v)) for v in h])
    S, _ = oracle.shared_bf16(cfg, x, s1, s3, s2)
    np.testing.assert_allclose(S, f(s2) @ hb, rtol=1e-12, atol=1e-13)


def _tiny_layer(w=None, layer=0):
    w = w or _tiny()
    return dict(x=W.x_bf16(w, layer), router_w=W.router_bf16(w, layer), bias=W.bias_f32(w, layer),
                experts=[W.expert_blocks(w, layer, e) for e in range(w.n_routed)],
                shared=W.shared_weights(w, layer))


def test_layer_is_weighted_sum_plus_shared():
    """out = sum_i G_i E_i + S (the atlas's y_routed + y_shared)."""
    w = _tiny()
    cfg = oracle.cfg_of(w)
    L = _tiny_layer(w)
    r = oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"], L["experts"], w.shared_kind, *L["shared"])
    z = oracle.router_logits(L["x"], L["router_w"])
    w_r, idx_r, _ = oracle.route_from_logits(cfg, z, L["bias"])
    assert np.array_equal(idx_r, r.topk_idx) and np.array_equal(w_r, r.topk_w)
    for t in range(w.m):
        xf = np.array([oracle.bf16_value(int(v)) for v in L["x"][t]], dtype=np.float32)
        xq8 = oracle.quantize_q8_1(xf)
        y = np.zeros(w.dim)
        for i, e in enumerate(idx_r[t]):
            E, _ = oracle.expert_kquant(cfg, xq8, *L["experts"][e])
            y += float(w_r[t, i]) * E
        S, _ = oracle.shared_bf16(cfg, L["x"][t], *L["shared"])
        np.testing.assert_allclose(r.out[t], y + S, rtol=1e-13, atol=1e-13)


def test_layer_zeroed_parts():
    """A zero down projection removes exactly that part of the output."""
    w = _tiny()
    cfg = oracle.cfg_of(w)
    L = _tiny_layer(w)
    full = oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"], L["experts"], 0, *L["shared"])
    zero_sh2 = np.zeros_like(L["shared"][2])
    routed = oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"], L["experts"], 0, L["shared"][0],
                              L["shared"][1], zero_sh2)
    zero_experts = [(a, b, np.zeros_like(c)) for a, b, c in L["experts"]]
    shared = oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"], zero_experts, 0, *L["shared"])
    np.testing.assert_allclose(full.out, routed.out + shared.out, rtol=1e-12, atol=1e-12)


def test_layer_token_subset_and_threads():
    w = _tiny().with_(m=6)
    cfg = oracle.cfg_of(w)
    L = _tiny_layer(w)
    a = oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"], L["experts"], 0, *L["shared"], nthreads=1)
    b = oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"], L["experts"], 0, *L["shared"], tokens=[4, 1],
                         nthreads=3)
    np.testing.assert_array_equal(b.out, a.out[[4, 1]])
    np.testing.assert_array_equal(b.topk_idx, a.topk_idx[[4, 1]])


def test_layer_missing_expert_is_an_error():
    w = _tiny()
    cfg = oracle.cfg_of(w)
    L = _tiny_layer(w)
    experts = list(L["experts"])
    z = oracle.router_logits(L["x"], L["router_w"])
    _, idx, _ = oracle.route_from_logits(cfg, z, L["bias"])
    experts[int(idx[0, 0])] = None
    with pytest.raises(RuntimeError):
        oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"], experts, 0, *L["shared"])


def test_clip_saturates_on_scaled_rows():
    """Rows scaled by 50 drive the SwiGLU clamps (the long-prefill workload's purpose)."""
    w = _tiny().with_(outlier_frac=0.25)
    cfg = oracle.cfg_of(w)
    L = _tiny_layer(w)
    rows = W.outlier_rows(w, 0)
    assert rows.size == 1
    r = oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"], L["experts"], 0, *L["shared"],
                         tokens=rows.tolist())
    assert r.clipped > 0


# --------------------------------------------------------------------- sizes

def test_parameter_accounting():
    """The atlas Parameters table: router 1,966,848; routed expert 35,389,440
    (x 384); shared 35,389,440; total 13,626,901,248 per instance."""
    w = W.WORKLOADS["decode_m1_40layer"]
    per_expert = 3 * w.dim * w.inter
    router = w.n_routed * w.dim + 2 * w.n_routed
    assert per_expert == 35_389_440
    assert router == 1_966_848
    assert router + (w.n_routed + 1) * per_expert == 13_626_901_248
    # the K-quant byte sizes stand for exactly those element counts
    assert w.w1_bytes // 84 * 256 == w.inter * w.dim
    assert w.w2_bytes // 110 * 256 == w.dim * w.inter
    assert w.expert_bytes == 12_810_240


@pytest.mark.parametrize("variant", ["base", "kquant_shared", "topk1_no_norm", "no_clip_temp", "sigmoid",
                                     "softmax", "image_tokens", "outliers", "ties"])
def test_layer_equals_the_brute_force_dense_layer(variant):
    """The factored oracle against its brute-force mode (every matrix
    dequantised to dense f64 up front, textbook loops over all tokens, the
    picks by k rounds of the best remaining key): equal to about 1e-12
    relative, picks and weights identical."""
    base = _tiny().with_(m=6)
    w = {"base": base, "kquant_shared": base.with_(shared_kind=W.SHARED_KQUANT),
         "topk1_no_norm": base.with_(topk=1, norm_topk_prob=False), "no_clip_temp": base.with_(
             swiglu_limit=0.0, gate_temp=0.6, route_scale=2.0), "sigmoid": base.with_(score_func=1),
         "softmax": base.with_(score_func=2), "image_tokens": base.with_(image_frac=0.5),
         "outliers": base.with_(outlier_frac=0.34), "ties": base}[variant]
    cfg = oracle.cfg_of(w)
    L = _tiny_layer(w)
    im = W.image_mask(w, 0)
    bv = None if im is None else W.bias_vl_f32(w, 0)
    gl = None
    if variant == "ties":  # equal logits on most experts: the tie rule decides the picks
        gl = np.full((w.m, w.n_routed), 0.25, dtype=np.float32)
        gl[:, 5] = 0.3
    a = oracle.moe_layer(cfg, L["x"], L["router_w"], L["bias"] * (0 if variant == "ties" else 1), L["experts"],
                         w.shared_kind, *L["shared"], given_logits=gl, bias_vl=bv, image_mask=im)
    b = oracle.moe_layer_dense(cfg, L["x"], L["router_w"], L["bias"] * (0 if variant == "ties" else 1),
                               L["experts"], w.shared_kind, *L["shared"], given_logits=gl, bias_vl=bv,
                               image_mask=im)
    np.testing.assert_array_equal(a.topk_idx, b.topk_idx)
    np.testing.assert_array_equal(a.topk_w, b.topk_w)
    scale = np.abs(a.out).max()
    np.testing.assert_allclose(b.out, a.out, rtol=1e-12, atol=1e-12 * scale)
    if variant == "ties":
        assert np.all(a.topk_idx[:, 0] == 5) and np.all(a.topk_idx[:, 1] == 0)
