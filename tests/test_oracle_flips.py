"""Pins of the oracle's requantisation flip candidates (reading C-F1 of
moe_oracle.c) and of the test helper that takes them.

The oracle lists, for one token, every q8_1 code, q8_1 block scale and bf16
value of h that gate and up projections known only to within
kappa * sum |terms| can change, with the change each makes to the output.
These tests restate the expert FFN in numpy (dequantised matrices, the
clipped SwiGLU, q8_1 and bf16 rounding written out here), move g and u by
random amounts inside that window, and check that the moved output differs
from the oracle's by exactly the changes of the candidates matching the codes
that moved, and that every moved code has its candidate."""
import numpy as np
import pytest

import oracle
import synth.workloads as W
from _helpers import take_flips

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _swiglu(g, u, L):
    """silu(min(g, L)) * clip(u, -L, L); no clamps for L <= 0."""
    if L > 0:
        g = np.minimum(g, L)
        u = np.clip(u, -L, L)
    return g / (1.0 + np.exp(-g)) * u


def _q8(h32):
    """q8_1 of an f32 vector: per block of 32, d = amax / 127 in f32, codes
    round-half-away(h / d) in f32, values fp16(d) * code."""
    hb = h32.reshape(-1, 32)
    amax = np.abs(hb).max(axis=1).astype(np.float32)
    d = (amax / np.float32(127)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (hb / d[:, None]).astype(np.float32)
    q = np.where(amax[:, None] == 0, 0, np.sign(v) * np.floor(np.abs(v) + np.float32(0.5)))
    d16 = d.astype(np.float16)
    return q.astype(np.int64), d16, (q * d16.astype(np.float64)[:, None]).reshape(-1), amax


def _bf16(h32):
    a = h32.astype(np.float32).view(np.uint32).astype(np.uint64)
    b = ((a + 0x7FFF + ((a >> 16) & 1)) >> 16).astype(np.uint16)
    return b, (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _f(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class _Token:
    """One token of a tiny workload, its experts dense in f64."""

    def __init__(self, w, t):
        self.w, self.t = w, t
        self.cfg = oracle.cfg_of(w)
        self.x = W.x_bf16(w, 0)
        self.experts = [W.expert_blocks(w, 0, e) for e in range(w.n_routed)]
        self.sh = W.shared_weights(w, 0)
        r = oracle.moe_layer(self.cfg, self.x, W.router_bf16(w, 0), W.bias_f32(w, 0), self.experts, w.shared_kind,
                             *self.sh, tokens=[t])
        self.ref, self.tw, self.ti = r.out[0], r.topk_w[0], r.topk_idx[0]
        xf = _f(self.x[t]).astype(np.float32)
        xh = oracle.dequant_q8_1(oracle.quantize_q8_1(xf), w.dim)
        self.slots = []   # (weight, A1, A3, A2, input, kquant)
        for e, g in zip(self.ti, self.tw):
            w1, w3, w2 = self.experts[e]
            self.slots.append((float(g), oracle.dequant_matrix(2, w1, w.inter, w.dim),
                               oracle.dequant_matrix(2, w3, w.inter, w.dim),
                               oracle.dequant_matrix(3, w2, w.dim, w.inter), xh, True))
        if w.shared_kind == W.SHARED_KQUANT:
            s1, s3, s2 = self.sh
            self.slots.append((1.0, oracle.dequant_matrix(2, s1, w.inter, w.dim),
                               oracle.dequant_matrix(2, s3, w.inter, w.dim),
                               oracle.dequant_matrix(3, s2, w.dim, w.inter), xh, True))
        else:
            s1, s3, s2 = self.sh
            self.slots.append((1.0, _f(s1), _f(s3), _f(s2), _f(self.x[t]), False))

    def gu(self, s):
        G, A1, A3, A2, xin, kq = self.slots[s]
        return A1 @ xin, A3 @ xin, np.abs(A1) @ np.abs(xin), np.abs(A3) @ np.abs(xin)

    def h32(self, s, dg=0.0, du=0.0):
        g, u, _, _ = self.gu(s)
        return _swiglu(g + dg, u + du, self.w.swiglu_limit).astype(np.float32)

    def output(self, hs):
        """sum over slots of weight * W2 (requantised h); hs[s] = f32 h."""
        y = np.zeros(self.w.dim)
        for s, (G, A1, A3, A2, xin, kq) in enumerate(self.slots):
            v = _q8(hs[s])[2] if kq else _bf16(hs[s])[1]
            y += G * (A2 @ v)
        return y

    def flips(self, kappa):
        return oracle.flip_candidates(self.cfg, self.x, self.t, self.tw, self.ti, self.experts, self.w.shared_kind,
                                      *self.sh, kappa, max_c=4096)


def _tiny(kind):
    return W.WORKLOADS["tiny"].with_(m=8, shared_kind=kind)


@pytest.mark.parametrize("t", [0, 5])
@pytest.mark.parametrize("kind", [W.SHARED_BF16, W.SHARED_KQUANT])
def test_numpy_restatement_is_the_oracle(kind, t):
    T = _Token(_tiny(kind), t)
    y = T.output([T.h32(s) for s in range(len(T.slots))])
    np.testing.assert_allclose(y, T.ref, rtol=0, atol=1e-12 * np.abs(T.ref).max())


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_q8_code_candidates_cover_every_moved_code(seed):
    """g, u moved inside the window, each block's largest |h| held (so its
    scale stays): the output moves by exactly the sum of the changes of the
    code candidates that match the moved codes."""
    kappa = 2.0 ** -12
    T = _Token(_tiny(W.SHARED_KQUANT), 3 + seed)
    F = T.flips(kappa)
    assert F.total < 4096
    cand = {(int(m[0]), int(m[2]), int(m[3])): i for i, m in enumerate(F.meta) if m[1] == oracle.FLIP_Q8_CODE}
    rng = np.random.default_rng(seed)
    hs, expect, moved = [], np.zeros(T.w.dim), 0
    for s in range(len(T.slots)):
        g, u, sg, su = T.gu(s)
        dg = kappa * sg * rng.uniform(-1, 1, g.shape)
        du = kappa * su * rng.uniform(-1, 1, u.shape)
        h0 = T.h32(s)
        q0, d0, _, a0 = _q8(h0)
        h = T.h32(s, dg, du)
        for b in range(h.size // 32):
            blk = slice(32 * b, 32 * b + 32)
            i0 = int(np.argmax(np.abs(h0[blk])))
            h[32 * b + i0] = h0[32 * b + i0]
            if np.abs(h[blk]).max() != a0[b]:
                h[blk] = h0[blk]   # another element overtook the largest: keep the block
        q1, d1, _, _ = _q8(h)
        assert np.array_equal(d1, d0)
        for b, i in zip(*np.nonzero(q1 != q0)):
            key = (s, 32 * int(b) + int(i), int(q1[b, i]))
            assert key in cand, f"moved code {key} has no candidate"
            expect += F.delta[cand[key]]
            moved += 1
        hs.append(h)
    assert moved > 10   # the window moves codes
    y = T.output(hs)
    np.testing.assert_allclose(y - T.ref, expect, rtol=0, atol=1e-9 * np.abs(T.ref).max())


@pytest.mark.parametrize("t", [1, 6])
def test_q8_scale_candidates(t):
    """The largest |h| of a block pushed to the far end of its window: where
    that changes fp16(d) there is a scale candidate for exactly that d, and
    its change is the output's."""
    kappa = 2.0 ** -16
    T = _Token(_tiny(W.SHARED_KQUANT), t)
    F = T.flips(kappa)
    scale = {(int(m[0]), int(m[2])): [] for m in F.meta}
    for i, m in enumerate(F.meta):
        if m[1] == oracle.FLIP_Q8_SCALE:
            scale.setdefault((int(m[0]), int(m[2])), []).append(i)
    L = T.w.swiglu_limit
    seen = 0
    for s in range(len(T.slots)):
        g, u, sg, su = T.gu(s)
        h0 = T.h32(s)
        q0, d0, _, a0 = _q8(h0)
        for b in range(h0.size // 32):
            i0 = 32 * b + int(np.argmax(np.abs(h0[32 * b:32 * b + 32])))
            dg, du = kappa * sg[i0], kappa * su[i0]
            corners = [_swiglu(g[i0] + a, u[i0] + c, L) for a in (-dg, dg) for c in (-du, du)]
            far = np.float32(max(corners, key=abs))
            h = h0.copy()
            h[i0] = far
            if np.abs(h[32 * b:32 * b + 32]).max() != abs(far):
                continue
            _, d1, _, _ = _q8(h)
            if d1[b] == d0[b]:
                continue
            alts = [int(F.meta[i][3]) for i in scale.get((s, b), [])]
            want = int(np.float16(d1[b]).view(np.uint16))
            assert want in alts, f"slot {s} block {b}: fp16(d) {want:#x} not among {alts}"
            i = scale[(s, b)][alts.index(want)]
            hs = [T.h32(k) for k in range(len(T.slots))]
            hs[s] = h
            np.testing.assert_allclose(T.output(hs) - T.ref, F.delta[i], rtol=0, atol=1e-9 * np.abs(T.ref).max())
            seen += 1
    assert seen > 0


@pytest.mark.parametrize("seed", [0, 1])
def test_bf16_candidates_cover_every_moved_value(seed):
    """The bf16 shared expert: g, u moved inside the window; every bf16
    value of h that moved has its candidate and the output moves by the sum of
    their changes."""
    kappa = 2.0 ** -14
    T = _Token(_tiny(W.SHARED_BF16), 2 + seed)
    F = T.flips(kappa)
    k = len(T.slots) - 1
    cand = {(int(m[2]), int(m[3])): i for i, m in enumerate(F.meta) if m[1] == oracle.FLIP_BF16}
    assert all(int(m[0]) == k for m in F.meta if m[1] == oracle.FLIP_BF16)
    rng = np.random.default_rng(10 + seed)
    g, u, sg, su = T.gu(k)
    # only elements whose window holds at most 16 bf16 values move (a wider
    # one, around h = 0, lists its two ends only)
    L = T.w.swiglu_limit
    gs = -1.2784645427610738   # the minimum of silu
    gstar = np.where(np.abs(g - gs) < kappa * sg, gs, g - kappa * sg)
    corners = np.stack([_swiglu(g + a * kappa * sg, u + c * kappa * su, L) for a in (-1, 1) for c in (-1, 1)] +
                       [_swiglu(gstar, u + c * kappa * su, L) for c in (-1, 1)])
    key = lambda b: np.where(b & 0x8000, -(b.astype(np.int64) & 0x7FFF), b.astype(np.int64))
    span = key(_bf16(corners.max(axis=0).astype(np.float32))[0]) - key(_bf16(corners.min(axis=0).astype(np.float32))[0])
    narrow = span <= 16
    assert narrow.mean() > 0.9
    h = T.h32(k, narrow * kappa * sg * rng.uniform(-1, 1, g.shape), narrow * kappa * su * rng.uniform(-1, 1, u.shape))
    b0, _ = _bf16(T.h32(k))
    b1, _ = _bf16(h)
    expect = np.zeros(T.w.dim)
    moved = np.nonzero(b0 != b1)[0]
    assert moved.size > 3
    for j in moved:
        assert (int(j), int(b1[j])) in cand, f"moved bf16 value of h[{j}] has no candidate"
        expect += F.delta[cand[(int(j), int(b1[j]))]]
    hs = [T.h32(s) for s in range(k)] + [h]
    np.testing.assert_allclose(T.output(hs) - T.ref, expect, rtol=0, atol=1e-9 * np.abs(T.ref).max())


def test_no_window_no_candidates():
    T = _Token(_tiny(W.SHARED_KQUANT), 0)
    assert T.flips(0.0).total == 0


def test_take_flips_recovers_a_planted_subset():
    """Output changes as random columns; an error made of a subset of them
    plus noise well below their size gives back exactly that subset."""
    rng = np.random.default_rng(7)
    delta = rng.standard_normal((200, 2048)) * rng.uniform(0.5, 2.0, (200, 1))
    pick = rng.choice(200, 12, replace=False)
    resid = delta[pick].sum(axis=0) + 1e-3 * rng.standard_normal(2048)
    rest, used = take_flips(resid, delta)
    assert sorted(used) == sorted(pick.tolist())
    assert np.abs(rest).max() < 1e-2
    # an error no candidate explains takes none
    rest, used = take_flips(rng.standard_normal(2048) * 0.05, delta)
    assert used == []
