"""The seeded input generator: deterministic, thread-count independent, and
drawing the distributions the workload recipes state."""
import ctypes

import numpy as np

import synth
import synth.workloads as W


def test_counter_based_and_thread_independent():
    k = synth.key(0, 3, synth.T_X)
    a = synth.normal_bf16((64, 512), k, 1.0)
    n = 64 * 512
    b = np.empty(n, dtype=np.uint16)
    synth.host_lib().syn_fill_normal_bf16(b.ctypes.data, n, 512, k, 1.0, None, 1)
    np.testing.assert_array_equal(a.ravel(), b)
    # element i depends on (key, i) only: a slice of a bigger fill is the same
    q_all = synth.q2k_blocks(10, k)
    q_tail = synth.q2k_blocks(4, k, block0=6)
    np.testing.assert_array_equal(q_all[6 * 84:], q_tail)


def test_streams_differ():
    assert synth.key(0, 0, synth.T_W1, 1) != synth.key(0, 0, synth.T_W1, 2)
    assert synth.key(0, 0, synth.T_W1, 1) != synth.key(0, 1, synth.T_W1, 1)
    assert synth.key(0, 0, synth.T_W1, 1) != synth.key(0, 0, synth.T_W3, 1)


def test_normal_and_uniform_moments():
    f = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    x = f(synth.normal_bf16((1 << 18,), synth.key(1, 0, synth.T_X), 1.0))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    u = synth.uniform_f32(1 << 16, synth.key(1, 0, synth.T_BIAS), -0.1, 0.1)
    assert u.min() >= -0.1 and u.max() < 0.1 and abs(u.mean()) < 2e-3


def test_kquant_fields():
    blk = synth.q2k_blocks(4096, synth.key(2, 0, synth.T_W1)).reshape(-1, 84)
    d = blk[:, 80:82].copy().view(np.float16).astype(np.float64).ravel()
    dm = blk[:, 82:84].copy().view(np.float16).astype(np.float64).ravel()
    for v in (d, dm):
        assert v.min() >= 1e-3 * (1 - 1e-3) and v.max() <= 4e-3 * (1 + 1e-3)
    nib = np.concatenate([blk[:, :16] & 15, blk[:, :16] >> 4]).ravel()
    assert np.bincount(nib, minlength=16).min() > 0.9 * nib.size / 16
    b3 = synth.q3k_blocks(4096, synth.key(2, 0, synth.T_W2)).reshape(-1, 110)
    d3 = b3[:, 108:110].copy().view(np.float16).astype(np.float64).ravel()
    assert d3.min() >= 5e-4 * (1 - 1e-3) and d3.max() <= 2e-3 * (1 + 1e-3)


def test_half_bits_is_correctly_rounded():
    rng = np.random.default_rng(0)
    for v in np.concatenate([rng.uniform(1e-3, 4e-3, 2000), rng.uniform(-70000, 70000, 2000),
                             rng.uniform(-1e-6, 1e-6, 2000)]):
        assert synth.half_bits(v) == int(np.array([v]).astype(np.float16).view(np.uint16)[0])


def test_permutation_and_workload_recipes():
    p = synth.permutation(1000, synth.key(0, 0, synth.T_HOT))
    assert sorted(p.tolist()) == list(range(1000))
    hot = W.hot_experts(W.WORKLOADS["prefill_m512_hot"], 0)
    assert hot.size == 32 and len(set(hot.tolist())) == 32
    b = W.bias_f32(W.WORKLOADS["prefill_m512_hot"], 0)
    assert np.all(b[hot] > 0.39) and np.sum(b > 0.39) == 32
    rows = W.outlier_rows(W.WORKLOADS["prefill_m4096_outliers"], 0)
    assert rows.size == 41
    w = W.WORKLOADS["prefill_m4096_outliers"].with_(m=4096, dim=256)
    x = W.x_bf16(w, 0)
    f = (x.astype(np.uint32) << 16).view(np.float32)
    big = np.abs(f).max(axis=1)
    assert set(np.nonzero(big > 12)[0].tolist()) <= set(rows.tolist())
    assert np.median(big[rows]) > 50
