"""The bench line's accounting on the CPU: algorithmic bytes and flops per
layer call worked out by hand from the block formats and the layer's shapes,
the bound each workload takes, and the rule that a recorded DRAM traffic
figure is used only while the kernel sources it was taken on are unchanged."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import synth.workloads as W  # noqa: E402

D, I, N, K = 5120, 2304, 384, 6
Q2K_BYTES, Q3K_BYTES = 84, 110  # bytes per 256-value super-block
EXPERT = 2 * I * (D // 256) * Q2K_BYTES + D * (I // 256) * Q3K_BYTES  # W1, W3 (Q2_K) + W2 (Q3_K)


def test_expert_bytes_from_the_block_formats():
    assert EXPERT == 12_810_240
    assert W.WORKLOADS["decode_m1_40layer"].expert_bytes == EXPERT


def test_decode_call_bytes_and_flops():
    w = W.WORKLOADS["decode_m1_40layer"]
    router = N * D * 2 + N * 4          # bf16 W_R and the f32 bias
    shared = 3 * D * I * 2              # bf16 shared expert
    io = D * 2 + D * 4                  # x in (bf16), out (f32)
    assert bench.algorithmic_bytes(w, K) == router + K * EXPERT + shared + io == 151_604_736
    # router GEMV + 3 projections per picked expert + the shared expert's 3
    assert bench.algorithmic_flops(w) == 2 * N * D + 2 * K * 3 * D * I + 2 * 3 * D * I == 499_384_320


def test_prefill_call_bytes_and_flops():
    w = W.WORKLOADS["prefill_m4096_outliers"]
    m = 4096
    assert bench.algorithmic_bytes(w, N) == (N * D * 2 + N * 4) + N * EXPERT + 3 * D * I * 2 + m * D * 6
    assert bench.algorithmic_bytes(w, N) == pytest.approx(5.12e9, rel=1e-3)
    flops = 2 * m * N * D + 2 * m * K * 3 * D * I + 2 * m * 3 * D * I
    assert bench.algorithmic_flops(w) == flops == 2_045_478_174_720


def test_decode_is_byte_bound_and_long_prefill_tensor_bound():
    hbm, tfs, _, _ = bench.peaks()
    d = bench.roofline(W.WORKLOADS["decode_m1_40layer"], K, 0.0636, "k", None)
    assert d["bound"] == "hbm" and d["unit"] == "GB/s"
    assert d["achieved"] == pytest.approx(151_604_736 / 63.6e-6 / 1e9)
    assert d["frac"] == pytest.approx(d["achieved"] / hbm)
    p = bench.roofline(W.WORKLOADS["prefill_m4096_outliers"], N, 7.74, "k", None)
    assert p["bound"] == "tensor" and p["unit"] == "TFLOP/s"
    assert p["frac"] == pytest.approx(2_045_478_174_720 / 7.74e-3 / 1e12 / tfs)
    assert p["bound_us"] == pytest.approx(2_045_478_174_720 / (tfs * 1e12) * 1e6)


def test_recorded_traffic_only_on_matching_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic_decode_m1_40layer.txt").write_text(
        "# a comment line\nsources_sha256_16: 0123456789abcdef\ndram_bytes_per_layer_call: 154766080\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "sources_hash", lambda kind: "0123456789abcdef" if kind == "decode" else "x")
    assert bench.recorded_traffic("decode_m1_40layer") == 154766080.0
    monkeypatch.setattr(bench, "sources_hash", lambda kind: "fedcba9876543210")
    assert bench.recorded_traffic("decode_m1_40layer") is None
    assert bench.recorded_traffic("prefill_m4096_outliers") is None  # no file


def test_sources_hash_covers_each_family():
    for kind in ("decode", "prefill"):
        h = bench.sources_hash(kind)
        assert len(h) == 16 and int(h, 16) >= 0
    assert "common.cuh" in bench.KERNEL_SOURCES["decode"] and "k_prefill_kq.cu" in bench.KERNEL_SOURCES["prefill"]
