"""The five seeded synthetic MoE-layer workloads and their input recipes.

Shapes follow the DeepSeek V4.1 configuration (dim 5120, moe_inter_dim 2304,
384 routed experts, 6 active, route_scale 1.5, swiglu_limit 10) from the
open-model-atlas page "DeepSeek V4.1 · Mixture of experts" (config.json
listing); the tiny workload shrinks every size.  No public dataset is
involved: every tensor is drawn by this package's counter-based generator.

Recipe (all workloads):
  x       bf16 N(0,1) [m, dim]; in the long-prefill workload ceil(1% of m)
          rows (the first of a seeded permutation) are scaled by 50 before
          rounding to bf16.
  router  bf16 N(0, sigma^2), sigma = 1/sqrt(dim), [n_routed, dim].
  bias    f32 U(-0.1, 0.1) [n_routed]; in the hot-expert workload the first
          32 experts of a seeded permutation get +0.5 (added in f32).
  W1, W3  Q2_K [inter rows][dim/256 blocks]; scale/min nibbles, 2-bit quants
          uniform; fp16 d, dmin ~ U(1e-3, 4e-3).
  W2      Q3_K [dim rows][inter/256 blocks]; hmask bits, low quants, six-bit
          scale codes uniform; fp16 d ~ U(5e-4, 2e-3).
  shared  bf16 N(0, 0.02^2) w1 [inter, dim], w3 [inter, dim], w2 [dim, inter];
          or, in the m=8 workload, K-quant blocks drawn like the routed ones.
  vision  (variants only) bias_vl f32 U(-0.1, 0.1) [n_routed] and an image
          span: round(image_frac * m) consecutive tokens from a seeded start.
Layer l of a workload draws every tensor from the stream key
(seed, layer=l, tensor id, expert).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import (Q2K_BYTES, Q3K_BYTES, T_BIAS, T_BIAS_VL, T_HOT, T_IMAGE, T_OUTLIER, T_ROUTER, T_SH1, T_SH2, T_SH3,
               T_W1, T_W2, T_W3, T_X, key, normal_bf16, permutation, q2k_blocks, q3k_blocks, uniform_f32)

SHARED_BF16 = 0
SHARED_KQUANT = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dim: int
    inter: int
    n_routed: int
    topk: int
    m: int
    layers: int = 1
    shared_kind: int = SHARED_BF16
    hot_experts: int = 0
    hot_bias: float = 0.5
    outlier_frac: float = 0.0
    outlier_scale: float = 50.0
    gate_temp: float = 1.0
    norm_topk_prob: bool = True
    route_scale: float = 1.5
    swiglu_limit: float = 10.0
    seed: int = 0
    score_func: int = 0          # 0 sqrt-softplus, 1 sigmoid, 2 softmax (model.py Gate.forward)
    image_frac: float = 0.0      # share of the tokens inside an image span (they pick with bias_vl)

    # --- sizes of the raw expert blocks ---
    @property
    def w1_bytes(self) -> int:
        return self.inter * (self.dim // 256) * Q2K_BYTES

    @property
    def w2_bytes(self) -> int:
        return self.dim * (self.inter // 256) * Q3K_BYTES

    @property
    def expert_bytes(self) -> int:
        """one routed expert: w1 + w3 (Q2_K) + w2 (Q3_K)"""
        return 2 * self.w1_bytes + self.w2_bytes

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", dim=512, inter=256, n_routed=16, topk=2, m=4),
    "decode_m1_40layer": Workload("decode_m1_40layer", dim=5120, inter=2304, n_routed=384, topk=6, m=1,
                                  layers=40),
    "decode_m8_kquant_shared": Workload("decode_m8_kquant_shared", dim=5120, inter=2304, n_routed=384, topk=6,
                                        m=8, shared_kind=SHARED_KQUANT),
    "prefill_m512_hot": Workload("prefill_m512_hot", dim=5120, inter=2304, n_routed=384, topk=6, m=512,
                                 hot_experts=32),
    "prefill_m4096_outliers": Workload("prefill_m4096_outliers", dim=5120, inter=2304, n_routed=384, topk=6,
                                       m=4096, outlier_frac=0.01),
}
ORDER = ["tiny", "decode_m1_40layer", "decode_m8_kquant_shared", "prefill_m512_hot", "prefill_m4096_outliers"]


def outlier_rows(w: Workload, layer: int) -> np.ndarray:
    if w.outlier_frac <= 0:
        return np.zeros(0, dtype=np.int32)
    n = int(math.ceil(w.outlier_frac * w.m))
    return np.sort(permutation(w.m, key(w.seed, layer, T_OUTLIER))[:n])


def hot_experts(w: Workload, layer: int) -> np.ndarray:
    if w.hot_experts <= 0:
        return np.zeros(0, dtype=np.int32)
    return np.sort(permutation(w.n_routed, key(w.seed, layer, T_HOT))[: w.hot_experts])


def row_scale(w: Workload, layer: int) -> np.ndarray | None:
    rows = outlier_rows(w, layer)
    if rows.size == 0:
        return None
    s = np.ones(w.m, dtype=np.float64)
    s[rows] = w.outlier_scale
    return s


def x_bf16(w: Workload, layer: int) -> np.ndarray:
    return normal_bf16((w.m, w.dim), key(w.seed, layer, T_X), 1.0, row_scale(w, layer))


def router_bf16(w: Workload, layer: int) -> np.ndarray:
    return normal_bf16((w.n_routed, w.dim), key(w.seed, layer, T_ROUTER), 1.0 / math.sqrt(w.dim))


def bias_f32(w: Workload, layer: int) -> np.ndarray:
    b = uniform_f32(w.n_routed, key(w.seed, layer, T_BIAS), -0.1, 0.1)
    hot = hot_experts(w, layer)
    if hot.size:
        b[hot] = b[hot] + np.float32(w.hot_bias)
    return b


def bias_vl_f32(w: Workload, layer: int) -> np.ndarray:
    """the bias image tokens pick with"""
    return uniform_f32(w.n_routed, key(w.seed, layer, T_BIAS_VL), -0.1, 0.1)


def image_mask(w: Workload, layer: int) -> np.ndarray | None:
    """uint8 [m]: 1 for the tokens of the image span; None without one"""
    n = int(round(w.image_frac * w.m))
    if n <= 0:
        return None
    start = int(permutation(w.m - n + 1, key(w.seed, layer, T_IMAGE))[0])
    mask = np.zeros(w.m, dtype=np.uint8)
    mask[start:start + n] = 1
    return mask


def expert_blocks(w: Workload, layer: int, e: int):
    """(w1, w3, w2) raw bytes of routed expert e."""
    nb1 = w.inter * (w.dim // 256)
    nb2 = w.dim * (w.inter // 256)
    return (q2k_blocks(nb1, key(w.seed, layer, T_W1, e)),
            q2k_blocks(nb1, key(w.seed, layer, T_W3, e)),
            q3k_blocks(nb2, key(w.seed, layer, T_W2, e)))


def shared_weights(w: Workload, layer: int):
    """(w1, w3, w2): bf16 bits [inter,dim], [inter,dim], [dim,inter], or K-quant bytes."""
    if w.shared_kind == SHARED_BF16:
        return (normal_bf16((w.inter, w.dim), key(w.seed, layer, T_SH1), 0.02),
                normal_bf16((w.inter, w.dim), key(w.seed, layer, T_SH3), 0.02),
                normal_bf16((w.dim, w.inter), key(w.seed, layer, T_SH2), 0.02))
    nb1 = w.inter * (w.dim // 256)
    nb2 = w.dim * (w.inter // 256)
    return (q2k_blocks(nb1, key(w.seed, layer, T_SH1)),
            q2k_blocks(nb1, key(w.seed, layer, T_SH3)),
            q3k_blocks(nb2, key(w.seed, layer, T_SH2)))
