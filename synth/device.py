"""Device staging of the synthetic workloads: torch buffers for one layer's
inputs and the per-expert slot-pointer table.

Holds none of the method's arithmetic.  Small tensors are drawn on the host
and copied; the K-quant experts of the full-size workloads (~4.9 GB per
layer) are drawn directly on the GPU by the generator's CUDA twin, which
writes the same bytes as the host generator.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

from . import (Q2K_BYTES, Q3K_BYTES, T_ROUTER, T_SH1, T_SH2, T_SH3, T_W1, T_W2, T_W3, T_X, gpu_lib, key)
from .workloads import (SHARED_BF16, Workload, bias_f32, bias_vl_f32, expert_blocks, image_mask, router_bf16,
                        row_scale, shared_weights, x_bf16)

ALIGN = 256


def _a(n: int) -> int:
    return (n + ALIGN - 1) // ALIGN * ALIGN


def slot_layout(w: Workload):
    """byte offsets of w1, w3, w2 inside one expert slot, and the slot size"""
    o1 = 0
    o3 = _a(w.w1_bytes)
    o2 = o3 + _a(w.w1_bytes)
    return o1, o3, o2, _a(o2 + w.w2_bytes)


@dataclass
class DeviceLayer:
    w: Workload
    layer: int
    x: torch.Tensor            # bf16 bits as int16 [m, dim]
    router_w: torch.Tensor     # int16 [n_routed, dim]
    bias: torch.Tensor         # f32 [n_routed]
    experts: torch.Tensor      # uint8 [n_routed, slot]
    expert_ptrs: torch.Tensor  # int64 [n_routed, 3] device addresses
    sh1: torch.Tensor
    sh3: torch.Tensor
    sh2: torch.Tensor
    bias_vl: torch.Tensor | None = None     # f32 [n_routed]: the bias of image tokens
    image_mask: torch.Tensor | None = None  # uint8 [m]: 1 for image tokens


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with CUDA error {rc}")


def fill_experts_gpu(w: Workload, layer: int, buf: torch.Tensor) -> None:
    """Draw the routed experts 0..buf.shape[0]-1 of a layer into buf [slots, slot] on the GPU."""
    o1, o3, o2, slot = slot_layout(w)
    nb1 = w.inter * (w.dim // 256)
    nb2 = w.dim * (w.inter // 256)
    _check(gpu_lib().syn_gpu_fill_experts(buf.data_ptr(), buf.shape[0], slot, o1, o3, o2, nb1, nb2, w.seed, layer,
                                          _stream()), "fill experts")


def fill_experts_host(w: Workload, layer: int, buf: torch.Tensor, experts=None) -> None:
    """Copy host-drawn experts (all of them, or the given list) into buf."""
    o1, o3, o2, slot = slot_layout(w)
    host = torch.zeros((w.n_routed, slot), dtype=torch.uint8)
    for e in range(w.n_routed):
        blocks = experts[e] if experts is not None else expert_blocks(w, layer, e)
        if blocks is None:
            continue
        w1, w3, w2 = blocks
        host[e, o1:o1 + w.w1_bytes] = torch.from_numpy(w1)
        host[e, o3:o3 + w.w1_bytes] = torch.from_numpy(w3)
        host[e, o2:o2 + w.w2_bytes] = torch.from_numpy(w2)
    buf.copy_(host.to(buf.device))


def pointer_table(w: Workload, buf: torch.Tensor) -> torch.Tensor:
    """[n_routed, 3] device addresses; with fewer slots than experts, expert e
    uses slot e % slots (a profiling aid: same bytes per call, fewer held)."""
    o1, o3, o2, slot = slot_layout(w)
    base = buf.data_ptr()
    slots = buf.shape[0]
    t = torch.empty((w.n_routed, 3), dtype=torch.int64)
    for e in range(w.n_routed):
        s = e % slots
        t[e, 0] = base + s * slot + o1
        t[e, 1] = base + s * slot + o3
        t[e, 2] = base + s * slot + o2
    return t.to(buf.device)


def _bits_to_dev(a: np.ndarray, device) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def fill_normal_bf16_gpu(t: torch.Tensor, k: int, std: float, cols: int, rs: torch.Tensor | None = None) -> None:
    _check(gpu_lib().syn_gpu_fill_normal_bf16(t.data_ptr(), t.numel(), cols, k, std,
                                              None if rs is None else rs.data_ptr(), _stream()), "fill normal")


def stage_layer(w: Workload, layer: int, device="cuda", experts_on_gpu: bool = True,
                bulk_on_gpu: bool = False, slots: int = 0) -> DeviceLayer:
    """All of one layer's inputs on the device.

    experts_on_gpu: draw the routed experts with the GPU twin (else host).
    bulk_on_gpu: also draw the bf16 shared expert and the router on the GPU
    (fast; bytes can differ from the host draw in rare last-ulp cases, so
    parity tests keep it off).
    slots: expert slots held (default n_routed); fewer slots alias experts.
    """
    o1, o3, o2, slot = slot_layout(w)
    slots = slots or w.n_routed
    experts = torch.empty((slots, slot), dtype=torch.uint8, device=device)
    if experts_on_gpu:
        fill_experts_gpu(w, layer, experts)
    else:
        assert slots == w.n_routed
        fill_experts_host(w, layer, experts)
    ptrs = pointer_table(w, experts)
    x = _bits_to_dev(x_bf16(w, layer), device)
    bias = torch.from_numpy(bias_f32(w, layer)).to(device)
    if bulk_on_gpu:
        router = torch.empty((w.n_routed, w.dim), dtype=torch.int16, device=device)
        fill_normal_bf16_gpu(router, key(w.seed, layer, T_ROUTER), 1.0 / math.sqrt(w.dim), w.dim)
    else:
        router = _bits_to_dev(router_bf16(w, layer), device)
    if w.shared_kind == SHARED_BF16 and bulk_on_gpu:
        sh1 = torch.empty((w.inter, w.dim), dtype=torch.int16, device=device)
        sh3 = torch.empty((w.inter, w.dim), dtype=torch.int16, device=device)
        sh2 = torch.empty((w.dim, w.inter), dtype=torch.int16, device=device)
        fill_normal_bf16_gpu(sh1, key(w.seed, layer, T_SH1), 0.02, w.dim)
        fill_normal_bf16_gpu(sh3, key(w.seed, layer, T_SH3), 0.02, w.dim)
        fill_normal_bf16_gpu(sh2, key(w.seed, layer, T_SH2), 0.02, w.inter)
    else:
        s1, s3, s2 = shared_weights(w, layer)
        sh1, sh3, sh2 = (_bits_to_dev(a, device) for a in (s1, s3, s2))
    bias_vl = mask = None
    im = image_mask(w, layer)
    if im is not None:
        bias_vl = torch.from_numpy(bias_vl_f32(w, layer)).to(device)
        mask = torch.from_numpy(im).to(device)
    return DeviceLayer(w, layer, x, router, bias, experts, ptrs, sh1, sh3, sh2, bias_vl, mask)


def x_gpu(w: Workload, layer: int, out: torch.Tensor) -> None:
    """x of a layer drawn on the GPU (for timing loops that need many layers)."""
    rs = row_scale(w, layer)
    rs_t = None if rs is None else torch.from_numpy(rs).to(out.device)
    fill_normal_bf16_gpu(out, key(w.seed, layer, T_X), 1.0, w.dim, rs_t)
