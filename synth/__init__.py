"""Seeded synthetic inputs for the MoE-layer workloads.

This module is the only code that both sides of a parity check share: it
draws the inputs (activations, router, bias, K-quant expert blocks, shared
expert) and holds none of the method's arithmetic.  The host fill lives in
``synth.c`` and the GPU bulk fill in ``synth_gpu.cu``; both are built by
``synth.build.build()``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "_lib")
HOST_SO = os.path.join(_LIBDIR, "libsynth_host.so")
GPU_SO = os.path.join(_LIBDIR, "libsynth_gpu.so")

# tensor ids, mirroring synth_core.h
T_X, T_ROUTER, T_BIAS, T_W1, T_W3, T_W2, T_SH1, T_SH3, T_SH2, T_OUTLIER, T_HOT, T_BIAS_VL, T_IMAGE = range(1, 14)

Q2K_BYTES = 84   # bytes per Q2_K super-block of 256 weights
Q3K_BYTES = 110  # bytes per Q3_K super-block of 256 weights

_host = None
_gpu = None


def _threads() -> int:
    return max(1, min(os.cpu_count() or 1, 64))


def host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_SO):
            raise RuntimeError(f"{HOST_SO} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(HOST_SO)
        u64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.syn_stream_key.restype = u64
        lib.syn_stream_key.argtypes = [u64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
        lib.syn_draw_u64.restype = u64
        lib.syn_draw_u64.argtypes = [u64, u64]
        lib.syn_half_bits.restype = ctypes.c_uint16
        lib.syn_half_bits.argtypes = [dbl]
        lib.syn_fill_normal_bf16.argtypes = [vp, u64, u64, u64, dbl, vp, i32]
        lib.syn_fill_uniform_f32.argtypes = [vp, u64, u64, dbl, dbl, i32]
        lib.syn_fill_q2k.argtypes = [vp, u64, u64, u64, dbl, dbl, i32]
        lib.syn_fill_q3k.argtypes = [vp, u64, u64, u64, dbl, dbl, i32]
        lib.syn_permutation.argtypes = [vp, ctypes.c_int32, u64]
        _host = lib
    return _host


def gpu_lib():
    global _gpu
    if _gpu is None:
        if not os.path.exists(GPU_SO):
            raise RuntimeError(f"{GPU_SO} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(GPU_SO)
        u64, dbl, vp = ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
        lib.syn_gpu_fill_q2k.argtypes = [vp, u64, u64, u64, dbl, dbl, vp]
        lib.syn_gpu_fill_q3k.argtypes = [vp, u64, u64, u64, dbl, dbl, vp]
        lib.syn_gpu_fill_normal_bf16.argtypes = [vp, u64, u64, u64, dbl, vp, vp]
        lib.syn_gpu_fill_uniform_f32.argtypes = [vp, u64, u64, dbl, dbl, vp]
        lib.syn_gpu_fill_experts.argtypes = [vp, ctypes.c_uint32, u64, u64, u64, u64, u64, u64, u64,
                                             ctypes.c_uint32, vp]
        lib.syn_gpu_fill_experts.restype = ctypes.c_int
        for f in ("syn_gpu_fill_q2k", "syn_gpu_fill_q3k", "syn_gpu_fill_normal_bf16", "syn_gpu_fill_uniform_f32"):
            getattr(lib, f).restype = ctypes.c_int
        _gpu = lib
    return _gpu


def key(seed: int, layer: int, tensor: int, expert: int = 0) -> int:
    return int(host_lib().syn_stream_key(seed, layer, tensor, expert))


def draw(k: int, i: int) -> int:
    return int(host_lib().syn_draw_u64(k, i))


def half_bits(v: float) -> int:
    """IEEE binary16 bits of v (round to nearest even): the generator's fp16 field writer."""
    return int(host_lib().syn_half_bits(float(v)))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def normal_bf16(shape, k: int, std: float, row_scale: np.ndarray | None = None) -> np.ndarray:
    """bf16 bits (uint16) of std * row_scale[row] * N(0,1), element i from draws 2i, 2i+1."""
    shape = tuple(shape)
    n = int(np.prod(shape))
    cols = shape[-1] if len(shape) > 1 else 1
    out = np.empty(n, dtype=np.uint16)
    rs = None
    if row_scale is not None:
        rs = np.ascontiguousarray(row_scale, dtype=np.float64)
    host_lib().syn_fill_normal_bf16(_ptr(out), n, cols, k, std, None if rs is None else _ptr(rs), _threads())
    return out.reshape(shape)


def uniform_f32(n: int, k: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    host_lib().syn_fill_uniform_f32(_ptr(out), n, k, lo, hi, _threads())
    return out


def q2k_blocks(nblocks: int, k: int, dlo: float = 1e-3, dhi: float = 4e-3, block0: int = 0) -> np.ndarray:
    out = np.empty(nblocks * Q2K_BYTES, dtype=np.uint8)
    host_lib().syn_fill_q2k(_ptr(out), nblocks, block0, k, dlo, dhi, _threads())
    return out


def q3k_blocks(nblocks: int, k: int, dlo: float = 5e-4, dhi: float = 2e-3, block0: int = 0) -> np.ndarray:
    out = np.empty(nblocks * Q3K_BYTES, dtype=np.uint8)
    host_lib().syn_fill_q3k(_ptr(out), nblocks, block0, k, dlo, dhi, _threads())
    return out


def permutation(n: int, k: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    host_lib().syn_permutation(_ptr(out), n, k)
    return out
