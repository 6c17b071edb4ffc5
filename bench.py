#!/usr/bin/env python
"""Benchmark of the moe_v41 hot path on GB300.

Default workload: the full-shape decode step, 40 independent MoE layers
(dim 5120, inter 2304, 384 routed experts, top-6, m = 1, bf16 shared expert),
every routed expert resident in HBM behind a slot-pointer table.  One step is
one pass of all 40 layers for one token: router + selection on the device,
q8_1(x), Q2_K gate/up + clipped SwiGLU + q8_1(h), Q3_K down, G-weighted sum,
shared expert added last.

Prints one JSON line (rank 0).  `value` is tokens/s through the 40-layer step
with inputs resident in HBM; `e2e` is the same metric through the C-ABI with
host buffers copied in and out inside the timed region.  The `prefill` object
holds the same measurements for the long-prefill workload (one layer call of
4096 tokens with x50 outlier rows per step), the metric's other size.
`--impl reference` times the CPU oracle instead (the reference arm of this
benchmark).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth.workloads as W  # noqa: E402

HBM_FALLBACK_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_m1_40layer", choices=sorted(W.WORKLOADS))
    ap.add_argument("--layers", type=int, default=0, help="layers per step (default: the workload's)")
    ap.add_argument("--resident-layers", type=int, default=0,
                    help="distinct layer weight sets held on the device (default: all layers)")
    ap.add_argument("--resident-experts", type=int, default=0,
                    help="expert slots held per layer (default: all; fewer alias experts, for small profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--prefill-workload", default="prefill_m4096_outliers", choices=sorted(W.WORKLOADS))
    ap.add_argument("--prefill-steps", type=int, default=30)
    ap.add_argument("--prefill-m", type=int, default=0, help="tokens of the prefill call (default: the workload's)")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the 8-token decode and 512-token prefill lines")
    ap.add_argument("--no-streamed", action="store_true")
    ap.add_argument("--streamed-layers", type=int, default=4, help="layers of the host arena (streamed leg)")
    ap.add_argument("--streamed-slots", type=int, default=256, help="HBM expert slots of the streamed leg")
    ap.add_argument("--streamed-tokens", type=int, default=64, help="timed tokens of the streamed leg")
    ap.add_argument("--prefetch-k", type=int, default=6, help="predicted next-layer experts fetched ahead")
    ap.add_argument("--streamed-reps", type=int, default=3, help="repetitions of each streamed configuration")
    ap.add_argument("--streamed-only", action="store_true",
                    help="run only the streamed leg and print its JSON object (the main run starts it this way)")
    ap.add_argument("--mma-rates", action="store_true",
                    help="only measure tcgen05.mma issue rates (kinds, widths, A in shared or tensor memory)")
    ap.add_argument("--graph", type=int, default=1,
                    help="1: time the decode step as one CUDA-graph replay of its layer calls; 0: eager launches")
    return ap.parse_args()


# ------------------------------------------------------------------ utils

BF16_FALLBACK_TFS = 1900.0


def peaks():
    """(HBM GB/s, dense bf16/fp16 TFLOP/s burst, sustained, kind)"""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)) or None, \
            "measured"
    except Exception:
        return HBM_FALLBACK_GBS, BF16_FALLBACK_TFS, 1700.0, "fallback"


def algorithmic_bytes(w: W.Workload, distinct: float) -> float:
    """Bytes the method must move for one layer call: router weight and bias,
    the distinct routed experts' blocks, the shared expert, x in, out out."""
    router = w.n_routed * w.dim * 2 + w.n_routed * 4
    shared = 3 * w.dim * w.inter * 2 if w.shared_kind == W.SHARED_BF16 else w.expert_bytes
    return router + distinct * w.expert_bytes + shared + w.m * w.dim * 2 + w.m * w.dim * 4


def algorithmic_flops(w: W.Workload) -> float:
    """Multiply-adds x 2 the method performs for one layer call: the router
    GEMV/GEMM, three projections per (token, picked expert), and the shared
    expert's three projections per token."""
    router = 2.0 * w.m * w.n_routed * w.dim
    routed = 2.0 * w.m * w.topk * 3 * w.dim * w.inter
    shared = 2.0 * w.m * 3 * w.dim * w.inter
    return router + routed + shared


def roofline(w: W.Workload, distinct: float, per_call_ms: float, kernel: str, traffic):
    """The slower of the byte and the flop bound of one layer call (decode is
    byte-bound; long prefill is tensor-bound), achieved against it."""
    hbm, tfs, tfs_sus, kind = peaks()
    sec = per_call_ms / 1000.0
    nbytes = algorithmic_bytes(w, distinct)
    flops = algorithmic_flops(w)
    t_bytes = nbytes / (hbm * 1e9)
    t_flops = flops / (tfs * 1e12)
    if t_bytes >= t_flops:
        r = {"bound": "hbm", "achieved": nbytes / sec / 1e9, "peak": hbm, "unit": "GB/s",
             "frac": nbytes / sec / 1e9 / hbm, "peak_kind": f"{kind} (copy bandwidth)"}
        r["frac_of_8tbs"] = r["achieved"] / 8000.0
    else:
        r = {"bound": "tensor", "achieved": flops / sec / 1e12, "peak": tfs, "unit": "TFLOP/s",
             "frac": flops / sec / 1e12 / tfs,
             "peak_kind": f"{kind} dense bf16 burst (fp16 runs at the same rate)"}
        r["hbm_achieved_gbs"] = nbytes / sec / 1e9
        r["hbm_frac"] = r["hbm_achieved_gbs"] / hbm
    r.update({"kernel": kernel, "traffic": traffic, "algorithmic_bytes_per_call": nbytes,
              "algorithmic_flops_per_call": flops, "us_per_call": per_call_ms * 1000.0,
              "bound_us": max(t_bytes, t_flops) * 1e6})
    return r


KERNEL_SOURCES = {
    "decode": ["k_decode.cu", "select.cuh", "common.cuh", "internal.h"],
    "prefill": ["k_prefill.cu", "k_prefill_kq.cu", "tc.cuh", "k_route.cu", "select.cuh", "common.cuh", "internal.h"],
}


def sources_hash(kind: str) -> str:
    """Hash of the sources of one kernel family: a recorded ncu traffic figure
    is used only while it still describes the code that runs."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_mixture_experts_router_gb300", "csrc")
    for f in KERNEL_SOURCES[kind]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per layer call from the committed ncu summary, if it was
    taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    kind = "decode" if W.WORKLOADS[workload].m <= 8 else "prefill"
    if kv.get("sources_sha256_16") != sources_hash(kind):
        return None
    try:
        return float(kv["dram_bytes_per_layer_call"])
    except (KeyError, ValueError):
        return None


class Clocks:
    """SM clock and clock-event reasons sampled every millisecond during the
    timed region, through NVML (read-only queries; the GPU's settings are
    never changed), else by nvidia-smi every 100 ms."""
    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.thread = None
        self.samples = []
        self.max_mhz = None
        self.nvml = None
        self.handle = None

    def _nvml_open(self):
        import ctypes
        try:
            L = ctypes.CDLL("libnvidia-ml.so.1")
            if L.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            bus = None
            try:
                import torch
                pr = torch.cuda.get_device_properties(self.index)
                bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0".encode()
            except Exception:
                bus = None
            ok = bus is not None and L.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) == 0
            if not ok and L.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) != 0:
                return False
            mx = ctypes.c_uint()
            if L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.nvml, self.handle = L, h
            return True
        except (OSError, AttributeError):
            return False

    def _poll(self):
        import ctypes
        L, h = self.nvml, self.handle
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            L.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_flag:
            if L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and get_reasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((float(mhz.value), int(rs.value)))
            time.sleep(0.001)

    def start(self):
        import threading
        self.samples = []
        self.stop_flag = False
        if self._nvml_open():
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self.stop_flag = True
            self.thread.join()
            self.thread = None
            sm = [m for m, _ in self.samples]
            reasons = sorted({n for _, r in self.samples for bit, n in self.REASONS.items() if r & bit})
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "samples": len(sm), "source": "nvml, 1 ms", "reasons": reasons}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [s.strip() for s in line.split(",")]
            if len(f) < 6:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "source": "nvidia-smi, 100 ms", "reasons": sorted(reasons)}


# ----------------------------------------------------------- oracle (CPU)

def _oracle_inputs(w: W.Workload, layer: int, tokens):
    import oracle
    x, R, b, sh = W.x_bf16(w, layer), W.router_bf16(w, layer), W.bias_f32(w, layer), W.shared_weights(w, layer)
    z = oracle.router_logits(x[sorted(set(tokens))], R)
    _, idx, _ = oracle.route_from_logits(oracle.cfg_of(w), z, b)
    experts = [None] * w.n_routed
    for e in np.unique(idx):
        experts[int(e)] = W.expert_blocks(w, layer, int(e))
    return x, R, b, experts, sh


def _oracle_run(w: W.Workload, inp, token: int):
    import oracle
    x, R, b, experts, sh = inp
    oracle.moe_layer(oracle.cfg_of(w), x, R, b, experts, w.shared_kind, *sh, tokens=[token], nthreads=1)


def cpu_baseline(w: W.Workload, layers_per_step: int, n_units: int, threads: int, target_s: float = 0.0):
    """Time the oracle, as it stands, on a token sample of a one-layer
    workload (the prefill calls): a fixed sample of distinct tokens spread
    over the batch, run over `threads` host threads, repeated until the
    timed work reaches `target_s` seconds (or exactly n_units units when
    target_s is 0).  Returns (tokens/s, seconds, units, description)."""
    base = max(1, min(n_units, threads))
    stride = max(1, w.m // base)
    sample = [(u % w.layers if w.layers > 1 else 0, ((u // max(1, w.layers)) * stride) % w.m) for u in range(base)]
    layers = sorted(set(l for l, _ in sample))
    with ThreadPoolExecutor(min(threads, 8)) as ex:
        inputs = dict(zip(layers, ex.map(lambda l: _oracle_inputs(w, l, [t for ll, t in sample if ll == l]),
                                         layers)))

    def run(n):
        units = [sample[i % base] for i in range(n)]
        t0 = time.perf_counter()
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda u: _oracle_run(w, inputs[u[0]], u[1]), units))
        return time.perf_counter() - t0

    n = n_units
    if target_s > 0:
        dt0 = run(base)  # calibration (not reported)
        n = max(base, min(64 * base, int(math.ceil(target_s / max(dt0, 1e-3))) * base))
    dt = run(n)
    # a step moves one token through layers_per_step layer calls
    tps = n / layers_per_step / dt
    desc = (f"{n} (layer, token) units of {w.name} cycling over {base} distinct units ({len(layers)} layers, "
            f"tokens spread over the batch) on {threads} threads; tokens/s = units / layers per step / seconds")
    return tps, dt, n, desc


class OracleSteps:
    """The oracle, as it stands, timed on steps of a decode workload on the
    host cores.  A full step is what the GPU step does: every token of the
    call (m of them) through every layer of the step (L), i.e. m * L
    (layer, token) units, submitted together to `threads` host threads and
    waited for.  A bounded step takes the first `units` of those units (the
    tokens of layer 0, then of layer 1, ...).  Used by the reference arm and
    by the cpu_baseline of the decode lines, so both report the same thing."""

    def __init__(self, w: W.Workload, L: int, threads: int):
        self.w, self.L, self.threads = w, L, threads
        self.full = [(l, t) for l in range(L) for t in range(w.m)]
        with ThreadPoolExecutor(min(threads, 8)) as ex:
            self.inputs = dict(zip(range(L), ex.map(lambda l: _oracle_inputs(w, l, list(range(w.m))), range(L))))
        self.ex = ThreadPoolExecutor(threads)

    def unit_seconds(self) -> float:
        """wall time of one unit on one thread (calibration, not reported)"""
        t0 = time.perf_counter()
        _oracle_run(self.w, self.inputs[0], 0)
        return time.perf_counter() - t0

    def step(self, units: int) -> float:
        todo = self.full[:units]
        t0 = time.perf_counter()
        list(self.ex.map(lambda u: _oracle_run(self.w, self.inputs[u[0]], u[1]), todo))
        return time.perf_counter() - t0

    def close(self):
        self.ex.shutdown()

    def describe(self, units: int, steps: int) -> str:
        full = len(self.full)
        what = "a full step" if units == full else f"a bounded step: {units} of the {full}"
        return (f"{steps} steps of {self.w.name}, each {what} (layer, token) units ({self.w.m} token(s) x "
                f"{self.L} layers), submitted together to {self.threads} host threads and waited for; "
                f"tokens/s = units / layers per step / seconds")


def oracle_decode_baseline(w: W.Workload, L: int, threads: int, target_s: float):
    """cpu_baseline of a decode line: whole steps until about target_s seconds."""
    o = OracleSteps(w, L, threads)
    try:
        units = len(o.full)
        o.step(units)  # warm-up and calibration
        t1 = o.step(units)
        n = max(1, int(round(target_s / max(t1, 1e-3))))
        dt = sum(o.step(units) for _ in range(n))
        tps = n * units / L / dt
        return tps, dt, n, o.describe(units, n) + f", {dt:.1f} s"
    finally:
        o.close()


# ------------------------------------------------------------------- GPU

def max_over_ranks(vals, device=None):
    """Each value's largest over the ranks of the process group (the job ends
    when its slowest rank does); identity without a group of several ranks."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tokens_per_s(world: int, m: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank moves m tokens per step through the
    step's layers (weak scaling), over the slowest rank's time."""
    return world * m * steps / (ms / 1000.0)


def run_ours(args, rank, world, local_rank):
    import torch
    import quantized_mixture_experts_router_gb300 as Q
    from synth.device import stage_layer

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = W.WORKLOADS[args.workload]
    L = args.layers or w.layers
    free, total = torch.cuda.mem_get_info()
    per_layer = w.n_routed * (w.expert_bytes + 1024) + 3 * w.dim * w.inter * 2 + w.n_routed * w.dim * 2
    resident = args.resident_layers or L
    fit = max(1, int((free - (8 << 30)) // per_layer))
    rotated = resident > fit
    resident = min(resident, fit)
    layers = [stage_layer(w, l, device=dev, experts_on_gpu=True, bulk_on_gpu=True, slots=args.resident_experts)
              for l in range(resident)]
    # x of every layer of the step (the layer's own seeded rows)
    xs = [layers[l % resident].x if l < resident else stage_x(w, l, dev) for l in range(L)]
    cfg = Q.make_cfg(w.dim, w.inter, w.n_routed, w.topk, w.gate_temp, w.norm_topk_prob, w.route_scale,
                     w.swiglu_limit, max_tokens=w.m)
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    Q.moe_v41_workspace_init(ws)
    out = torch.empty((L, w.m, w.dim), dtype=torch.float32, device=dev)
    tw = torch.empty((L, w.m, w.topk), dtype=torch.float32, device=dev)
    ti = torch.empty((L, w.m, w.topk), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def layer_call(l, x=None):
        # on the current stream: the launch stream, or the capture stream of a graph
        d = layers[l % resident]
        Q.moe_v41_forward(cfg, xs[l] if x is None else x, w.m, d.router_w, d.bias, d.expert_ptrs, w.shared_kind,
                          d.sh1, d.sh3, d.sh2, out[l], tw[l], ti[l], None, ws)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        for l in range(L):
            layer_call(l)
    st = Q.moe_v41_read_status(ws, stream, clear=True)
    if st:
        raise RuntimeError(f"device status {st} during warm-up")
    distinct = float(np.mean([np.unique(ti[l].cpu().numpy()).size for l in range(L)]))

    # --- device-resident timed region: the step's L layer calls captured once
    # as a CUDA graph and replayed K times (routing never leaves the device,
    # so a step has no host round trip), or launched eagerly with one event
    # per layer boundary
    K = args.steps
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for l in range(L):
                layer_call(l)
        graph.replay()
        torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(L + 1)] for _ in range(K)] if graph is None else []
    barrier()
    clocks = Clocks(local_rank)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(K):
        if graph is not None:
            graph.replay()
            continue
        for l in range(L):
            evs[k][l].record(stream)
            layer_call(l)
        evs[k][L].record(stream)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end)
    if graph is not None:
        per_call_ms = ms / (K * L)
    else:
        per_call_ms = statistics.fmean(evs[k][l].elapsed_time(evs[k][l + 1]) for k in range(K) for l in range(L))
    st = Q.moe_v41_read_status(ws, stream, clear=True)
    if st:
        raise RuntimeError(f"device status {st} during the timed region")

    # --- end to end through host buffers
    e2e = None
    if not args.no_e2e:
        # the step's inputs and results as one pinned buffer each: one host->device
        # copy in and one device->host copy out per step
        xh = torch.empty((L, w.m, w.dim), dtype=torch.int16).pin_memory()
        for l in range(L):
            xh[l].copy_(xs[l].cpu())
        oh = torch.empty((L, w.m, w.dim), dtype=torch.float32).pin_memory()
        xd = torch.empty((L, w.m, w.dim), dtype=torch.int16, device=dev)
        Ke = max(1, K // 2)

        def e2e_step():
            xd.copy_(xh, non_blocking=True)
            for l in range(L):
                layer_call(l, xd[l])
            oh.copy_(out, non_blocking=True)
        for _ in range(2):
            e2e_step()
        barrier()
        # the same capture as the device-resident region, host copies included
        e2e_graph = None
        if args.graph:
            e2e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graph):
                e2e_step()
            e2e_graph.replay()
            barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Ke):
            if e2e_graph is not None:
                e2e_graph.replay()
            else:
                e2e_step()
        e1.record(stream)
        barrier()
        e_ms = e0.elapsed_time(e1)
        e2e = dict(ms=e_ms, steps=Ke, h2d=L * w.m * w.dim * 2, d2h=L * w.m * w.dim * 4)

    # max over ranks
    ms, e_ms_max = max_over_ranks([ms, e2e["ms"] if e2e else 0.0], dev)
    if e2e:
        e2e["ms"] = e_ms_max
    launches = Q.moe_v41_kernel_launches(cfg, w.m, w.shared_kind)
    del graph, layers, xs, out, tw, ti, ws
    torch.cuda.empty_cache()
    return dict(w=w, L=L, K=K, ms=ms, per_call_ms=per_call_ms, distinct=distinct, clocks=clk, e2e=e2e,
                resident=resident, rotated=rotated, launches_per_call=launches, graph=bool(args.graph),
                kernel=("k_decode_layer (the whole layer call, one launch)" if launches == 1 else
                        f"the prefill kernels of one layer call ({launches} launches)"),
                resident_experts=args.resident_experts)


def run_call(args, local_rank, w: W.Workload, K: int):
    """A one-layer workload (the prefill calls, the 8-token decode call): one
    layer call of m tokens per step, timed with events per call; then the
    same calls through host buffers."""
    import torch
    import quantized_mixture_experts_router_gb300 as Q
    from synth.device import stage_layer

    dev = torch.device("cuda", local_rank)
    d = stage_layer(w, 0, device=dev, experts_on_gpu=True, bulk_on_gpu=True, slots=args.resident_experts)
    cfg = Q.make_cfg(w.dim, w.inter, w.n_routed, w.topk, w.gate_temp, w.norm_topk_prob, w.route_scale,
                     w.swiglu_limit, max_tokens=w.m)
    ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    Q.moe_v41_workspace_init(ws)
    out = torch.empty((w.m, w.dim), dtype=torch.float32, device=dev)
    tw = torch.empty((w.m, w.topk), dtype=torch.float32, device=dev)
    ti = torch.empty((w.m, w.topk), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def call(x):
        Q.moe_v41_forward(cfg, x, w.m, d.router_w, d.bias, d.expert_ptrs, w.shared_kind, d.sh1, d.sh3, d.sh2, out,
                          tw, ti, None, ws, stream)

    for _ in range(3):
        call(d.x)
    st = Q.moe_v41_read_status(ws, stream, clear=True)
    if st:
        raise RuntimeError(f"device status {st} during prefill warm-up")
    distinct = float(np.unique(ti.cpu().numpy()).size)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    torch.cuda.synchronize()
    clocks = Clocks(local_rank)
    clocks.start()
    for k in range(K):
        evs[k].record(stream)
        call(d.x)
    evs[K].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    per_call = [evs[k].elapsed_time(evs[k + 1]) for k in range(K)]
    st = Q.moe_v41_read_status(ws, stream, clear=True)
    if st:
        raise RuntimeError(f"device status {st} during the prefill timed region")
    e2e = None
    if not args.no_e2e:
        xh = d.x.cpu().pin_memory()
        oh = torch.empty((w.m, w.dim), dtype=torch.float32).pin_memory()
        xd = torch.empty_like(d.x)

        def e2e_call():
            xd.copy_(xh, non_blocking=True)
            call(xd)
            oh.copy_(out, non_blocking=True)
        for _ in range(2):
            e2e_call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            e2e_call()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e = dict(ms=e0.elapsed_time(e1), steps=K, h2d=w.m * w.dim * 2, d2h=w.m * w.dim * 4)
    launches = Q.moe_v41_kernel_launches(cfg, w.m, w.shared_kind)
    # the slowest rank's figures
    mean_ms, min_ms, e_ms = max_over_ranks([statistics.fmean(per_call), min(per_call), e2e["ms"] if e2e else 0.0], dev)
    if e2e:
        e2e["ms"] = e_ms
    del d, ws, out, tw, ti
    torch.cuda.empty_cache()
    return dict(w=w, K=K, per_call_ms=mean_ms, per_call_min_ms=min_ms, distinct=distinct,
                clocks=clk, e2e=e2e, launches_per_call=launches, resident_experts=args.resident_experts)


def _mem_available() -> int:
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def streamed_in_child(args):
    """The streamed leg in a process of its own, after the other legs have
    released their device memory.  (Run after them in one process, single
    runs took 0.7-1.3 ms per layer call instead of 0.39-0.47; run_streamed's
    untimed pass over the arena is what removed that, this keeps the legs
    apart as well.)"""
    import gc

    import torch
    gc.collect()
    torch.cuda.empty_cache()  # the child needs the device memory the earlier legs held
    cmd = [sys.executable, os.path.abspath(__file__), "--streamed-only", "--workload", args.workload,
           "--warmup", str(args.warmup), "--streamed-layers", str(args.streamed_layers),
           "--streamed-slots", str(args.streamed_slots), "--streamed-tokens", str(args.streamed_tokens),
           "--prefetch-k", str(args.prefetch_k), "--streamed-reps", str(args.streamed_reps)]
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
    if p.returncode != 0:
        return {"skipped": "streamed leg failed: " + (p.stderr.strip().splitlines() or ["?"])[-1]}
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    sm = json.loads(lines[-1]) if lines else {"skipped": "streamed leg printed no result"}
    sm["process"] = "a child process of its own, after one untimed host -> HBM pass over the arena"
    return sm


def run_streamed(args, local_rank):
    """The decode workload with the routed experts streamed: every expert of
    a few layers in a page-locked host arena, a least-recently-used set of HBM
    slots, one token at a time through the layers with moe_v41_forward_streamed
    (route, host span, fetch, forward), once without and once with the next
    layer's experts predicted and fetched ahead.  Each token's layers take the
    same x (a stand-in for the residual stream's layer-to-layer correlation),
    so a prediction of prefetch_k = topk is the next layer's true routing."""
    import torch
    import quantized_mixture_experts_router_gb300 as Q
    from synth.device import fill_experts_gpu, slot_layout, stage_layer

    dev = torch.device("cuda", local_rank)
    torch.cuda.empty_cache()
    w = W.WORKLOADS[args.workload]
    o1, o3, o2, slot = slot_layout(w)
    layer_bytes = w.n_routed * slot
    Ls = args.streamed_layers
    avail = _mem_available()
    while Ls > 1 and Ls * layer_bytes * 3 > avail:
        Ls -= 1
    if Ls * layer_bytes * 3 > avail:
        return {"skipped": f"host memory: {avail / 1e9:.0f} GB available, one layer's arena is {layer_bytes / 1e9:.1f} GB"}
    S = args.streamed_slots
    free, _ = torch.cuda.mem_get_info()
    if S * slot + layer_bytes + Ls * 100e6 > free - (4 << 30):
        S = max(2 * w.topk, int((free - (4 << 30) - layer_bytes - Ls * 100e6) // slot))
    cudart = torch.cuda.cudart()
    arena = torch.empty((Ls, w.n_routed, slot), dtype=torch.uint8)
    rc = cudart.cudaHostRegister(arena.data_ptr(), arena.numel(), 0)
    if int(rc) != 0:
        return {"skipped": f"cudaHostRegister of the {arena.numel() / 1e9:.1f} GB arena failed ({int(rc)})"}
    try:
        stagebuf = torch.empty((w.n_routed, slot), dtype=torch.uint8, device=dev)
        for l in range(Ls):
            fill_experts_gpu(w, l, stagebuf)
            arena[l].copy_(stagebuf)
        # one untimed host -> HBM pass over the whole arena before any timed
        # run (the first timed run over freshly registered pages was slow)
        for l in range(Ls):
            stagebuf.copy_(arena[l], non_blocking=True)
        torch.cuda.synchronize()
        # the link's own rate: plain arena -> HBM copies of whole expert slots
        nprobe = min(16, w.n_routed)
        probe = stagebuf[:nprobe]
        probe.copy_(arena[0, :nprobe], non_blocking=True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(3):
            probe.copy_(arena[0, :nprobe], non_blocking=True)
        torch.cuda.synchronize()
        link_gbs = 3 * nprobe * slot / (time.perf_counter() - t0) / 1e9
        del stagebuf, probe
        layers = [stage_layer(w, l, device=dev, experts_on_gpu=True, bulk_on_gpu=True, slots=1) for l in range(Ls)]
        xs = [stage_x(w.with_(seed=w.seed + 7000 + t), 0, dev) for t in range(16)]
        cfg = Q.make_cfg(w.dim, w.inter, w.n_routed, w.topk, w.gate_temp, w.norm_topk_prob, w.route_scale,
                         w.swiglu_limit, max_tokens=w.m)
        ws = torch.empty(Q.moe_v41_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
        Q.moe_v41_workspace_init(ws)
        out = torch.empty((w.m, w.dim), dtype=torch.float32, device=dev)
        tw = torch.empty((w.m, w.topk), dtype=torch.float32, device=dev)
        ti = torch.empty((w.m, w.topk), dtype=torch.int32, device=dev)
        stream = torch.cuda.current_stream()
        copy_stream = torch.cuda.Stream(device=dev)
        runs = []
        # each configuration several times, alternating: single runs on one box have taken up to 2.8x the
        # usual time (copies at ~48 GB/s instead of ~160), in either configuration, cause not established
        plan_runs = [(rep, P) for rep in range(args.streamed_reps)
                     for P in ([0, args.prefetch_k] if args.prefetch_k > 0 else [0])]
        for rep, P in plan_runs:
            slots = torch.empty((S, slot), dtype=torch.uint8, device=dev)
            tables = torch.empty((Ls, w.n_routed, 3), dtype=torch.int64, device=dev)
            cache = Q.ExpertCache(Ls, w.n_routed, S, slot, o1, o3, o2, arena, slots, tables)
            host = torch.empty(w.m * w.topk + P, dtype=torch.int32, pin_memory=True)

            def token(t):
                x = xs[t % len(xs)]
                for l in range(Ls):
                    d = layers[l]
                    n = layers[l + 1] if l + 1 < Ls else None
                    Q.moe_v41_forward_streamed(cfg, cache, l, x, w.m, d.router_w, d.bias,
                                               None if n is None else n.router_w, None if n is None else n.bias, P,
                                               w.shared_kind, d.sh1, d.sh3, d.sh2, out, tw, ti, ws, host, stream,
                                               copy_stream)
            Tw = max(args.warmup, S // (w.topk * Ls) + 4)
            for t in range(Tw):
                token(t)
            torch.cuda.synchronize()
            st0 = cache.stats()
            T = args.streamed_tokens
            t0 = time.perf_counter()
            for t in range(Tw, Tw + T):
                token(t)
            torch.cuda.synchronize()
            sec = time.perf_counter() - t0
            st1 = cache.stats()
            status = Q.moe_v41_read_status(ws, stream, clear=True)
            if status:
                raise RuntimeError(f"device status {status} in the streamed leg")
            dd = {k: st1[k] - st0[k] for k in st1}
            calls = T * Ls
            runs.append({"prefetch_k": P, "rep": rep, "ms_per_layer_call": 1000.0 * sec / calls, "tokens_per_s": T / sec,
                         "tokens_per_s_40_layers": T / sec * Ls / 40.0,
                         "hit_rate": dd["hits"] / max(1, dd["hits"] + dd["misses"]),
                         "prefetch_hits_per_call": dd["prefetch_hits"] / calls,
                         "misses_per_call": dd["misses"] / calls, "bytes_copied_per_call": dd["bytes_copied"] / calls,
                         "copy_gbs": dd["bytes_copied"] / sec / 1e9,
                         "link_bound_ms_per_call": dd["bytes_copied"] / calls / (link_gbs * 1e9) * 1e3,
                         "frac_of_link": dd["bytes_copied"] / sec / 1e9 / link_gbs})
            cache.close()
            del slots, tables, cache
        medians = {str(P): statistics.median(r["ms_per_layer_call"] for r in runs if r["prefetch_k"] == P)
                   for P in sorted(set(r["prefetch_k"] for r in runs))}
        return {"workload": w.name + " (experts streamed)", "arena_layers": Ls, "arena_bytes": arena.numel(),
                "median_ms_per_layer_call": medians,
                "slots": S, "slot_bytes": slot, "hbm_slot_bytes": S * slot, "timed_tokens": args.streamed_tokens,
                "layers_per_token": Ls, "link_gbs": link_gbs,
                "link": "arena -> HBM rate of plain copies of whole expert slots, measured in this run",
                "timing": "wall clock over the timed tokens, both streams drained at the ends",
                "x": "one seeded x per token, the same for every layer of the token", "runs": runs}
    finally:
        torch.cuda.synchronize()
        cudart.cudaHostUnregister(arena.data_ptr())


def stage_x(w, l, dev):
    import torch
    from synth.device import x_gpu
    t = torch.empty((w.m, w.dim), dtype=torch.int16, device=dev)
    x_gpu(w, l, t)
    return t


def mma_rates(local_rank):
    """tcgen05.mma throughput with every SM issuing back-to-back MMAs
    (M = 128, one K step each) into one accumulator: f16, bf16 and e4m3
    operands, widths 32..256, A from shared or from tensor memory.  Each
    figure is the launch's CUDA-event time; TFLOP/s counts 2 * 128 * N * K
    per MMA over all SMs.  (There is no int8 kind to measure: ptxas refuses
    tcgen05.mma .kind::i8 for sm_103a.)"""
    import ctypes
    import torch
    from quantized_mixture_experts_router_gb300.build import PEAKS_SO
    torch.cuda.set_device(local_rank)
    sms = torch.cuda.get_device_properties(local_rank).multi_processor_count
    L = ctypes.CDLL(PEAKS_SO)
    L.mma_rate_run.argtypes = [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_float),
                                                    ctypes.POINTER(ctypes.c_ulonglong)]
    res = []
    clocks = Clocks(local_rank)
    clocks.start()
    cases = [(kind, name, kd, a, n, 128, 1) for kind, name, kd in ((0, "f16", 16), (1, "bf16", 16), (3, "e4m3", 32))
             for a in (0, 1) for n in (32, 64, 128, 256)]
    # independent accumulators cycled through, and the M = 64 shape
    cases += [(0, "f16", 16, a, n, 128, nacc) for a in (0, 1) for n in (32, 64, 128) for nacc in (2, 4)
              if nacc * n <= (256 if a else 512)]
    cases += [(0, "f16", 16, 0, n, 64, nacc) for n in (64, 128, 256) for nacc in (1, 2) if nacc * n <= 512]
    for kind, name, kdepth, a_tmem, n, mm, nacc in cases:
        iters = max(2000, 4000000 // n) // 4 * 4
        ms = ctypes.c_float()
        clk = (ctypes.c_ulonglong * sms)()
        rc = L.mma_rate_run(kind, n, mm, nacc, a_tmem, iters, sms, ctypes.byref(ms), clk)
        tag = {"kind": name, "m": mm, "n": n, "nacc": nacc, "a": "tmem" if a_tmem else "smem"}
        if rc != 0:
            res.append(dict(tag, error=rc))
            continue
        flops = 2.0 * mm * n * kdepth * iters * sms
        cyc = statistics.median(list(clk))
        res.append(dict(tag, iters=iters, ms=ms.value, tflops=flops / (ms.value / 1e3) / 1e12,
                        cycles_per_mma=cyc / iters, macs_per_clk_sm=mm * n * kdepth * iters / cyc))
    clk = clocks.stop()
    print(json.dumps({"mma_rates": res, "sms": sms, "clocks": clk}), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = W.WORKLOADS[args.workload]
    L = args.layers or w.layers
    ncores = os.cpu_count() or 1

    if args.mma_rates:
        mma_rates(local_rank)
        return
    if args.streamed_only:
        print(json.dumps(run_streamed(args, local_rank)), flush=True)
        return

    if args.impl == "reference":
        # the CPU oracle as the reference arm: rank 0 only
        if rank != 0:
            return
        K, Wm = args.steps, args.warmup
        o = OracleSteps(w, L, ncores)
        try:
            unit_s = o.unit_seconds()
            full = len(o.full)
            # bounded steps when K + W full steps would not end within a few minutes
            waves = int(150.0 / ((K + Wm) * max(unit_s, 1e-3)))
            units = min(full, max(1, waves * ncores))
            for _ in range(Wm):
                o.step(units)
            dt = sum(o.step(units) for _ in range(K))
            desc = o.describe(units, K)
        finally:
            o.close()
        tps = K * units / L / dt
        line = {"impl": "reference", "metric": metric_name(w), "value": tps, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": K, "warmup": Wm, "ms_per_step": 1000.0 * dt / K, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config_of(w, L),
                "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": ncores, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = run_ours(args, rank, world, local_rank)
    sm = None if (args.no_streamed or world > 1) else streamed_in_child(args)
    calls = []
    if not args.no_prefill:
        pw = W.WORKLOADS[args.prefill_workload]
        if args.prefill_m:
            pw = pw.with_(m=args.prefill_m)
        calls.append(("prefill", pw, args.prefill_steps))
    if not args.no_extra:
        calls.append(("prefill_m512", W.WORKLOADS["prefill_m512_hot"], args.prefill_steps))
        calls.append(("decode_m8", W.WORKLOADS["decode_m8_kquant_shared"], max(args.prefill_steps, 30)))
    res_calls = [(key, run_call(args, local_rank, cw, K)) for key, cw, K in calls]
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    K = r["K"]
    value = job_tokens_per_s(world, w.m, K, r["ms"])
    traffic = recorded_traffic(args.workload)
    line = {
        "metric": metric_name(w), "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": r["ms"] / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8-dp4a/bf16-fma, f32 accumulate", "data": "synthetic",
        "config": config_of(w, L), "run": run_of(r),
        "roofline": roofline(w, r["distinct"], r["per_call_ms"], r["kernel"], traffic),
        "gpu_launches": (r["launches_per_call"] or 0) * L * K,
        "clocks": r["clocks"],
    }
    if r["e2e"]:
        e = r["e2e"]
        line["e2e"] = {"value": job_tokens_per_s(world, w.m, e["steps"], e["ms"]), "unit": "tokens/s",
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"]}
    if world == 1 and not args.no_cpu_baseline:
        tps, dt, n, desc = oracle_decode_baseline(w, L, ncores, 12.0)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": ncores, "kind": "oracle", "sample": desc}
    for key, pf in res_calls:
        pw = pf["w"]
        decode_like = pw.m <= 8
        p = {"workload": pw.name, "metric": metric_name(pw),
             "value": job_tokens_per_s(world, pw.m, 1, pf["per_call_ms"]), "unit": "tokens/s",
             "steps": pf["K"], "warmup": 3, "ms_per_step": pf["per_call_ms"], "ms_per_step_min": pf["per_call_min_ms"],
             "config": config_of(pw, 1), "run": run_of(pf),
             "roofline": roofline(pw, pf["distinct"], pf["per_call_ms"],
                                  ("k_decode_layer (the whole layer call, one launch)" if pf["launches_per_call"] == 1
                                   else f"the prefill kernels of one layer call ({pf['launches_per_call']} launches)"),
                                  # the recorded traffic is for the workload's own token count
                                  recorded_traffic(pw.name) if pw.m == W.WORKLOADS[pw.name].m else None),
             "gpu_launches": pf["launches_per_call"] * pf["K"], "clocks": pf["clocks"],
             "dtype": ("int8-dp4a, f32 accumulate" if decode_like else
                       "fp16 tensor-core GEMMs on exact-integer K-quant weights, bf16 router/shared, f32 accumulate")}
        if pf["e2e"]:
            e = pf["e2e"]
            p["e2e"] = {"value": job_tokens_per_s(world, pw.m, e["steps"], e["ms"]), "unit": "tokens/s",
                        "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"]}
        if world == 1 and not args.no_cpu_baseline:
            if decode_like:
                tps, dt, n, desc = oracle_decode_baseline(pw, 1, ncores, 6.0)
            else:
                tps, dt, n, desc = cpu_baseline(pw, 1, ncores, ncores, target_s=8.0)
                desc += f", {dt:.1f} s"
            p["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": ncores, "kind": "oracle", "sample": desc}
        line[key] = p
    if sm:
        line["streamed"] = sm
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def metric_name(w: W.Workload) -> str:
    return f"MoE-layer tokens/s, {w.name} (m={w.m}, {w.layers} layer(s) per step)"


def config_of(w: W.Workload, L: int):
    """The workload the line measures (the same keys in both arms)."""
    return {"workload": w.name, "dim": w.dim, "inter": w.inter, "n_routed": w.n_routed, "topk": w.topk, "m": w.m,
            "layers_per_step": L, "shared": "bf16" if w.shared_kind == W.SHARED_BF16 else "Q2_K/Q3_K",
            "experts": "Q2_K gate/up, Q3_K down, all resident in HBM",
            "l2": ("inputs larger than L2: each step streams the step's expert weights "
                   f"(>{algorithmic_bytes(w, min(w.n_routed, w.m * w.topk)) * L / 1e9:.1f} GB) through the "
                   "129 MB L2")}


def run_of(r):
    """How this run executed the workload (our arm only)."""
    c = {"distinct_experts_per_call": r["distinct"], "resident_layers": r.get("resident", 1)}
    if "graph" in r:
        c["launch"] = ("the step's layer calls captured once as a CUDA graph, replayed per step"
                       if r["graph"] else "eager launches, one event per layer boundary")
    if r.get("resident_experts"):
        c["resident_experts"] = r["resident_experts"]
        c["note_experts"] = "profiling run: expert e uses slot e % resident_experts"
    if r.get("rotated"):
        c["note"] = "device memory held fewer layers than the step; layers rotate over the resident ones"
    return c


if __name__ == "__main__":
    main()
