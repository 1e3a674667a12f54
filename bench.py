"""Benchmark of the routed MoE layer on one GB300 (or N independent replicas).

Headline (the JSON line's `value`): the decode MoE layer - hidden 6144, expert
intermediate 2048, 288 experts top-8 (fp32 softmax router), one bf16 shared
expert, NVFP4 routed experts all resident in HBM, 1 token per forward.  A step
is one pass of the whole hot path (route -> permute -> cache lookup -> expert
FFN gate/up -> down -> combine; three kernels for one token: router with the
permutation and lookup, gate/up, down with the combine) over one fresh token;
L2 is flushed between
steps outside the timed events (a buffer larger than L2 written, then another
read, so that no dirty line of the flush is written back inside a timed step).

The same run also measures (the `also` object), each in its own bounded pass:
  prefill  one layer on a 4096-token chunk, one launch per GEMM over all experts
           (tcgen05 NVFP4 grouped GEMMs): tokens/s, HBM and FP4 tensor fractions;
           and the same walked in launch groups of 64 experts;
  stack    16 decode layers, per-layer Zipf-skewed routing, 66 hot experts per
           layer in HBM, misses gathered from pinned host memory: tokens/s,
           hit rate, gather GB/s against the measured host->device link;
  flat     8 layers, 64 tokens per step, unbiased routing, 72 experts per layer
           cached by saliency, misses gathered from pinned host memory;
  stack_skip  the stack with the renorm-skip (tau 0.05): misses with a
           combine weight below tau dropped, the token's weights renormalised;
           with its error against the exact layer on the same inputs;
  stack_adaptive  the stack with the adaptive cache: per layer the 63 hottest
           resident at start and 3 spare slots, misses promoted into them,
           decayed-LFU eviction between forwards.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
decode workload instead (bounded sample, host cores).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoE-layer tokens/s (decode, 4096-tok prefill); % of HBM / FP4-TC / PCIe roofline"
UNIT = "tokens/s"
# the adaptive cache keeps three spare slots per layer ("Project Maya" page)
ADAPTIVE_SPARES = 3
# the stack passes warm up on this many distinct tokens (their misses touch
# most experts' host records once before the timed steps)
STACK_WARM_TOKENS = 256
# renorm-skip threshold of the stack_skip pass (an approximation of the layer)
SKIP_TAU = 0.05  # about one halving period of its counts on the 16-layer stack
FP4_OVER_BF16 = 6.0  # nominal dense FP4 / dense bf16 tensor throughput (13.5 / 2.25)
# DRAM bytes (read + write) of one launch of the roofline kernel on the full decode
# layer, from one ncu capture of the current kernel; None whenever the kernel has
# changed since it was captured
GU_TRAFFIC = 138_482_944 + 365_056
GU_TRAFFIC_SOURCE = "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch, full decode layer"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during a timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ helpers
def _events(torch, n):
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n)]


def prewarm(torch, fn, seconds=1.0):
    """Keeps the GPU busy for `seconds` so clocks and memory leave idle states."""
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        fn()
        torch.cuda.synchronize()


def link_h2d_gbs(torch, dev, mib=1024, reps=5):
    """Pinned host -> device copy bandwidth (cudaMemcpyAsync), best of reps."""
    h = torch.empty(mib << 20, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(mib << 20, dtype=torch.uint8, device=dev)
    d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    best = 1e30
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        d.copy_(h, non_blocking=True)
        b.record()
        b.synchronize()
        best = min(best, a.elapsed_time(b))
    del h, d
    return (mib << 20) / (best * 1e-3) / 1e9


class L2Flush:
    """Empties L2 between timed steps, outside the events: writes one buffer
    larger than L2, then reads another.  The read leaves L2 holding clean lines
    of neither input: after a write alone, up to the whole L2 is dirty and its
    write-back to HBM lands inside the next timed step (measured: +9.5 us on a
    164 MB read on this GPU)."""

    def __init__(self, torch, mib, dev):
        self.w = torch.empty(mib << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros((mib << 20) // 8, dtype=torch.int64, device=dev)
        self.mib = mib

    def __call__(self):
        self.w.zero_()
        self.r.sum()

    @staticmethod
    def describe_for(mib):
        return (f"flushed between steps outside the events: {mib} MiB written, then "
                f"{mib} MiB of another buffer read")


class ExplicitLayer:
    """One layer's hot path as the individual ABI calls (route, permute,
    lookup, gather, expert FFN, combine) on caller-owned buffers, so that the
    bench can put CUDA events around single launches."""

    def __init__(self, torch, moe, dw, layer, T):
        wl = dw.wl
        self.torch, self.moe, self.dw, self.layer, self.T = torch, moe, dw, layer, T
        H, I, E, k, Is = wl.H, wl.I, wl.E, wl.k, wl.Is
        dev = torch.device("cuda")
        i32, f32 = torch.int32, torch.float32
        self.b = {n: torch.zeros(sz, dtype=dt, device=dev) for n, sz, dt in (
            ("logits", T * E, f32), ("ids", T * k, i32), ("w", T * k, f32), ("p", T * k, f32),
            ("counts", E, i32), ("offsets", E + 1, i32), ("perm", T * k, i32),
            ("inv", T * k, i32), ("src", E, i32), ("act", E, i32), ("n_act", 2, i32),
            ("miss", E, i32), ("n_miss", 1, i32), ("status", 1, i32),
            ("o_route", T * k * H, f32), ("o_shared", T * H, f32))}
        b = self.b
        self.ws_bytes = moe.moe_ffn_workspace_bytes(0, T, H, I, E, k, Is)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        ra = moe.moe_route_args()
        ra.w_router = dw.w_router[layer].data_ptr()
        ra.bias = dw.bias[layer].data_ptr() if dw.bias[layer] is not None else None
        ra.T, ra.H, ra.E, ra.k = T, H, E, k
        ra.ids, ra.w, ra.p_sel, ra.logits = (b[n].data_ptr() for n in ("ids", "w", "p", "logits"))
        ra.status = b["status"].data_ptr()
        fa = moe.moe_ffn_args()
        fa.mode, fa.T, fa.H, fa.I, fa.E, fa.k = 0, T, H, I, E, k
        fa.cache, fa.gscale = dw.cache.handle, dw.gscale[layer].data_ptr()
        fa.src_slot, fa.act_list, fa.n_act = (b[n].data_ptr() for n in ("src", "act", "n_act"))
        fa.offsets, fa.perm, fa.w = (b[n].data_ptr() for n in ("offsets", "perm", "w"))
        fa.n_stage, fa.Is = dw.cache.n_stage, Is
        if Is:
            fa.s_gate, fa.s_up, fa.s_down = (t.data_ptr() for t in dw.shared[layer])
        fa.o_route = b["o_route"].data_ptr()
        fa.o_shared = b["o_shared"].data_ptr() if Is else None
        fa.workspace, fa.workspace_bytes = self.ws.data_ptr(), self.ws_bytes
        fa.status = b["status"].data_ptr()
        ca = moe.moe_combine_args()
        ca.T, ca.H, ca.k = T, H, k
        ca.o_route, ca.inv = b["o_route"].data_ptr(), b["inv"].data_ptr()
        ca.o_shared = b["o_shared"].data_ptr() if Is else None
        self.ra, self.fa, self.ca = ra, fa, ca
        S = max(dw.cache.n_stage, 1)
        self.max_miss = min(T * k, E)
        self.groups = (self.max_miss + S - 1) // S if dw.cache.n_stage > 0 else 1

    def step(self, x_ptr, y_ptr, sp, ev_fill=None, ev_gu=None, ev_dn=None):
        moe, b, dw = self.moe, self.b, self.dw
        wl = dw.wl
        self.ra.x = x_ptr
        moe.moe_route(self.ra, sp)
        moe.moe_permute(b["ids"].data_ptr(), self.T, wl.k, wl.E, b["counts"].data_ptr(),
                        b["offsets"].data_ptr(), b["perm"].data_ptr(), b["inv"].data_ptr(), 0,
                        128, b["status"].data_ptr(), sp)
        moe.expcache_lookup(dw.cache.handle, self.layer, b["counts"].data_ptr(),
                            b["src"].data_ptr(), b["act"].data_ptr(), b["n_act"].data_ptr(),
                            b["miss"].data_ptr(), b["n_miss"].data_ptr(),
                            b["status"].data_ptr(), sp)
        self.fa.x = x_ptr
        S = dw.cache.n_stage
        for g in range(self.groups):
            if S > 0:
                cnt = min(S, self.max_miss - g * S)
                if ev_fill:
                    ev_fill[g][0].record()
                moe.expcache_fill(dw.cache.handle, self.layer, b["miss"].data_ptr(),
                                  b["n_miss"].data_ptr(), g * S, cnt, 0, b["status"].data_ptr(),
                                  sp)
                if ev_fill:
                    ev_fill[g][1].record()
            self.fa.group = g
            self.fa.stages = 1
            if ev_gu:
                ev_gu[0].record()
            moe.moe_expert_ffn(self.fa, sp)
            if ev_gu:
                ev_gu[1].record()
            self.fa.stages = 2
            moe.moe_expert_ffn(self.fa, sp)
            if ev_dn:
                ev_dn.record()
        self.ca.y = y_ptr
        moe.moe_combine(self.ca, sp)

    def layer_launches(self):
        """Kernels one decode moe_layer_forward launches for this layer and T:
        router + permutation + slot lookup (one kernel for T <= 8, else the
        router GEMM, top-k and the permutation), then with staging slots and
        one group the FFN kernel that gathers the misses itself, otherwise per
        group the gather (if staging) and the gate/up and down kernels, and the
        combine unless a single group's down kernel writes y."""
        S = self.dw.cache.n_stage
        route = 1 if self.T <= 8 else 3
        if S > 0 and self.groups == 1:
            return route + 1
        return route + self.groups * (2 + (1 if S > 0 else 0)) + (0 if self.groups == 1 else 1)


# --------------------------------------------------------------- decode
def max_over_ranks(torch, value, world, device):
    """The largest of `value` over the job's ranks: the job's timed region ends
    when its slowest rank does."""
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, steps, tokens_per_step, total_ms):
    """Whole-job throughput: every rank processed `steps` steps of
    `tokens_per_step` tokens within `total_ms` (the max over ranks)."""
    return world * steps * tokens_per_step / (total_ms * 1e-3)


def rank_draw0(rank, n_steps, base=1_000_000):
    """First token draw of a rank: the ranks draw disjoint token ranges."""
    return base + rank * n_steps


def bench_decode(args, torch, moe, gen, gd, dev, rank, world, local_rank, peaks, wl=None):
    # the captured DRAM traffic is that of the NVFP4 decode layer's gate/up kernel
    traffic_captured = wl is None and not args.small
    wl = wl or gen.WORKLOADS["decode"]
    H, I, E, k, Is = wl.H, wl.I, wl.E, wl.k, wl.Is
    T = 1
    # --small: the same layer with only 16 distinct expert records (expert e
    # reads slot e mod 16): same kernels and launch shapes, ~0.5 GB on the
    # device, for profiler captures; not a bench value
    dw = gd.build(wl, T_max=T, slot_alias=16 if args.small else 0)
    layer = dw.moe_layers[0]
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    n_steps = args.warmup + args.steps
    xs = torch.empty((n_steps, H), dtype=torch.bfloat16, device=dev)
    gen.dev_x_bf16(wl.seed, 0, rank_draw0(rank, n_steps), n_steps, H, xs.data_ptr(), sp)
    ys = torch.empty((n_steps, H), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(torch, args.flush_mb, dev)
    ex = ExplicitLayer(torch, moe, dw, 0, T)

    # ---- pass 1 (headline): moe_layer_forward, each step replayed from a CUDA graph
    layer.forward(xs[0:1], ys[0:1])  # eager once before capture
    torch.cuda.synchronize()
    graphs = []
    for i in range(n_steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            layer.forward(xs[i:i + 1], ys[i:i + 1], stream=stream)
        graphs.append(g)
    torch.cuda.synchronize()

    def warm():
        for i in range(args.warmup):
            flush()
            graphs[i].replay()
    prewarm(torch, warm, args.prewarm_s)
    ev = _events(torch, args.steps)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for j in range(args.steps):
        flush()
        ev[j][0].record(stream)
        graphs[args.warmup + j].replay()
        ev[j][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    total_ms = sum(a.elapsed_time(b) for a, b in ev)
    del graphs
    assert layer.read_status() == 0, "device status set during the bench"

    # ---- pass 2: events at the layer's own launch boundaries (its timing hook),
    # eager launches, one step at a time: router kernel (with the permutation,
    # lookup and the shared expert's gate/up), gate/up kernel (routed, with the
    # shared expert's down), down kernel (routed, with the combine)
    hev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in hev:  # torch creates the CUDA event on its first record
        e.record(stream)
    torch.cuda.synchronize()
    moe.moe_layer_set_timing(layer.handle, [e.cuda_event for e in hev])
    k_ms = [[], [], []]
    for j in range(args.steps):
        flush()
        layer.forward(xs[args.warmup + j:args.warmup + j + 1],
                      ys[args.warmup + j:args.warmup + j + 1], stream=stream)
        hev[3].synchronize()
        for i in range(3):
            k_ms[i].append(hev[i].elapsed_time(hev[i + 1]))
    moe.moe_layer_set_timing(layer.handle, [])
    rt_ms, gu_ms, dn_ms = (statistics.mean(v) for v in k_ms)
    assert layer.read_status() == 0, "device status set during the bench"

    # ---- e2e: the public call with host buffers: the token in pinned host
    # memory (the layer's first kernel copies it in), the output written by
    # the layer's last kernel into pinned host memory
    xh = torch.empty((n_steps, H), dtype=torch.bfloat16, pin_memory=True)
    xh.copy_(xs.cpu())
    yh = torch.empty((n_steps, H), dtype=torch.bfloat16, pin_memory=True)
    e2e_steps = min(args.steps, 500)
    for i in range(args.warmup):
        layer.forward(xh[i:i + 1], yh[i:i + 1])
    torch.cuda.synchronize()
    e2e_ms = []
    for j in range(e2e_steps):
        i = args.warmup + j
        flush()
        a, bb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        layer.forward(xh[i:i + 1], yh[i:i + 1])
        bb.record(stream)
        bb.synchronize()
        e2e_ms.append(a.elapsed_time(bb))
    assert layer.read_status() == 0

    total_ms = max_over_ranks(torch, total_ms, world, dev)
    rb = gen.record_bytes(H, I, wl.fmt)
    # algorithmic bytes of the three kernels of the one-token sequence: the
    # router kernel (router weights, the shared expert's gate/up, x, h_shared,
    # logits), gate/up (the k records' gate and up rows with their scales, the
    # shared down, x, h written, h_shared read, o_shared written), down (the k
    # records' down rows and scales, h read, o_route written, the combine's
    # reads of o_route and o_shared, y)
    blk = 32 if wl.fmt == gen.MXFP4 else 16
    rt_bytes = E * H * 4 + 2 * Is * H * 2 + T * H * 2 + T * Is * 4 + T * E * 4
    gu_bytes = (k * (2 * I * H // 2 + 2 * I * H // blk) + H * Is * 2 + T * H * 2
                + T * k * I * 4 + T * Is * 4 + T * H * 4)
    dn_bytes = (k * (H * I // 2 + H * I // blk) + T * k * I * 4 + (T * k + T) * H * 4 * 2
                + T * H * 2)
    step_bytes = k * rb + 3 * Is * H * 2 + E * H * 4 + 2 * T * H * 2
    rt_gbs = rt_bytes / (rt_ms * 1e-3) / 1e9
    gu_gbs = gu_bytes / (gu_ms * 1e-3) / 1e9
    dn_gbs = dn_bytes / (dn_ms * 1e-3) / 1e9
    hbm = peaks["hbm_gbs"]
    res = {
        "value": round(job_tokens_per_s(world, args.steps, T, total_ms), 2),
        "ms_per_step": round(total_ms / args.steps, 5),
        "roofline": {"bound": "hbm",
                     "kernel": "k_decode_gu as the layer launches it for one token (routed "
                               "gate/up of the 8 experts, SiLU*mul, + the bf16 shared "
                               "expert's down)",
                     "achieved": round(gu_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gu_gbs / hbm, 4),
                     "traffic": GU_TRAFFIC if traffic_captured else None,
                     "traffic_source": GU_TRAFFIC_SOURCE if traffic_captured else "not captured",
                     "bytes_per_launch": gu_bytes, "avg_launch_ms": round(gu_ms, 5)},
        "kernels": {
            "k_route_permute_small": {"ms": round(rt_ms, 5), "GB/s": round(rt_gbs, 1),
                                      "frac_hbm": round(rt_gbs / hbm, 4),
                                      "bytes": rt_bytes},
            "k_decode_gu": {"ms": round(gu_ms, 5), "GB/s": round(gu_gbs, 1),
                            "frac_hbm": round(gu_gbs / hbm, 4), "bytes": gu_bytes},
            "k_decode_down": {"ms": round(dn_ms, 5), "GB/s": round(dn_gbs, 1),
                              "frac_hbm": round(dn_gbs / hbm, 4), "bytes": dn_bytes},
            "timing": "the layer's timing hook: events at its launch boundaries, eager "
                      "launches, L2 flushed before each step",
            "step_bytes": step_bytes,
            "step_frac_hbm": round(step_bytes / (total_ms / args.steps * 1e-3) / 1e9 / hbm, 4)},
        "e2e": {"value": round(e2e_steps / (sum(e2e_ms) * 1e-3), 2), "unit": UNIT,
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
                "call": "moe_layer_forward on pinned host buffers: the token copied in by "
                        "the layer's first kernel, the output written by its last kernel into "
                        "pinned host memory, both inside the events"},
        "gpu_launches": ex.layer_launches() * args.steps,
        "clocks": clk,
        "wall_s": round(wall, 3),
    }
    dw.close()
    return res


# --------------------------------------------------------------- prefill
def _mx(gen, name):
    """The workload with MXFP4 records (own seed)."""
    import dataclasses
    wl = gen.WORKLOADS[name]
    return dataclasses.replace(wl, name=name + "-mx", fmt=gen.MXFP4, seed=wl.seed + 100)


PREFILL_GEMM_LABEL = ("supplementary, the routed FP4 GEMMs above the HBM ridge: 64 experts "
                      "(H=6144, I=2048, NVFP4, all resident), 8192 tokens top-8, 1024 routes per "
                      "expert, no shared expert")
PREFILL_MX_LABEL = ("prefill MoE layer with MXFP4 records (E8M0 scale per 32; MXFP4 "
                    "activations): 4096 tokens, H=6144, I=2048, 288 experts top-8, bf16 shared "
                    "expert, all resident, one launch per GEMM")


def _prefill_gemm_wl():
    import gen
    return gen.Workload("prefill-gemm", H=6144, I=2048, E=64, k=8, T=8192, layers=1, Is=0,
                        seed=6, prefill=True, group=0)


PREFILL_GEMM_WL = None


def bench_prefill(args, torch, moe, gen, gd, dev, peaks, group=None, wl=None, label=None):
    custom = wl is not None
    wl = wl if custom else gen.WORKLOADS["prefill"]
    if args.prefill_experts > 0:
        # profiler captures only: fewer experts and proportionally fewer tokens,
        # the same tokens per expert (tile shapes) and kernels
        E2 = args.prefill_experts
        wl = gen.Workload(**{**wl.__dict__, "name": "prefill-part", "E": E2,
                             "T": max(128, (wl.T * E2 // wl.E) // 128 * 128)})
    T, H, I, E, k, Is = wl.T, wl.H, wl.I, wl.E, wl.k, wl.Is
    # experts per launch group: all at once unless asked (every expert is
    # resident in HBM, so the walk needs no staging buffer)
    dw_group = (0 if args.prefill_group is None else args.prefill_group) if group is None else group
    dw = gd.build(wl, T_max=T, prefill_group=dw_group)
    layer = dw.moe_layers[0]
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    steps = args.prefill_steps
    n = args.warmup + steps
    xs = torch.empty((n, T, H), dtype=torch.bfloat16, device=dev)
    for i in range(n):
        gen.dev_x_bf16(wl.seed, 0, 3_000_000 + i * T, T, H, xs[i].data_ptr(), sp)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(torch, args.flush_mb, dev)

    def warm():
        for i in range(args.warmup):
            layer.forward(xs[i], y)
    prewarm(torch, warm, args.prewarm_s)
    ev = _events(torch, steps)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.2)
    torch.cuda.synchronize()
    for j in range(steps):
        flush()
        ev[j][0].record(stream)
        layer.forward(xs[args.warmup + j], y)
        ev[j][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    assert layer.read_status() == 0
    # e2e: the layer called on pinned host buffers (it copies the tokens in
    # with its first kernel; its last kernel writes the output into host memory)
    xh = xs[args.warmup:].cpu().pin_memory()
    yh = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    e2e = []
    for j in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        layer.forward(xh[j], yh)
        b.record(stream)
        b.synchronize()
        e2e.append(a.elapsed_time(b))
    # per-kernel pass: the layer's timing hook marks every kernel of the step
    # (router, permutation, token quantisation, tile tables, per launch group
    # the gate/up GEMM, h quantisation and down GEMM, the shared expert's two
    # GEMMs - the down one writes y - or else the combine); L2 flushed before
    # each step
    n_lg = (-(-min(T * k, E) // dw_group)) if dw_group else 1
    names = (["router", "permute", "quant_tokens", "tile_plan"]
             + [n for _ in range(n_lg) for n in ("gemm_gate_up", "quant_h", "gemm_down")]
             + (["gemm_shared_gate_up", "gemm_shared_down"] if Is else ["combine"]))
    hev = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
    for e in hev:
        e.record(stream)
    torch.cuda.synchronize()
    moe.moe_layer_set_timing(layer.handle, [e.cuda_event for e in hev])
    kt = {}
    n_hook = min(steps, 5)
    for j in range(n_hook):
        flush()
        layer.forward(xs[args.warmup + j], y)
        hev[-1].synchronize()
        for i, nm in enumerate(names):
            kt[nm] = kt.get(nm, 0.0) + hev[i].elapsed_time(hev[i + 1]) / n_hook
    moe.moe_layer_set_timing(layer.handle, [])
    assert layer.read_status() == 0
    rb = gen.record_bytes(H, I, wl.fmt)
    weight_bytes = E * rb + 3 * Is * H * 2 + E * H * 4
    flops_fp4 = 2.0 * T * k * (2 * I * H + H * I)
    flops_bf16 = 2.0 * T * 3 * Is * H
    gbs = (weight_bytes + 2 * T * H * 2) / (ms * 1e-3) / 1e9
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    # the routed GEMMs alone: FP4 tensor rate, and the weights (+ activation
    # codes and scales) they read against the HBM peak
    blk = 32 if wl.fmt == gen.MXFP4 else 16
    gu_ms, dn_ms = kt["gemm_gate_up"], kt["gemm_down"]
    R = T * k
    gu_bytes = E * (2 * I * H // 2 + 2 * I * H // blk) + R * (H // 2 + H // 16)
    dn_bytes = E * (H * I // 2 + H * I // blk) + R * (I // 2 + I // 16)
    gemm = {
        "gate_up": {"ms": round(gu_ms, 4),
                    "fp4_tflops": round(2.0 * R * 2 * I * H / (gu_ms * 1e-3) / 1e12, 1),
                    "frac_fp4": round(2.0 * R * 2 * I * H / (gu_ms * 1e-3) / 1e12 / fp4_peak, 4),
                    "frac_hbm": round(gu_bytes / (gu_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
        "down": {"ms": round(dn_ms, 4),
                 "fp4_tflops": round(2.0 * R * H * I / (dn_ms * 1e-3) / 1e12, 1),
                 "frac_fp4": round(2.0 * R * H * I / (dn_ms * 1e-3) / 1e12 / fp4_peak, 4),
                 "frac_hbm": round(dn_bytes / (dn_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
        "routes_per_expert": round(R / E, 1),
        "timing": "the layer's timing hook: events around each kernel, L2 flushed before each "
                  f"step, mean of {n_hook} steps"}
    res = {
        "workload": label or (
            "prefill MoE layer: 4096 tokens, H=6144, I=2048, 288 experts top-8, bf16 "
            "shared expert, all experts resident, experts walked in act_list order in "
            + (f"launch groups of {dw_group}" if dw_group else "one launch per GEMM")),
        "value": round(T / (ms * 1e-3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
        "roofline": {
            "bound": "hbm", "unit": "GB/s",
            "kernel": "prefill expert FFN (NVFP4 quantisation + tcgen05 mxf4nvf4 grouped GEMMs + "
                      "bf16 shared-expert GEMMs) and router, whole step",
            "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
            "frac": round(gbs / peaks["hbm_gbs"], 4),
            "bytes_per_step": weight_bytes + 2 * T * H * 2},
        "fp4_tensor": {"achieved_tflops": round(flops_fp4 / (ms * 1e-3) / 1e12, 1),
                       "peak_tflops": round(fp4_peak, 1),
                       "frac": round(flops_fp4 / (ms * 1e-3) / 1e12 / fp4_peak, 4),
                       "peak_source": "measured bf16 burst x 6 (nominal FP4/bf16 ratio)",
                       "routed_fp4_tflop_per_step": round(flops_fp4 / 1e12, 3),
                       "shared_bf16_tflop_per_step": round(flops_bf16 / 1e12, 3)},
        "e2e": {"value": round(T / (statistics.mean(e2e) * 1e-3), 1), "unit": UNIT,
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
                "call": "moe_layer_forward on pinned host buffers (tokens copied in by the "
                        "layer's first kernel, output written into host memory by its last)"},
        "kernels_ms": {nm: round(v, 4) for nm, v in kt.items()},
        "routed_gemms": gemm,
        "clocks": clk,
    }
    dw.close()
    return res


# ------------------------------------------------- slot budgets (Maya page)
def bench_stack_budget(args, torch, moe, gen, gd, dev, link_gbs, calib_tokens=512, floor=33):
    """The 16-layer stack with per-layer slot budgets from the library's planner
    (expcache_plan_slots): every layer's route counts over a separate seeded
    calibration batch (the library's router on the device), the same total
    HBM slots as 66 per layer, a floor of 33; then the stack pass on fresh
    tokens (hit rate and tok/s beside the fixed 66 per layer)."""
    wl = gen.WORKLOADS["stack"]
    L = wl.layers if args.layers <= 0 else min(args.layers, wl.layers)
    E, H, k = wl.E, wl.H, wl.k
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    counts = torch.zeros((L, E), dtype=torch.int32, device=dev)
    x = torch.empty((calib_tokens, H), dtype=torch.bfloat16, device=dev)
    wr = torch.empty((E, H), dtype=torch.float32, device=dev)
    ids = torch.empty((calib_tokens, k), dtype=torch.int32, device=dev)
    w = torch.empty((calib_tokens, k), dtype=torch.float32, device=dev)
    lg = torch.empty((calib_tokens, E), dtype=torch.float32, device=dev)
    for l in range(L):
        gen.dev_router_f32(wl.seed, l, E, H, wr.data_ptr(), sp)
        gen.dev_x_bf16(wl.seed, l, 9_000_000, calib_tokens, H, x.data_ptr(), sp)
        b, _ = gen.zipf_bias(wl.seed, l, E, wl.zipf_alpha)
        bd = torch.from_numpy(b).to(dev)
        ra = moe.moe_route_args()
        ra.x, ra.w_router, ra.bias = x.data_ptr(), wr.data_ptr(), bd.data_ptr()
        ra.T, ra.H, ra.E, ra.k = calib_tokens, H, E, k
        ra.ids, ra.w, ra.p_sel, ra.logits = ids.data_ptr(), w.data_ptr(), None, lg.data_ptr()
        moe.moe_route(ra, sp)
        counts[l] = torch.bincount(ids.flatten().long(), minlength=E).int()
    ls = torch.zeros(L + 1, dtype=torch.int32, device=dev)
    order = torch.zeros((L, E), dtype=torch.int32, device=dev)
    total = L * wl.hot
    moe.expcache_plan_slots(counts.data_ptr(), L, E, total, floor, ls.data_ptr(),
                            order.data_ptr(), sp)
    torch.cuda.synchronize()
    n = (ls[1:] - ls[:-1]).tolist()
    resident = [order[l, :n[l]].tolist() for l in range(L)]
    res = bench_multilayer(args, torch, moe, gen, gd, dev, "stack", link_gbs, resident=resident)
    res["workload"] = (f"{L} decode layers, 1 token per step, per-layer Zipf bias, "
                       f"{total} HBM slots split by the greedy per-layer budget (floor {floor}) "
                       f"from {calib_tokens} calibration tokens per layer, misses gathered from "
                       "pinned host memory")
    res["slots_per_layer"] = n
    return res


# ------------------------------------------- prefill over a partly cached layer
def bench_prefill_streamed(args, torch, moe, gen, gd, dev, peaks, link_gbs, resident_ms=None):
    """4096-token prefill of the stack's layer (66 hot experts in HBM, the
    other 222 in pinned host memory), the misses gathered on the layer's
    second stream into the two halves of a 64-slot staging ring while the
    GEMMs run: tok/s, the gathered bytes against the measured host link, and
    the time saved against running the gather and the all-resident step one
    after the other."""
    wl = gen.WORKLOADS["stack"]
    T, H, I, k = 4096, wl.H, wl.I, wl.k
    dw = gd.build(wl, layers=1, T_max=T, n_stage=64, prefill_min_tokens=8, prefill_group=0)
    layer = dw.moe_layers[0]
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    steps = max(3, args.prefill_steps // 2)
    n = args.warmup + steps
    xs = torch.empty((n, T, H), dtype=torch.bfloat16, device=dev)
    for i in range(n):
        gen.dev_x_bf16(wl.seed, 0, 7_000_000 + i * T, T, H, xs[i].data_ptr(), sp)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(torch, args.flush_mb, dev)
    for i in range(args.warmup):
        layer.forward(xs[i], y)
    ev = _events(torch, steps)
    from routed_expert_layer_router_gb300.layer import device_view
    nact = moe.moe_layer_debug_ptrs(layer.handle)["n_act"]
    miss = 0
    torch.cuda.synchronize()
    for j in range(steps):
        flush()
        ev[j][0].record(stream)
        layer.forward(xs[args.warmup + j], y)
        ev[j][1].record(stream)
        ev[j][1].synchronize()
        na, nh = device_view(nact, (2,), torch.int32).tolist()
        miss += na - nh
    assert layer.read_status() == 0
    ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    rb = gen.record_bytes(H, I)
    gbytes = miss / steps * rb
    res = {
        "workload": "prefill of the stack's layer: 4096 tokens, 66 hot experts of 288 in HBM, "
                    "the misses gathered from pinned host memory through a 64-slot staging "
                    "ring (2 x 32) on a second stream while the tensor-core GEMMs run",
        "value": round(T / (ms * 1e-3), 1), "unit": UNIT, "ms_per_step": round(ms, 3),
        "misses_per_step": round(miss / steps, 1),
        "roofline": {"bound": "link", "achieved": round(gbytes / (ms * 1e-3) / 1e9, 1),
                     "peak": round(link_gbs, 1), "unit": "GB/s",
                     "frac": round(gbytes / (ms * 1e-3) / 1e9 / link_gbs, 4),
                     "bytes_per_step": int(gbytes),
                     "peak_source": "measured pinned host->device cudaMemcpyAsync (1 GiB)"},
    }
    if resident_ms:
        serial = gbytes / (link_gbs * 1e9) * 1e3 + resident_ms
        res["overlap"] = {"gather_at_link_ms": round(gbytes / (link_gbs * 1e9) * 1e3, 3),
                          "all_resident_step_ms": round(resident_ms, 3),
                          "saved_ms_vs_one_after_the_other": round(serial - ms, 3)}
    dw.close()
    return res


# ------------------------------------------------------------------- router
def bench_route(args, torch, moe, gen, dev, T=4096):
    """The router alone at the prefill shape (T tokens, fp32 weights [E][H]):
    moe_route per call, CUDA events around each, L2 flushed between calls."""
    wl = gen.WORKLOADS["prefill"]
    H, E, k = wl.H, wl.E, wl.k
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    wr = torch.empty((E, H), dtype=torch.float32, device=dev)
    gen.dev_router_f32(wl.seed, 0, E, H, wr.data_ptr(), sp)
    n = args.warmup + args.prefill_steps
    xs = torch.empty((n, T, H), dtype=torch.bfloat16, device=dev)
    for i in range(n):
        gen.dev_x_bf16(wl.seed, 0, 5_000_000 + i * T, T, H, xs[i].data_ptr(), sp)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    lg = torch.empty((T, E), dtype=torch.float32, device=dev)
    split = torch.empty(moe.moe_route_split_bytes(E, H), dtype=torch.uint8, device=dev)
    flush = L2Flush(torch, args.flush_mb, dev)

    def timed(use_split):
        a = moe.moe_route_args()
        a.w_router, a.T, a.H, a.E, a.k = wr.data_ptr(), T, H, E, k
        a.ids, a.w, a.logits = ids.data_ptr(), w.data_ptr(), lg.data_ptr()
        if use_split:
            a.w_split, a.w_split_bytes = split.data_ptr(), split.numel()
        for i in range(args.warmup):
            a.x = xs[i].data_ptr()
            moe.moe_route(a, sp)
        ev = _events(torch, args.prefill_steps)
        torch.cuda.synchronize()
        for j in range(args.prefill_steps):
            flush()
            a.x = xs[args.warmup + j].data_ptr()
            ev[j][0].record(stream)
            moe.moe_route(a, sp)
            ev[j][1].record(stream)
        torch.cuda.synchronize()
        return sum(x.elapsed_time(y) for x, y in ev) / args.prefill_steps * 1e3

    us_tc, us_simt = timed(True), timed(False)
    flops = 2.0 * T * E * H
    return {"workload": f"router: {T} tokens, H={H}, {E} experts top-{k}, fp32 weights and "
                        "logits, softmax/top-k",
            "us_per_call": round(us_tc, 2),
            "path": "tensor cores: weights split into three bf16 pieces, 64-deep partial sums "
                    "added with compensation",
            "fp32_equiv_tflops": round(flops / (us_tc * 1e-6) / 1e12, 2),
            "simt": {"us_per_call": round(us_simt, 2), "path": "SIMT fp32 FMA, Kahan per "
                     "32-value chunk", "fp32_tflops": round(flops / (us_simt * 1e-6) / 1e12, 2)}}


# --------------------------------------------------------------- stack / flat
def _saliency_order(torch, moe, gen, wl, layers, dev, n_tokens=512):
    """Per layer, experts by decreasing routing-weight mass over a separate
    seeded calibration batch (computed with the library's router)."""
    orders = []
    for l in range(layers):
        wr = torch.empty((wl.E, wl.H), dtype=torch.float32, device=dev)
        gen.dev_router_f32(wl.seed, l, wl.E, wl.H, wr.data_ptr(), 0)
        x = torch.empty((n_tokens, wl.H), dtype=torch.bfloat16, device=dev)
        gen.dev_x_bf16(wl.seed + 1000, l, 0, n_tokens, wl.H, x.data_ptr(), 0)
        ids = torch.empty((n_tokens, wl.k), dtype=torch.int32, device=dev)
        w = torch.empty((n_tokens, wl.k), dtype=torch.float32, device=dev)
        lg = torch.empty((n_tokens, wl.E), dtype=torch.float32, device=dev)
        a = moe.moe_route_args()
        a.x, a.w_router, a.T, a.H, a.E, a.k = x.data_ptr(), wr.data_ptr(), n_tokens, wl.H, wl.E, wl.k
        a.ids, a.w, a.logits = ids.data_ptr(), w.data_ptr(), lg.data_ptr()
        moe.moe_route(a, 0)
        torch.cuda.synchronize()
        sal = torch.zeros(wl.E, dtype=torch.float64, device=dev)
        sal.index_add_(0, ids.view(-1).long(), w.view(-1).double())
        s = sal.cpu().numpy()
        orders.append(sorted(range(wl.E), key=lambda e: (-s[e], e)))
    return orders


def _skip_error(torch, dw, xs, i0, n, L, T):
    """The renorm-skip against the exact layer on the same cache and inputs:
    per layer and token max |y_skip - y_exact| / rms(y_exact), and the routes
    dropped per layer forward (one token per forward: k - active experts)."""
    from routed_expert_layer_router_gb300 import moe
    from routed_expert_layer_router_gb300.layer import MoELayer, device_view
    wl = dw.wl
    errs, dropped = [], []
    exact = [MoELayer(dw.cache, l, dw.w_router[l], dw.gscale[l], wl.k, bias=dw.bias[l],
                      shared=dw.shared[l], T_max=T) for l in range(L)]
    try:
        ys = torch.empty((T, wl.H), dtype=torch.bfloat16, device=xs.device)
        ye = torch.empty_like(ys)
        for i in range(i0, i0 + n):
            for l in range(L):
                dw.moe_layers[l].forward(xs[i, l], ys)
                na = int(device_view(moe.moe_layer_debug_ptrs(dw.moe_layers[l].handle)["n_act"],
                                     (2,), torch.int32)[0].item())
                exact[l].forward(xs[i, l], ye)
                a, b = ys.float(), ye.float()
                errs.append(((a - b).abs().max() / b.pow(2).mean().sqrt()).item())
                dropped.append(wl.k * T - na)
    finally:
        for m in exact:
            m.close()
    return {"dropped_routes_per_layer_step": round(sum(dropped) / len(dropped), 2),
            "error_vs_exact": {"max_abs_over_rms_mean": round(sum(errs) / len(errs), 4),
                               "max_abs_over_rms_max": round(max(errs), 4),
                               "forwards": len(errs)}}


def bench_multilayer(args, torch, moe, gen, gd, dev, name, link_gbs, spares=0, skip_tau=0.0,
                     resident=None):
    """resident (per layer): the experts each layer caches, instead of the
    workload's rule (its slot run is sized to them)."""
    wl = gen.WORKLOADS[name]
    L = wl.layers if args.layers <= 0 else min(args.layers, wl.layers)
    T = wl.T
    order = _saliency_order(torch, moe, gen, wl, L, dev) if wl.hot_rule == "saliency" else None
    n_stage = 64 if T > 1 else None
    # one host copy per expert id, shared by the layers (host memory bound;
    # the bytes each miss moves over the link are the same)
    # spares > 0: the adaptive cache, its spare slots taken from the hot budget
    dw = gd.build(wl, layers=L, T_max=T, saliency_order=order, n_stage=n_stage,
                  alias_host_records=True, spares=spares, skip_tau=skip_tau,
                  resident=None if resident is None else resident[:L])
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    steps = args.stack_steps
    # Warm-up on a stream of distinct tokens, not a few tokens repeated: the
    # first device read of a host record is several times slower than later
    # ones, and a few repeated tokens leave most experts' records unread until
    # the timed steps.  The adaptive cache also learns from the routes it sees;
    # its gather pass runs on fresh tokens too, so that its hit rate is that of
    # new input.
    n_warm = max(args.warmup, -(-STACK_WARM_TOKENS // T))  # steps of T tokens
    g0 = n_warm + (steps if spares > 0 else 0)  # first token of the gather pass
    n = g0 + steps
    xs = torch.empty((n, L, T, wl.H), dtype=torch.bfloat16, device=dev)
    for i in range(n):
        for l in range(L):
            gen.dev_x_bf16(wl.seed, l, 5_000_000 + i * T, T, wl.H, xs[i, l].data_ptr(), sp)
    y = torch.empty((L, T, wl.H), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(torch, args.flush_mb, dev)
    layers = dw.moe_layers

    def fwd(i):
        for l in range(L):
            layers[l].forward(xs[i, l], y[l])

    if n_warm > args.warmup:
        for i in range(n_warm):
            fwd(i)
        torch.cuda.synchronize()
    else:
        prewarm(torch, lambda: [fwd(i) for i in range(args.warmup)], args.prewarm_s)
    ev = _events(torch, steps)
    torch.cuda.synchronize()
    host_ms = []
    for j in range(steps):
        flush()
        t_h = time.perf_counter()
        ev[j][0].record(stream)
        fwd(n_warm + j)
        ev[j][1].record(stream)
        # a decode step ends on the host (the next token depends on this one)
        ev[j][1].synchronize()
        host_ms.append((time.perf_counter() - t_h) * 1e3)
    torch.cuda.synchronize()
    # median over the steps (and p10 / p90 beside it): a few steps of a fresh
    # stream can take several times the rest
    step_ms = sorted(a.elapsed_time(b) for a, b in ev)
    ms = statistics.median(step_ms)
    p10, p90 = step_ms[int(0.1 * (steps - 1))], step_ms[int(0.9 * (steps - 1))]
    for l in range(L):
        assert layers[l].read_status() == 0
    # gather pass: the same forwards, with the layer timing hook's events at
    # every launch step of each layer; a gather's time is the interval that
    # ends at its own mark (the mark before it closes the permutation or the
    # previous group's down kernel)
    S = dw.cache.n_stage
    groups = (min(T * wl.k, wl.E) + S - 1) // S if S > 0 else 1
    # marks before the first group: start, router (+ permutation), and the
    # adaptive cache's step when it is a kernel of its own (more than 8 tokens)
    first = (2 if T <= 8 else 3) + (1 if spares > 0 and T > 8 else 0)
    # one staging group: the FFN kernel gathers the misses itself (one mark);
    # else per group a gather and the FFN, then the combine
    ffn_gathers = S > 0 and groups == 1
    marks = first + (1 if ffn_gathers else groups * (3 if S > 0 else 2)) + (1 if groups > 1 else 0)
    hev = [[torch.cuda.Event(enable_timing=True) for _ in range(marks)] for _ in range(L)]
    for e in (e for row in hev for e in row):  # torch creates the CUDA event on its first record
        e.record(stream)
    torch.cuda.synchronize()
    for l in range(L):
        moe.moe_layer_set_timing(layers[l].handle, [e.cuda_event for e in hev[l]])
    from routed_expert_layer_router_gb300.layer import device_view
    nact = [moe.moe_layer_debug_ptrs(layers[l].handle)["n_act"] for l in range(L)]
    fill_ms, miss, act = 0.0, 0, 0
    part_ms = [0.0] * (marks - 1)  # per interval between marks, summed over layers and steps
    hook_ms = 0.0                  # whole steps of this pass
    pev = _events(torch, steps)
    pass_ms = []
    for j in range(steps if S > 0 else 0):
        flush()
        pev[j][0].record(stream)
        fwd(g0 + j)
        pev[j][1].record(stream)
        torch.cuda.synchronize()
        pass_ms.append(pev[j][0].elapsed_time(pev[j][1]))
        hook_ms += pass_ms[-1]
        for l in range(L):
            for i in range(1, marks):
                part_ms[i - 1] += hev[l][i - 1].elapsed_time(hev[l][i])
            if ffn_gathers:  # the FFN launch that moves the misses
                fill_ms += hev[l][first - 1].elapsed_time(hev[l][first])
            else:
                for g in range(groups):
                    i = first + g * 3
                    fill_ms += hev[l][i - 1].elapsed_time(hev[l][i])
        for l in range(L):
            # n_act of the layer's last forward: [active, hits]
            na, nh = (int(v) for v in device_view(nact[l], (2,), torch.int32).tolist())
            act += na
            miss += na - nh
    for l in range(L):
        moe.moe_layer_set_timing(layers[l].handle, [])
        assert layers[l].read_status() == 0
    skip_res = None
    if skip_tau > 0:
        skip_res = _skip_error(torch, dw, xs, g0, min(steps, 16), L, T)
    rb = gen.record_bytes(wl.H, wl.I)
    gather_gbs = miss * rb / (fill_ms * 1e-3) / 1e9 if fill_ms > 0 else 0.0
    res = {
        "workload": (f"{L} decode layers, {T} token(s) per step, "
                     + (("per-layer Zipf bias (alpha 1.556), 66 hot experts per layer in HBM"
                         + (f", renorm-skip of misses with weight < {skip_tau} (approximate)"
                            if skip_tau > 0 else "")
                         if spares == 0 else
                         f"per-layer Zipf bias (alpha 1.556), 66 slots per layer in HBM: the "
                         f"{66 - spares} hottest resident at start and {spares} spares, adaptive "
                         f"cache (promotion on miss, decayed LFU eviction)")
                        if name == "stack" else
                        "unbiased routing, 72 experts per layer cached by saliency")
                     + ", misses gathered from pinned host memory"),
        "value": round(T / (ms * 1e-3), 2), "unit": UNIT + " (whole stack)",
        "ms_per_step": round(ms, 4),
        "ms_per_step_p10_p90": [round(p10, 4), round(p90, 4)],
        "host_ms_per_step_median": round(statistics.median(host_ms), 4),
        "per_layer_tokens_s": round(T * L / (ms * 1e-3), 1),
        "hit_rate": round(1 - miss / max(act, 1), 4),
        "misses_per_layer_step": round(miss / (steps * L), 2),
        "roofline": {"bound": "link",
                     "kernel": ("k_decode_ffn with the misses' gather inside (bytes gathered / "
                                "the whole launch: a lower bound of the link rate)"
                                if ffn_gathers else "k_gather (expcache_fill)"),
                     "achieved": round(gather_gbs, 1), "peak": round(link_gbs, 1),
                     "unit": "GB/s", "frac": round(gather_gbs / link_gbs, 4) if link_gbs else None,
                     "peak_source": "measured pinned host->device cudaMemcpyAsync (1 GiB)"},
        "host_records": "one host copy per expert id, shared by the layers",
    }
    if skip_res is not None:
        res["renorm_skip"] = {"tau": skip_tau, **skip_res}
    if S > 0 and steps > 0:
        # the gather pass's own step time and its launch-step intervals, per
        # layer (us): router (+ permutation, + the adaptive cache's step for up
        # to 8 tokens), the policy step (more tokens), then the FFN with its
        # gather (one staging group) or per group the gather, gate/up and down
        res["gather_pass"] = {"ms_per_step": round(hook_ms / steps, 4),
                              "ms_per_step_median": round(statistics.median(pass_ms), 4),
                              "us_per_layer": [round(v * 1e3 / (steps * L), 1) for v in part_ms]}
    dw.close()
    return res


# ------------------------------------------------------- CPU oracle timing
def oracle_sample(seconds: float, wl_name: str = "decode", mode: int = 0, batch: int = 1):
    """Times the oracle (as it stands) on tokens of the workload's layer, `batch`
    tokens per call, until `seconds` of CPU work are spent (record generation
    excluded); mode 1 = prefill numerics.  Returns (tokens/s, tokens, threads, s)."""
    import gen
    import oracle
    wl = gen.WORKLOADS[wl_name]
    Wr = gen.router_f32(wl.seed, 0, wl.E, wl.H)
    sh = gen.shared_bf16(wl.seed, 0, wl.Is, wl.H)
    g = gen.global_scales(wl.seed, 0, wl.E)
    x = gen.x_bf16(wl.seed, 0, 2_000_000, 64, wl.H)
    ids, *_ = oracle.route(x, Wr, None, wl.k)
    n_done, t_spent = 0, 0.0
    recs = {}
    while t_spent < seconds and n_done + batch <= 64:
        sl = slice(n_done, n_done + batch)
        need = [int(e) for e in set(ids[sl].ravel().tolist()) if int(e) not in recs]
        if need:
            for e, r in zip(need, gen.expert_records(wl.seed, 0, need, wl.H, wl.I)):
                recs[e] = r
        t0 = time.perf_counter()
        oracle.layer_forward(x[sl], wl.H, wl.I, wl.E, wl.k, Wr, None,
                             {int(e): recs[int(e)] for e in ids[sl].ravel()}, g, shared_w=sh,
                             mode=mode)
        t_spent += time.perf_counter() - t0
        n_done += batch
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return n_done / t_spent, n_done, threads, t_spent


def _oracle_single_thread(seconds: float, wl_name: str, mode: int):
    """oracle_sample in a child process with OMP_NUM_THREADS=1."""
    import subprocess
    code = ("import json, bench; print(json.dumps(bench.oracle_sample(%r, %r, %d, 1)))"
            % (seconds, wl_name, mode))
    env = {**os.environ, "OMP_NUM_THREADS": "1"}
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         cwd=os.path.dirname(os.path.abspath(__file__)), timeout=600)
    tps, n, threads, spent = json.loads(out.stdout.strip().splitlines()[-1])
    return tps, n, spent


def _cpu_model() -> str:
    try:
        out = subprocess_run(["lscpu"])
        for ln in out.splitlines():
            if ln.strip().startswith("Model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part")):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def subprocess_run(cmd):
    import subprocess
    return subprocess.run(cmd, capture_output=True, text=True, timeout=30).stdout


def cpu_baseline(seconds: float) -> dict:
    """The oracle timed on this host: decode tokens and prefill tokens (the
    4096-token layer's numerics, a sample of its tokens), on all cores
    (OpenMP over the tokens of a call and the rows of each product) and on
    one thread, with the CPU model."""
    tps, n, threads, spent = oracle_sample(seconds)
    res = {"value": round(tps, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
           "sample": f"{n} decode tokens of the same layer ({spent:.1f} s)",
           "cpu_model": _cpu_model()}
    try:
        t1, n1, s1 = _oracle_single_thread(seconds / 3, "decode", 0)
        res["single_thread"] = {"value": round(t1, 4), "unit": UNIT, "cores": 1,
                                "sample": f"{n1} decode tokens ({s1:.1f} s)"}
    except Exception as exc:
        res["single_thread"] = {"error": repr(exc)}
    try:
        tp, n_p, _, sp_ = oracle_sample(seconds / 2, "prefill", 1, batch=threads)
        res["prefill"] = {"value": round(tp, 4), "unit": UNIT, "cores": threads,
                          "sample": f"{n_p} tokens of the 4096-token prefill layer in its "
                                    f"prefill numerics, {threads} per call ({sp_:.1f} s)"}
        t1, n1, s1 = _oracle_single_thread(seconds / 3, "prefill", 1)
        res["prefill_single_thread"] = {"value": round(t1, 4), "unit": UNIT, "cores": 1,
                                        "sample": f"{n1} prefill tokens ({s1:.1f} s)"}
    except Exception as exc:
        res["prefill"] = {"error": repr(exc)}
    return res


def reference_steps(steps: int, warmup: int, budget_s: float, wl_name: str = "decode"):
    """The reference arm's steps: one decode token of the oracle (as it stands)
    each, drawn in turn from a pool of 64 seeded tokens.  `warmup` untimed
    steps, then `steps` timed ones, as many of them as fit in `budget_s` of
    oracle time (record generation excluded; the count is reported).
    Returns (timed steps, warm-up steps, seconds, threads)."""
    import gen
    import oracle
    wl = gen.WORKLOADS[wl_name]
    pool = 64
    Wr = gen.router_f32(wl.seed, 0, wl.E, wl.H)
    sh = gen.shared_bf16(wl.seed, 0, wl.Is, wl.H)
    g = gen.global_scales(wl.seed, 0, wl.E)
    x = gen.x_bf16(wl.seed, 0, 2_000_000, pool, wl.H)
    ids, *_ = oracle.route(x, Wr, None, wl.k)
    recs = {}

    def step(i):
        j = i % pool
        need = [int(e) for e in set(ids[j].ravel().tolist()) if int(e) not in recs]
        if need:
            for e, r in zip(need, gen.expert_records(wl.seed, 0, need, wl.H, wl.I)):
                recs[e] = r
        t0 = time.perf_counter()
        oracle.layer_forward(x[j:j + 1], wl.H, wl.I, wl.E, wl.k, Wr, None,
                             {int(e): recs[int(e)] for e in ids[j].ravel()}, g, shared_w=sh)
        return time.perf_counter() - t0

    n_warm, t_warm = 0, 0.0
    while n_warm < warmup and t_warm < budget_s:
        t_warm += step(n_warm)
        n_warm += 1
    n_done, t_spent = 0, 0.0
    while n_done < steps and (n_done == 0 or t_spent < budget_s):
        t_spent += step(n_warm + n_done)
        n_done += 1
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return n_done, n_warm, t_spent, threads


def run_reference(args, rank, world):
    if rank != 0:
        return None
    budget = min(max(args.ref_seconds, 5.0), 120.0)
    n, n_warm, spent, threads = reference_steps(args.steps, args.warmup, budget)
    tps = n / spent
    cut = "" if n == args.steps else f"; {args.steps} asked, cut to what fits in {budget:.0f} s"
    return {
        "impl": "reference", "metric": METRIC, "value": round(tps, 4), "unit": UNIT,
        "n_gpus": world, "steps": n, "warmup": n_warm, "ms_per_step": round(spent / n * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": "decode MoE layer: H=6144, I=2048, 288 experts top-8, bf16 shared "
                               "expert, NVFP4 experts; 1 token per forward", "global_batch": 1,
                   "seq_len": 1, "parallelism": "cpu"},
        "cpu_baseline": {"value": round(tps, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{n} timed decode tokens after {n_warm} untimed ones, one per "
                                   f"step ({spent:.1f} s of oracle time; record generation "
                                   f"excluded{cut})"},
        "e2e": {"value": round(tps, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_ours(args, rank, world, local_rank):
    import torch

    import gen
    import gen.device as gd
    from routed_expert_layer_router_gb300 import moe

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    # a non-default stream: graph capture and all timing happen on it
    torch.cuda.set_stream(torch.cuda.Stream(device=dev))
    moe.lib()
    global PREFILL_GEMM_WL
    PREFILL_GEMM_WL = _prefill_gemm_wl()
    peaks, peak_kind = _peaks()
    if args.only == "prefill":
        return {"prefill": bench_prefill(args, torch, moe, gen, gd, dev, peaks)}
    if args.only == "route":
        return {"route": bench_route(args, torch, moe, gen, dev)}
    if args.only in ("stack", "flat"):
        link = link_h2d_gbs(torch, dev)
        return {args.only: bench_multilayer(args, torch, moe, gen, gd, dev, args.only, link)}
    if args.only == "stack_skip":
        link = link_h2d_gbs(torch, dev)
        return {args.only: bench_multilayer(args, torch, moe, gen, gd, dev, "stack", link,
                                            skip_tau=SKIP_TAU)}
    if args.only == "stack_adaptive":
        link = link_h2d_gbs(torch, dev)
        return {args.only: bench_multilayer(args, torch, moe, gen, gd, dev, "stack", link,
                                            spares=ADAPTIVE_SPARES)}
    if args.only == "stack_budget":
        link = link_h2d_gbs(torch, dev)
        return {args.only: bench_stack_budget(args, torch, moe, gen, gd, dev, link)}
    if args.only == "prefill_streamed":
        link = link_h2d_gbs(torch, dev)
        return {args.only: bench_prefill_streamed(args, torch, moe, gen, gd, dev, peaks, link)}
    if args.only == "prefill_gemm":
        return {args.only: bench_prefill(args, torch, moe, gen, gd, dev, peaks, group=0,
                                         wl=PREFILL_GEMM_WL, label=PREFILL_GEMM_LABEL)}
    if args.only == "prefill_mx":
        return {args.only: bench_prefill(args, torch, moe, gen, gd, dev, peaks, group=0,
                                         wl=_mx(gen, "prefill"), label=PREFILL_MX_LABEL)}
    if args.only == "decode_mx":
        return {args.only: bench_decode(args, torch, moe, gen, gd, dev, rank, world, local_rank,
                                        peaks, wl=_mx(gen, "decode"))}
    d = bench_decode(args, torch, moe, gen, gd, dev, rank, world, local_rank, peaks)
    d["roofline"]["peak_source"] = (f"{peak_kind}: MEASURED_PEAKS.json hbm_gbs (copy)"
                                    if peak_kind == "measured" else "fallback 6.8 TB/s")
    out = {
        "metric": METRIC, "value": d["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": d["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4 weights (e2m1 + e4m3 per 16), fp32 accumulation, bf16 activations",
        "data": "synthetic (seeded; random-init NVFP4 experts, N(0,1) bf16 tokens)",
        "config": {"workload": "decode MoE layer: H=6144, I=2048, 288 experts top-8, fp32 "
                               "softmax router, bf16 shared expert I=2048, NVFP4 routed experts "
                               "all resident in HBM, 1 token per forward",
                   "global_batch": world, "seq_len": 1, "parallelism": f"replicas{world}",
                   "l2": L2Flush.describe_for(args.flush_mb),
                   "timing": "moe_layer_forward captured in one CUDA graph per step, CUDA events around each replay"},
        "roofline": d["roofline"], "kernels": d["kernels"], "e2e": d["e2e"],
        "gpu_launches": d["gpu_launches"], "clocks": d["clocks"], "wall_s": d["wall_s"],
    }
    torch.cuda.empty_cache()
    if rank == 0 and not args.decode_only and not args.small and args.only != "decode":
        also = {}
        # the link-bound stacks first: after the prefill passes (two 6 GB
        # layers built and freed) the gathers over the host link measured slower
        try:
            link = link_h2d_gbs(torch, dev)
            also["link_h2d_gbs"] = round(link, 1)
            for name, wname, sp, tau in (("stack", "stack", 0, 0.0), ("flat", "flat", 0, 0.0),
                                         ("stack_adaptive", "stack", ADAPTIVE_SPARES, 0.0),
                                         ("stack_skip", "stack", 0, SKIP_TAU)):
                try:
                    also[name] = bench_multilayer(args, torch, moe, gen, gd, dev, wname, link,
                                                  spares=sp, skip_tau=tau)
                except Exception as exc:
                    also[name] = {"error": repr(exc)}
                torch.cuda.empty_cache()
        except Exception as exc:
            also["link_h2d_gbs"] = {"error": repr(exc)}
        try:
            link = link if isinstance(also.get("link_h2d_gbs"), float) else link_h2d_gbs(torch, dev)
            also["stack_budget"] = bench_stack_budget(args, torch, moe, gen, gd, dev, link)
        except Exception as exc:
            also["stack_budget"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        try:
            also["prefill"] = bench_prefill(args, torch, moe, gen, gd, dev, peaks)
        except Exception as exc:  # reported, not hidden
            also["prefill"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        try:
            also["prefill_streamed"] = bench_prefill_streamed(
                args, torch, moe, gen, gd, dev, peaks, link_h2d_gbs(torch, dev),
                resident_ms=also["prefill"].get("ms_per_step"))
        except Exception as exc:
            also["prefill_streamed"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        for name, kw in (("prefill_gemm", dict(wl=PREFILL_GEMM_WL, label=PREFILL_GEMM_LABEL)),
                         ("prefill_mx", dict(wl=_mx(gen, "prefill"), label=PREFILL_MX_LABEL))):
            try:
                also[name] = bench_prefill(args, torch, moe, gen, gd, dev, peaks, group=0, **kw)
            except Exception as exc:
                also[name] = {"error": repr(exc)}
            torch.cuda.empty_cache()
        try:
            a2 = argparse.Namespace(**{**vars(args), "steps": min(args.steps, 300)})
            dm = bench_decode(a2, torch, moe, gen, gd, dev, rank, world, local_rank, peaks,
                              wl=_mx(gen, "decode"))
            also["decode_mx"] = {kk: dm[kk] for kk in ("value", "ms_per_step", "roofline",
                                                         "kernels")}
            also["decode_mx"]["workload"] = ("the decode layer with MXFP4 records (E8M0 scale "
                                             "per 32 values), 1 token per forward")
        except Exception as exc:
            also["decode_mx"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        try:  # the same layer walked in launch groups of 64 experts
            g64 = bench_prefill(args, torch, moe, gen, gd, dev, peaks,
                                group=gen.WORKLOADS["prefill"].group)
            also["prefill_groups64"] = {k: g64[k] for k in ("workload", "value", "unit",
                                                             "ms_per_step")}
        except Exception as exc:
            also["prefill_groups64"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        out["also"] = also
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--flush-mb", type=int, default=512)
    ap.add_argument("--prefill-group", type=int, default=None,
                    help="experts per prefill launch group (default: the workload's 64; 0 = all)")
    ap.add_argument("--prewarm-s", type=float, default=1.0)
    ap.add_argument("--prefill-steps", type=int, default=10)
    ap.add_argument("--stack-steps", type=int, default=20)
    ap.add_argument("--layers", type=int, default=0, help="layers of stack/flat (0 = all)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-only", action="store_true")
    ap.add_argument("--small", action="store_true",
                    help="16 distinct expert records (profiler captures only)")
    ap.add_argument("--only", default="",
                    choices=["", "decode", "prefill", "route", "stack", "flat",
                             "stack_adaptive", "stack_skip", "stack_budget", "prefill_streamed",
                             "prefill_gemm", "prefill_mx", "decode_mx"],
                    help="run one secondary workload alone (profiler captures)")
    ap.add_argument("--prefill-experts", type=int, default=0,
                    help="prefill with fewer experts, same tokens per expert (profiling)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    out = run_ours(args, rank, world, local_rank)
    if args.only:
        if rank == 0:
            print(json.dumps(out), flush=True)
        return
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
