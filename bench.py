"""Benchmark of the routed MoE layer on one GB300 (or N independent replicas).

Default workload: the decode MoE layer - hidden 6144, expert intermediate 2048,
288 experts top-8 (fp32 softmax router), one bf16 shared expert, NVFP4 routed
experts all resident in HBM, 1 token per forward.  A step is one pass of the
whole hot path (route -> permute -> cache lookup -> expert FFN gate/up ->
down -> combine) over one fresh token; L2 is flushed between steps (a write
of a buffer larger than L2, outside the timed events).

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
same workload instead (bounded sample, host cores).
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


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region."""

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
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
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


# --------------------------------------------------------------- our arm
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
    wl = gen.WORKLOADS["decode"]
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
    gen.dev_x_bf16(wl.seed, 0, 1_000_000 + rank * n_steps, n_steps, H, xs.data_ptr(), sp)
    ys = torch.empty((n_steps, H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(args.flush_mb << 20, dtype=torch.uint8, device=dev)

    # explicit buffers for the step made of the individual ABI calls
    i32, f32 = torch.int32, torch.float32
    b = {
        "logits": torch.empty((T, E), dtype=f32, device=dev),
        "ids": torch.empty((T, k), dtype=i32, device=dev),
        "w": torch.empty((T, k), dtype=f32, device=dev),
        "p": torch.empty((T, k), dtype=f32, device=dev),
        "counts": torch.empty(E, dtype=i32, device=dev),
        "offsets": torch.empty(E + 1, dtype=i32, device=dev),
        "perm": torch.empty(T * k, dtype=i32, device=dev),
        "inv": torch.empty(T * k, dtype=i32, device=dev),
        "src": torch.empty(E, dtype=i32, device=dev),
        "act": torch.empty(E, dtype=i32, device=dev),
        "n_act": torch.empty(2, dtype=i32, device=dev),
        "miss": torch.empty(E, dtype=i32, device=dev),
        "n_miss": torch.empty(1, dtype=i32, device=dev),
        "status": torch.zeros(1, dtype=i32, device=dev),
        "o_route": torch.empty((T * k, H), dtype=f32, device=dev),
        "o_shared": torch.empty((T, H), dtype=f32, device=dev),
    }
    ws_bytes = moe.moe_ffn_workspace_bytes(0, T, H, I, E, k, Is)
    ffn_ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ra = moe.moe_route_args()
    ra.w_router, ra.bias = dw.w_router[0].data_ptr(), None
    ra.T, ra.H, ra.E, ra.k = T, H, E, k
    ra.ids, ra.w, ra.p_sel, ra.logits = (b["ids"].data_ptr(), b["w"].data_ptr(),
                                         b["p"].data_ptr(), b["logits"].data_ptr())
    ra.status = b["status"].data_ptr()
    fa = moe.moe_ffn_args()
    fa.mode, fa.T, fa.H, fa.I, fa.E, fa.k = 0, T, H, I, E, k
    fa.cache, fa.gscale = dw.cache.handle, dw.gscale[0].data_ptr()
    fa.src_slot, fa.act_list, fa.n_act = b["src"].data_ptr(), b["act"].data_ptr(), b["n_act"].data_ptr()
    fa.offsets, fa.perm, fa.w = b["offsets"].data_ptr(), b["perm"].data_ptr(), b["w"].data_ptr()
    fa.group, fa.n_stage, fa.Is = 0, 0, Is
    fa.s_gate, fa.s_up, fa.s_down = (t.data_ptr() for t in dw.shared[0])
    fa.o_route, fa.o_shared = b["o_route"].data_ptr(), b["o_shared"].data_ptr()
    fa.workspace, fa.workspace_bytes = ffn_ws.data_ptr(), ws_bytes
    fa.status = b["status"].data_ptr()
    ca = moe.moe_combine_args()
    ca.T, ca.H, ca.k = T, H, k
    ca.o_route, ca.inv, ca.o_shared = b["o_route"].data_ptr(), b["inv"].data_ptr(), b["o_shared"].data_ptr()

    def step(i, ev=None):
        ra.x = xs[i].data_ptr()
        moe.moe_route(ra, sp)
        moe.moe_permute(b["ids"].data_ptr(), T, k, E, b["counts"].data_ptr(),
                        b["offsets"].data_ptr(), b["perm"].data_ptr(), b["inv"].data_ptr(), 0, 128,
                        b["status"].data_ptr(), sp)
        moe.expcache_lookup(dw.cache.handle, 0, b["counts"].data_ptr(), b["src"].data_ptr(),
                            b["act"].data_ptr(), b["n_act"].data_ptr(), b["miss"].data_ptr(),
                            b["n_miss"].data_ptr(), b["status"].data_ptr(), sp)
        fa.x = xs[i].data_ptr()
        fa.stages = 1
        if ev:
            ev[0].record(stream)
        moe.moe_expert_ffn(fa, sp)
        if ev:
            ev[1].record(stream)
        fa.stages = 2
        moe.moe_expert_ffn(fa, sp)
        if ev:
            ev[2].record(stream)
        ca.y = ys[i].data_ptr()
        moe.moe_combine(ca, sp)

    launches_per_step = 2 + 1 + 1 + 1 + 1 + 1  # route(2) permute lookup gu down combine

    # ---- pass 1 (headline): each step replayed from a CUDA graph -------------
    step(0)  # eager once before capture (one-time kernel attribute set-up)
    torch.cuda.synchronize()
    graphs = []
    for i in range(n_steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(i)
        graphs.append(g)
    torch.cuda.synchronize()
    for i in range(args.warmup):
        flush.zero_()
        graphs[i].replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for j in range(args.steps):
        flush.zero_()
        ev[j][0].record(stream)
        graphs[args.warmup + j].replay()
        ev[j][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(bb) for a, bb in ev]
    total_ms = sum(step_ms)

    # ---- pass 2: per-kernel events around the FFN launches (eager) -----------
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for j in range(args.steps):
        flush.zero_()
        step(args.warmup + j, kev[j])
    torch.cuda.synchronize()
    gu_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in kev)
    dn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in kev)
    assert int(b["status"].item()) == 0, "device status set during the bench"

    # ---- e2e: the public call with host buffers --------------------------------
    xh = torch.empty((n_steps, H), dtype=torch.bfloat16, pin_memory=True)
    xh.copy_(xs.cpu())
    yh = torch.empty((n_steps, H), dtype=torch.bfloat16, pin_memory=True)
    xd = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    yd = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    e2e_steps = min(args.steps, 500)
    for i in range(args.warmup):
        xd.copy_(xh[i:i + 1], non_blocking=True)
        layer.forward(xd, yd)
        yh[i:i + 1].copy_(yd, non_blocking=True)
    torch.cuda.synchronize()
    e2e_ms = []
    for j in range(e2e_steps):
        i = args.warmup + j
        flush.zero_()
        a, bb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        xd.copy_(xh[i:i + 1], non_blocking=True)
        layer.forward(xd, yd)
        yh[i:i + 1].copy_(yd, non_blocking=True)
        bb.record(stream)
        bb.synchronize()
        e2e_ms.append(a.elapsed_time(bb))
    assert layer.read_status() == 0

    # ---- aggregate over ranks -------------------------------------------------
    tot = torch.tensor([total_ms], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(tot, op=torch.distributed.ReduceOp.MAX)
    total_ms = float(tot.item())

    peaks, peak_kind = _peaks()
    rb = gen.record_bytes(H, I)
    gu_bytes = k * (2 * I * H // 2 + 2 * I * H // 16) + 2 * Is * H * 2 + T * H * 2 + (T * k * I + T * Is) * 4
    dn_bytes = k * (H * I // 2 + H * I // 16) + H * Is * 2 + (T * k * I + T * Is) * 4 + (T * k + T) * H * 4
    step_bytes = k * rb + 3 * Is * H * 2 + E * H * 4 + 2 * T * H * 2
    gu_gbs = gu_bytes / (gu_ms * 1e-3) / 1e9
    dn_gbs = dn_bytes / (dn_ms * 1e-3) / 1e9
    value = world * args.steps * T / (total_ms * 1e-3)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4 weights (e2m1+e4m3/16), fp32 accumulate, bf16 activations",
        "data": "synthetic (seeded; random-init NVFP4 experts, N(0,1) bf16 tokens)",
        "config": {"workload": "decode MoE layer: H=6144, I=2048, 288 experts top-8, fp32 softmax "
                               "router, bf16 shared expert I=2048, NVFP4 routed experts all "
                               "resident in HBM, 1 token per forward",
                   "global_batch": world * T, "seq_len": 1, "parallelism": f"replicas{world}",
                   "l2": f"flushed between steps ({args.flush_mb} MiB write, outside the events)",
                   "timing": "CUDA-graph replay per step, CUDA events around each replay"},
        "roofline": {"bound": "hbm", "kernel": "k_decode_gu (routed NVFP4 gate/up + shared bf16 "
                                               "gate/up, SiLU*mul)",
                     "achieved": round(gu_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gu_gbs / peaks["hbm_gbs"], 4), "traffic": None,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "bytes_per_launch": gu_bytes, "avg_launch_ms": round(gu_ms, 5)},
        "kernels": {
            "k_decode_gu": {"ms": round(gu_ms, 5), "GB/s": round(gu_gbs, 1),
                            "frac_hbm": round(gu_gbs / peaks["hbm_gbs"], 4)},
            "k_decode_down": {"ms": round(dn_ms, 5), "GB/s": round(dn_gbs, 1),
                              "frac_hbm": round(dn_gbs / peaks["hbm_gbs"], 4)},
            "step_hbm_frac": round(step_bytes / (total_ms / args.steps * 1e-3) / 1e9
                                   / peaks["hbm_gbs"], 4),
        },
        "e2e": {"value": round(e2e_steps / (sum(e2e_ms) * 1e-3), 2), "unit": UNIT,
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
                "call": "moe_layer_forward with pinned host input/output copies in the events"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s": round(wall, 3),
    }
    dw.close()
    return out


# ------------------------------------------------------- CPU oracle timing
def oracle_sample(seconds: float, wl_name: str = "decode"):
    """Times the oracle (as it stands) on decode tokens of the same workload
    until `seconds` of CPU work are spent; returns (tokens/s, tokens, threads)."""
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
    while t_spent < seconds and n_done < 64:
        need = [e for e in ids[n_done] if e not in recs]
        if need:
            for e, r in zip(need, gen.expert_records(wl.seed, 0, need, wl.H, wl.I)):
                recs[int(e)] = r
        t0 = time.perf_counter()
        oracle.layer_forward(x[n_done:n_done + 1], wl.H, wl.I, wl.E, wl.k, Wr, None,
                             {int(e): recs[int(e)] for e in ids[n_done]}, g, shared_w=sh)
        t_spent += time.perf_counter() - t0
        n_done += 1
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return n_done / t_spent, n_done, threads, t_spent


def run_reference(args, rank, world):
    if rank != 0:
        return None
    budget = min(max(args.ref_seconds, 5.0), 120.0)
    tps, n, threads, spent = oracle_sample(budget)
    return {
        "impl": "reference", "metric": METRIC, "value": round(tps, 4), "unit": UNIT,
        "n_gpus": world, "steps": n, "warmup": 0, "ms_per_step": round(spent / n * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": "decode MoE layer: H=6144, I=2048, 288 experts top-8, bf16 shared "
                               "expert, NVFP4 experts; 1 token per forward", "global_batch": 1,
                   "seq_len": 1, "parallelism": "cpu"},
        "cpu_baseline": {"value": round(tps, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{n} decode tokens ({spent:.1f} s of oracle time; records "
                                   f"generation excluded)"},
        "e2e": {"value": round(tps, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--flush-mb", type=int, default=512)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--small", action="store_true",
                    help="16 distinct expert records (profiler captures only)")
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
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            tps, n, threads, spent = oracle_sample(args.cpu_seconds)
            out["cpu_baseline"] = {"value": round(tps, 4), "unit": UNIT, "cores": threads,
                                   "kind": "oracle",
                                   "sample": f"{n} decode tokens of the same layer ({spent:.1f} s)"}
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
