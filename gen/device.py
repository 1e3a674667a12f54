"""Builds a workload's inputs on the GPU and wires them into the library:
router weights, global scales, shared expert, per-layer bias, expert records
(resident ones written straight into cache slots by the device generator,
the others into a pinned host arena), and one MoELayer per layer.

Holds no arithmetic of the layer: generation is the seeded generator, the
cache/placement decisions follow the workload recipe (all resident; the
smallest Zipf ranks; or a given saliency order).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import gen
from routed_expert_layer_router_gb300.layer import ExpertCache, HostArena, MoELayer


@dataclass
class DeviceWorkload:
    wl: gen.Workload
    layers: int
    cache: ExpertCache
    moe_layers: list
    w_router: list
    gscale: list            # device [E,3] per layer
    gscale_host: list       # numpy [E,3] per layer
    bias: list              # device or None per layer
    bias_host: list
    shared: list            # (g, u, d) device per layer or None
    resident: list          # per layer: sorted list of resident experts
    host_arena: HostArena | None = None
    # generator layer index whose records layer l uses (l itself, or 0 when
    # host records are aliased across layers)
    record_layer: list = field(default_factory=list)
    extra: dict = field(default_factory=dict)

    def close(self):
        for m in self.moe_layers:
            m.close()
        self.cache.close()
        if self.host_arena is not None:
            self.host_arena.close()


def _hot_set(wl: gen.Workload, layer: int, bias_rank, saliency_order, drop: int = 0):
    """The layer's hot experts (the `hot` first by rule), less the `drop`
    coldest of them."""
    if wl.hot <= 0 or wl.hot >= wl.E:
        return list(range(wl.E - drop))
    if wl.hot_rule == "zipf":
        return sorted(int(e) for e in np.argsort(bias_rank)[:wl.hot - drop])
    if wl.hot_rule == "saliency":
        return sorted(int(e) for e in saliency_order[layer][:wl.hot - drop])
    raise ValueError(wl.hot_rule)


def build(wl: gen.Workload, layers: int | None = None, T_max: int | None = None,
          n_stage: int | None = None, saliency_order=None, prefill_min_tokens: int | None = None,
          alias_host_records: bool = False, resident=None, slot_alias: int = 0,
          stream=None, prefill_group: int | None = None, spares: int = 0,
          skip_tau: float = 0.0) -> DeviceWorkload:
    """Device-resident layer(s) of workload `wl`.

    layers: how many of the workload's layers to build (default: all).
    n_stage: staging slots (default: enough for every miss of one layer).
    saliency_order: per layer, experts by decreasing saliency (hot_rule "saliency").
    alias_host_records: store one host copy per expert id shared by all layers
      (the host-index table maps every layer to it) when host memory is short;
      the records then repeat across layers for both the GPU and the oracle.
    skip_tau: > 0 turns on the layers' renorm-skip of low-weight misses.
    spares: > 0 turns on the adaptive cache: each layer's slot run gets that
      many free slots beyond its residents (by default the hot set less its
      `spares` coldest, so the run keeps the hot budget), every expert has a host record
      (any of them can be evicted and gathered again), and the cache's
      policy keeps that many spares per layer.
    """
    L = wl.layers if layers is None else layers
    E, H, I, k = wl.E, wl.H, wl.I, wl.k
    T_max = T_max or wl.T
    dev = torch.device("cuda")
    rb = gen.record_bytes(H, I, wl.fmt)
    s = torch.cuda.current_stream() if stream is None else stream
    sp = s.cuda_stream

    bias_host, ranks = [], []
    for l in range(L):
        if wl.zipf_alpha > 0:
            b, r = gen.zipf_bias(wl.seed, l, E, wl.zipf_alpha)
        else:
            b, r = None, np.arange(1, E + 1, dtype=np.int32)
        bias_host.append(b)
        ranks.append(r)
    rec_layer = [0 if alias_host_records else l for l in range(L)]
    if resident is None:
        # under the adaptive policy the spares come out of the hot budget
        resident = [_hot_set(wl, l, ranks[l], saliency_order, drop=spares) for l in range(L)]
    else:
        resident = [sorted(int(e) for e in r) for r in resident]
    n_res = [len(r) for r in resident]
    layer_slots = np.concatenate([[0], np.cumsum([n + spares for n in n_res])]).astype(np.int32)
    n_cache = int(layer_slots[-1])
    miss_max = E if spares > 0 else max(E - n for n in n_res)
    # experts with a host record in layer l: the non-resident ones, or all of
    # them under the adaptive policy
    hosted = [list(range(E)) if spares > 0 else [e for e in range(E) if e not in set(resident[l])]
              for l in range(L)]
    if n_stage is None:
        n_stage = min(miss_max, T_max * k) if miss_max > 0 else 0

    # host arena for non-resident records
    host_arena, host_index = None, None
    if miss_max > 0:
        host_index = np.full((L, E), -1, np.int64)
        if alias_host_records:
            ids = sorted(set(e for l in range(L) for e in hosted[l]))
            pos = {e: i for i, e in enumerate(ids)}
            for l in range(L):
                for e in hosted[l]:
                    host_index[l, e] = pos[e]
            host_arena = HostArena(len(ids), rb)
            fill_list = [(0, e, pos[e]) for e in ids]
        else:
            fill_list = []
            for l in range(L):
                for e in hosted[l]:
                    host_index[l, e] = len(fill_list)
                    fill_list.append((l, e, len(fill_list)))
            host_arena = HostArena(len(fill_list), rb)
        # generate on the device in batches and copy down into the arena
        batch = 16
        buf = torch.empty((batch, rb), dtype=torch.uint8, device=dev)
        for i0 in range(0, len(fill_list), batch):
            chunk = fill_list[i0:i0 + batch]
            for j, (l, e, _) in enumerate(chunk):
                gen.dev_expert_record(wl.seed, rec_layer[l], e, H, I, buf[j].data_ptr(), sp,
                                      fmt=wl.fmt)
            s.synchronize()
            for j, (l, e, idx) in enumerate(chunk):
                torch.from_numpy(host_arena.array[idx]).copy_(buf[j].cpu())
        del buf
        host_arena.register()

    if slot_alias > 0:
        # profiling only: every layer's experts share slot_alias records (expert
        # e reads slot e mod slot_alias); the outputs are not those of the workload
        assert L == 1 and miss_max == 0
        n_cache = slot_alias
        layer_slots = np.array([0, slot_alias], np.int32)
    cache = ExpertCache(L, E, H, I, n_cache, n_stage, layer_slots=layer_slots,
                        host_arena=host_arena, host_index=host_index, fmt=wl.fmt)
    for l in range(L):
        for j, e in enumerate(resident[l]):
            slot = int(layer_slots[l]) + (j % slot_alias if slot_alias > 0 else j)
            if slot_alias == 0 or j < slot_alias:
                gen.dev_expert_record(wl.seed, rec_layer[l], e, H, I, cache.slot_ptr(slot), sp,
                                      fmt=wl.fmt)
            cache.set_resident(l, e, slot, s)
    if spares > 0:
        cache.set_policy(spares)

    w_router, gscale, gscale_host, bias, shared, mls = [], [], [], [], [], []
    pmin = prefill_min_tokens if prefill_min_tokens is not None else (
        max(T_max, 1) if wl.prefill else 0)
    for l in range(L):
        wr = torch.empty((E, H), dtype=torch.float32, device=dev)
        gen.dev_router_f32(wl.seed, l, E, H, wr.data_ptr(), sp)
        gh = gen.global_scales(wl.seed, l, E)
        g = torch.from_numpy(gh).to(dev)
        b = torch.from_numpy(bias_host[l]).to(dev) if bias_host[l] is not None else None
        sh = None
        if wl.Is > 0:
            sg = torch.empty((wl.Is, H), dtype=torch.bfloat16, device=dev)
            su = torch.empty((wl.Is, H), dtype=torch.bfloat16, device=dev)
            sd = torch.empty((H, wl.Is), dtype=torch.bfloat16, device=dev)
            gen.dev_shared_bf16(wl.seed, l, wl.Is, H, sg.data_ptr(), su.data_ptr(), sd.data_ptr(), sp)
            sh = (sg, su, sd)
        w_router.append(wr)
        gscale.append(g)
        gscale_host.append(gh)
        bias.append(b)
        shared.append(sh)
        mls.append(MoELayer(cache, l, wr, g, k, bias=b, shared=sh, T_max=T_max,
                            prefill_min_tokens=pmin,
                            prefill_group=wl.group if prefill_group is None else prefill_group,
                            skip_tau=skip_tau))
    s.synchronize()
    return DeviceWorkload(wl, L, cache, mls, w_router, gscale, gscale_host, bias, bias_host,
                          shared, resident, host_arena, record_layer=rec_layer)
