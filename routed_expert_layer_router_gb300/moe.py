"""Thin ctypes binding of libmoe.so (include/moe.h): the same call names,
argument marshalling only.  Every step of the layer runs in the library's
CUDA kernels; there is no fallback - if the library is missing or fails to
load, these functions raise.

Tensors are passed as device pointers (``tensor.data_ptr()``); streams as
``torch.cuda.Stream.cuda_stream`` integers (0 = legacy default stream).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA = 0, 1, 2, 3
MOE_ERR_OOM, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE = 4, 5, 6
MOE_MODE_DECODE, MOE_MODE_PREFILL = 0, 1
MOE_STAGE_GATE_UP, MOE_STAGE_DOWN, MOE_STAGE_ALL = 1, 2, 3

vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t


class MoeError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} -> {status_string(status)} ({status})")
        self.status = status


class moe_route_args(ctypes.Structure):
    _fields_ = [("x", vp), ("w_router", vp), ("bias", vp), ("T", i32), ("H", i32), ("E", i32),
                ("k", i32), ("ids", vp), ("w", vp), ("p_sel", vp), ("logits", vp),
                ("workspace", vp), ("workspace_bytes", sz), ("status", vp),
                ("w_split", vp), ("w_split_bytes", sz)]


class expcache_desc(ctypes.Structure):
    _fields_ = [("L", i32), ("E", i32), ("H", i32), ("I", i32), ("n_cache_slots", i32),
                ("layer_slots", vp), ("n_stage", i32), ("host_arena", vp),
                ("host_arena_records", u64), ("host_index", vp), ("format", i32)]


class moe_ffn_args(ctypes.Structure):
    _fields_ = [("mode", i32), ("stages", i32), ("T", i32), ("H", i32), ("I", i32), ("E", i32),
                ("k", i32), ("x", vp), ("cache", vp), ("gscale", vp), ("src_slot", vp),
                ("act_list", vp), ("n_act", vp), ("offsets", vp), ("pad_offsets", vp),
                ("perm", vp), ("inv", vp), ("w", vp), ("group", i32), ("n_stage", i32),
                ("prefill_group", i32), ("Is", i32),
                ("s_gate", vp), ("s_up", vp), ("s_down", vp), ("o_route", vp), ("y_acc", vp),
                ("o_shared", vp), ("workspace", vp), ("workspace_bytes", sz), ("status", vp)]


class moe_combine_args(ctypes.Structure):
    _fields_ = [("T", i32), ("H", i32), ("k", i32), ("y_acc", vp), ("o_route", vp),
                ("inv", vp), ("o_shared", vp), ("y", vp)]


class moe_layer_desc(ctypes.Structure):
    _fields_ = [("H", i32), ("I", i32), ("E", i32), ("k", i32), ("Is", i32),
                ("w_router", vp), ("bias", vp), ("gscale", vp), ("s_gate", vp), ("s_up", vp),
                ("s_down", vp), ("cache", vp), ("layer", i32), ("T_max", i32),
                ("prefill_min_tokens", i32), ("prefill_group", i32),
                ("skip_tau", ctypes.c_float)]


# every function declared in include/moe.h: name -> (restype, argtypes)
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [i32]),
    "moe_abi_version": (i32, []),
    "moe_record_bytes": (u64, [i32, i32, i32]),
    "moe_route_workspace_bytes": (sz, [i32, i32]),
    "moe_route_split_bytes": (sz, [i32, i32]),
    "moe_route": (i32, [ctypes.POINTER(moe_route_args), vp]),
    "moe_permute": (i32, [vp, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp, vp]),
    "expcache_create": (i32, [ctypes.POINTER(expcache_desc), ctypes.POINTER(vp)]),
    "expcache_destroy": (i32, [vp]),
    "expcache_slot_ptr": (vp, [vp, i32]),
    "expcache_slot_table": (vp, [vp]),
    "expcache_set_resident": (i32, [vp, i32, i32, i32, vp]),
    "expcache_fill": (i32, [vp, i32, vp, vp, i32, i32, vp, vp, vp]),
    "expcache_lookup": (i32, [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]),
    "expcache_plan_slots": (i32, [vp, i32, i32, i32, i32, vp, vp, vp]),
    "expcache_set_policy": (i32, [vp, i32]),
    "expcache_policy_step": (i32, [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]),
    "expcache_policy_state": (i32, [vp, ctypes.POINTER(i32), vp, vp, vp, vp]),
    "moe_ffn_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32, i32]),
    "moe_expert_ffn": (i32, [ctypes.POINTER(moe_ffn_args), vp]),
    "moe_expert_ffn_noalloc": (i32, [ctypes.POINTER(moe_ffn_args), vp]),
    "moe_nvfp4_quantize": (i32, [vp, i32, i32, i32, vp, vp, vp, vp]),
    "moe_combine": (i32, [ctypes.POINTER(moe_combine_args), vp]),
    "moe_layer_create": (i32, [ctypes.POINTER(moe_layer_desc), ctypes.POINTER(vp)]),
    "moe_layer_destroy": (i32, [vp]),
    "moe_layer_forward": (i32, [vp, vp, i32, vp, vp]),
    "moe_layer_debug_ptrs": (i32, [vp, vp, vp, vp, vp, vp, vp]),
    "moe_layer_debug_prefill": (i32, [vp, vp, vp, vp]),
    "moe_layer_set_timing": (i32, [vp, vp, i32]),
    "moe_read_device_status": (i32, [vp, vp, ctypes.POINTER(ctypes.c_int32)]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ck(call: str, st: int) -> None:
    if st != MOE_OK:
        raise MoeError(call, st)


def status_string(st: int) -> str:
    return lib().moe_status_string(st).decode()


def moe_abi_version() -> int:
    return lib().moe_abi_version()


MOE_FMT_NVFP4, MOE_FMT_MXFP4 = 0, 1


def moe_record_bytes(H: int, I: int, fmt: int = MOE_FMT_NVFP4) -> int:
    return int(lib().moe_record_bytes(H, I, fmt))


def moe_route_workspace_bytes(T: int, E: int) -> int:
    return int(lib().moe_route_workspace_bytes(T, E))


def moe_route_split_bytes(E: int, H: int) -> int:
    return int(lib().moe_route_split_bytes(E, H))


def moe_route(args: moe_route_args, stream: int = 0) -> None:
    _ck("moe_route", lib().moe_route(ctypes.byref(args), stream))


def moe_permute(ids, T, k, E, counts, offsets, perm, inv, pad_offsets=0, pad_align=128,
                status=0, stream: int = 0) -> None:
    _ck("moe_permute", lib().moe_permute(ids, T, k, E, counts, offsets, perm, inv,
                                         pad_offsets or None, pad_align, status or None, stream))


def expcache_create(desc: expcache_desc) -> int:
    h = vp()
    _ck("expcache_create", lib().expcache_create(ctypes.byref(desc), ctypes.byref(h)))
    return h.value


def expcache_destroy(cache: int) -> None:
    _ck("expcache_destroy", lib().expcache_destroy(cache))


def expcache_slot_ptr(cache: int, slot: int) -> int:
    p = lib().expcache_slot_ptr(cache, slot)
    if not p:
        raise MoeError("expcache_slot_ptr", MOE_ERR_INVALID_ARG)
    return p


def expcache_slot_table(cache: int) -> int:
    return lib().expcache_slot_table(cache)


def expcache_set_resident(cache, layer, expert, slot, stream: int = 0) -> None:
    _ck("expcache_set_resident", lib().expcache_set_resident(cache, layer, expert, slot, stream))


def expcache_fill(cache, layer, d_expert_ids, d_n, first, max_count, d_dst_slots=0, status=0,
                  stream: int = 0) -> None:
    _ck("expcache_fill", lib().expcache_fill(cache, layer, d_expert_ids, d_n, first, max_count,
                                             d_dst_slots or None, status or None, stream))


def expcache_lookup(cache, layer, counts, src_slot, act_list, n_act, miss_ids, n_miss, status=0,
                    stream: int = 0) -> None:
    _ck("expcache_lookup", lib().expcache_lookup(cache, layer, counts, src_slot, act_list, n_act,
                                                 miss_ids, n_miss, status or None, stream))


def expcache_plan_slots(d_counts, L, E, total_slots, floor, d_layer_slots, d_order,
                        stream: int = 0) -> None:
    _ck("expcache_plan_slots", lib().expcache_plan_slots(d_counts, L, E, total_slots, floor,
                                                         d_layer_slots, d_order, stream))


def expcache_set_policy(cache, spares_per_layer: int) -> None:
    _ck("expcache_set_policy", lib().expcache_set_policy(cache, spares_per_layer))


def expcache_policy_step(cache, layer, counts, src_slot, n_act, miss_ids, n_miss, miss_dst,
                         meta=0, stream: int = 0) -> None:
    _ck("expcache_policy_step", lib().expcache_policy_step(cache, layer, counts, src_slot, n_act,
                                                           miss_ids, n_miss, miss_dst,
                                                           meta or None, stream))


def expcache_policy_state(cache) -> dict:
    """Device pointers of the adaptive policy's state (see moe.h)."""
    spares = i32()
    outs = [vp() for _ in range(4)]
    _ck("expcache_policy_state", lib().expcache_policy_state(
        cache, ctypes.byref(spares), *[ctypes.byref(o) for o in outs]))
    return dict(zip(["cnt", "last", "stamp", "freeslot"], [o.value for o in outs]),
                spares=spares.value)


def moe_ffn_workspace_bytes(mode, T, H, I, E, k, Is) -> int:
    return int(lib().moe_ffn_workspace_bytes(mode, T, H, I, E, k, Is))


def moe_expert_ffn(args: moe_ffn_args, stream: int = 0) -> None:
    _ck("moe_expert_ffn", lib().moe_expert_ffn(ctypes.byref(args), stream))


MOE_NOALLOC_SCRATCH_BYTES = 8 << 20


def moe_expert_ffn_noalloc(args: moe_ffn_args, stream: int = 0) -> None:
    """Decode expert FFN without caller workspace (for callers that cannot
    allocate device memory): the scratch is a fixed library-owned device
    array of MOE_NOALLOC_SCRATCH_BYTES shared by all calls; calls that overlap
    on the GPU race on it."""
    _ck("moe_expert_ffn_noalloc", lib().moe_expert_ffn_noalloc(ctypes.byref(args), stream))


def moe_nvfp4_quantize(x, dtype, T, K, codes, scales, G, stream: int = 0) -> None:
    """NVFP4 quantisation of T rows of K values (dtype 0 = bf16, 1 = fp32) into
    codes [T][K/2], scales in 512-byte atoms and G [T] (device pointers)."""
    _ck("moe_nvfp4_quantize", lib().moe_nvfp4_quantize(x, dtype, T, K, codes, scales, G, stream))


def moe_combine(args: moe_combine_args, stream: int = 0) -> None:
    _ck("moe_combine", lib().moe_combine(ctypes.byref(args), stream))


def moe_layer_create(desc: moe_layer_desc) -> int:
    h = vp()
    _ck("moe_layer_create", lib().moe_layer_create(ctypes.byref(desc), ctypes.byref(h)))
    return h.value


def moe_layer_destroy(layer: int) -> None:
    _ck("moe_layer_destroy", lib().moe_layer_destroy(layer))


def moe_layer_forward(layer: int, x: int, T: int, y: int, stream: int = 0) -> None:
    _ck("moe_layer_forward", lib().moe_layer_forward(layer, x, T, y, stream))


def moe_layer_debug_ptrs(layer: int) -> dict:
    outs = [vp() for _ in range(6)]
    _ck("moe_layer_debug_ptrs",
        lib().moe_layer_debug_ptrs(layer, *[ctypes.byref(o) for o in outs]))
    return dict(zip(["ids", "w", "p_sel", "perm", "src_slot", "n_act"], [o.value for o in outs]))


def moe_layer_debug_prefill(layer: int) -> dict:
    outs = [vp() for _ in range(3)]
    _ck("moe_layer_debug_prefill",
        lib().moe_layer_debug_prefill(layer, *[ctypes.byref(o) for o in outs]))
    return dict(zip(["h_rows", "offsets", "pad_offsets"], [o.value for o in outs]))


def moe_layer_set_timing(layer: int, events: list) -> None:
    """events: cudaEvent_t handles (ints); [] clears the hook."""
    arr = (vp * max(1, len(events)))(*events)
    _ck("moe_layer_set_timing", lib().moe_layer_set_timing(layer, arr, len(events)))


def moe_read_device_status(layer: int, stream: int = 0) -> int:
    v = ctypes.c_int32(0)
    _ck("moe_read_device_status", lib().moe_read_device_status(layer, stream, ctypes.byref(v)))
    return v.value
