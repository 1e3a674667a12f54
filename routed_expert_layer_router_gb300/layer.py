"""Python handles over the C ABI: an expert cache and a layer, holding the
torch / numpy buffers they point into so that those stay alive.  Marshalling
only: every computation runs in libmoe.so."""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import moe


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return int(t)


class _DevView:
    """A raw device pointer seen as a tensor (CUDA array interface, no copy)."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3}


def device_view(ptr: int, shape, dtype=torch.int32) -> torch.Tensor:
    typestr = {torch.int32: "<i4", torch.float32: "<f4", torch.int64: "<i8",
               torch.uint8: "|u1"}[dtype]
    return torch.as_tensor(_DevView(ptr, shape, typestr), device="cuda")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


class HostArena:
    """Pinned, device-mapped host memory for expert records that are not
    resident in HBM.  Page-locked with cudaHostRegister (mapped), so the
    kernels can read it directly; freed (unregistered) on close()."""

    def __init__(self, n_records: int, record_bytes: int):
        self.n_records = n_records
        self.record_bytes = record_bytes
        n = max(n_records, 1) * record_bytes
        self._raw = np.empty(n + 4096, np.uint8)
        off = (-self._raw.ctypes.data) % 4096  # page-aligned records (16-byte loads)
        self.array = self._raw[off:off + n].reshape(max(n_records, 1), record_bytes)
        self._registered = False

    def register(self) -> None:
        if self._registered:
            return
        cudart = torch.cuda.cudart()
        # cudaHostRegisterMapped = 2 | cudaHostRegisterPortable = 1
        err = cudart.cudaHostRegister(self.array.ctypes.data, self.array.nbytes, 3)
        if int(err) != 0:
            raise RuntimeError(f"cudaHostRegister failed ({err}) for {self.array.nbytes} bytes")
        self._registered = True

    @property
    def ptr(self) -> int:
        return self.array.ctypes.data

    def close(self) -> None:
        if self._registered:
            torch.cuda.cudart().cudaHostUnregister(self.array.ctypes.data)
            self._registered = False


class ExpertCache:
    """expcache handle: n_cache_slots HBM cache slots + n_stage staging slots."""

    def __init__(self, L, E, H, I, n_cache_slots, n_stage=0, layer_slots=None,
                 host_arena: HostArena | None = None, host_index=None,
                 fmt: int = moe.MOE_FMT_NVFP4):
        self.L, self.E, self.H, self.I, self.fmt = L, E, H, I, fmt
        self.record_bytes = moe.moe_record_bytes(H, I, fmt)
        self.n_cache_slots, self.n_stage = n_cache_slots, n_stage
        self._layer_slots = None if layer_slots is None else np.ascontiguousarray(layer_slots, np.int32)
        self._host_index = None if host_index is None else np.ascontiguousarray(host_index, np.int64)
        self.host_arena = host_arena
        d = moe.expcache_desc()
        d.L, d.E, d.H, d.I = L, E, H, I
        d.n_cache_slots, d.n_stage = n_cache_slots, n_stage
        d.layer_slots = _ptr(self._layer_slots) or None
        d.host_arena = host_arena.ptr if host_arena is not None else None
        d.host_arena_records = host_arena.n_records if host_arena is not None else 0
        d.host_index = _ptr(self._host_index) or None
        d.format = fmt
        self.handle = moe.expcache_create(d)

    def slot_ptr(self, slot: int) -> int:
        return moe.expcache_slot_ptr(self.handle, slot)

    def set_resident(self, layer: int, expert: int, slot: int, stream=None) -> None:
        moe.expcache_set_resident(self.handle, layer, expert, slot, _stream(stream))

    def set_policy(self, spares_per_layer: int) -> None:
        """Turns on the adaptive policy (expcache_set_policy); synchronous."""
        torch.cuda.synchronize()
        moe.expcache_set_policy(self.handle, spares_per_layer)

    def policy_state(self) -> dict:
        """Copies of the adaptive policy's device state (numpy): cnt, last
        [L][E], stamp [L], events, free [n_cache_slots]."""
        p = moe.expcache_policy_state(self.handle)
        torch.cuda.synchronize()
        L, E, n = self.L, self.E, self.n_cache_slots
        st = device_view(p["stamp"], (L + 1,)).cpu().numpy().view(np.uint32)
        return {"spares": p["spares"],
                "cnt": device_view(p["cnt"], (L, E)).cpu().numpy().view(np.uint32),
                "last": device_view(p["last"], (L, E)).cpu().numpy().view(np.uint32),
                "stamp": st[:L].copy(), "events": int(st[L]),
                "free": device_view(p["freeslot"], (n,)).cpu().numpy().astype(np.uint8)}

    def table(self) -> torch.Tensor:
        """Copy of the device slot table [L][E]."""
        torch.cuda.synchronize()
        return device_view(moe.expcache_slot_table(self.handle), (self.L, self.E)).clone()

    def close(self) -> None:
        if self.handle:
            moe.expcache_destroy(self.handle)
            self.handle = 0


class MoELayer:
    """moe_layer handle for layer `layer` of `cache`."""

    def __init__(self, cache: ExpertCache, layer: int, w_router: torch.Tensor,
                 gscale: torch.Tensor, k: int, bias: torch.Tensor | None = None,
                 shared=None, T_max: int = 1, prefill_min_tokens: int = 0,
                 prefill_group: int = 64, skip_tau: float = 0.0):
        self.cache, self.layer = cache, layer
        self.H, self.I, self.E, self.k = cache.H, cache.I, cache.E, k
        self._keep = [w_router, gscale, bias, shared]
        d = moe.moe_layer_desc()
        d.H, d.I, d.E, d.k = cache.H, cache.I, cache.E, k
        d.Is = 0 if shared is None else shared[0].shape[0]
        self.Is = d.Is
        d.w_router, d.bias, d.gscale = _ptr(w_router), _ptr(bias) or None, _ptr(gscale)
        if shared is not None:
            d.s_gate, d.s_up, d.s_down = (_ptr(s) for s in shared)
        d.cache = cache.handle
        d.layer = layer
        d.T_max = T_max
        d.prefill_min_tokens = prefill_min_tokens
        d.prefill_group = prefill_group
        d.skip_tau = skip_tau
        self.T_max = T_max
        self.handle = moe.moe_layer_create(d)

    def forward(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        moe.moe_layer_forward(self.handle, x.data_ptr(), T, y.data_ptr(), _stream(stream))
        return y

    def debug(self, T: int) -> dict:
        """Copies of the last forward's router / permutation / lookup outputs."""
        p = moe.moe_layer_debug_ptrs(self.handle)
        torch.cuda.synchronize()

        def grab(ptr, n, dt):
            return device_view(ptr, (n,), dt).clone()

        k = self.k
        return {"ids": grab(p["ids"], T * k, torch.int32).view(T, k),
                "w": grab(p["w"], T * k, torch.float32).view(T, k),
                "p_sel": grab(p["p_sel"], T * k, torch.float32).view(T, k),
                "perm": grab(p["perm"], T * k, torch.int32),
                "src_slot": grab(p["src_slot"], self.E, torch.int32),
                "n_act": grab(p["n_act"], 2, torch.int32)}

    def debug_prefill(self, T: int) -> dict:
        """After a forward on the PREFILL path: h of every route before its
        NVFP4 quantisation, [T*k, I] fp32 in the permutation's order (row p is
        the route at expert-sorted position p), plus offsets [E+1]."""
        p = moe.moe_layer_debug_prefill(self.handle)
        torch.cuda.synchronize()
        E = self.E
        off = device_view(p["offsets"], (E + 1,), torch.int32).clone()
        pad = device_view(p["pad_offsets"], (E + 1,), torch.int32).clone()
        rows = int(pad[-1].item())
        h = device_view(p["h_rows"], (rows, self.I), torch.float32)
        # padded row of sorted position q of expert e: pad[e] + q - off[e]
        e_of = torch.repeat_interleave(torch.arange(E, device=off.device), (off[1:] - off[:-1]).long())
        q = torch.arange(int(off[-1].item()), device=off.device)
        idx = (pad[:-1].long()[e_of] + q - off[:-1].long()[e_of])
        return {"h": h[idx].clone(), "offsets": off}

    def read_status(self, stream=None) -> int:
        return moe.moe_read_device_status(self.handle, _stream(stream))

    def close(self) -> None:
        if self.handle:
            moe.moe_layer_destroy(self.handle)
            self.handle = 0
