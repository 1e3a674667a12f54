"""Seeded synthetic inputs for the routed MoE layer (shared by the oracle side
and the GPU side; holds none of the layer's arithmetic).

The definitions live in ``gen_core.h``; ``gen.c`` implements them on the host
and ``gen_cuda.cu`` on the device, bit for bit alike.  This module loads both
shared libraries (built by :func:`build`) and describes the five workloads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libgen_host.so")
_CUDA_SO = os.path.join(_HERE, "libgen_cuda.so")


def build(cuda: bool = True, verbose: bool = False) -> None:
    """Compile the host generator (gcc) and, if asked, the device one (nvcc)."""
    cmds = [["gcc", "-O3", "-fPIC", "-shared", "-ffp-contract=off", "-o", _HOST_SO,
             os.path.join(_HERE, "gen.c"), "-lpthread", "-lm"]]
    if cuda:
        cmds.append(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                     "-Xcompiler", "-fPIC", "-shared", "-o", _CUDA_SO,
                     os.path.join(_HERE, "gen_cuda.cu")])
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT) for c in cmds]
    for c, p in zip(cmds, procs):
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(c)}\n{out.decode()}")
        if verbose:
            print(out.decode())


GOLDEN = 0x9E3779B97F4A7C15  # splitmix64 increment (the golden-ratio constant)

_host = None
_cuda = None


def _lib_host():
    global _host
    if _host is None:
        if not os.path.exists(_HOST_SO):
            build(cuda=False)
        L = ctypes.CDLL(_HOST_SO)
        u64, i32, i64, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        L.gen_x_bf16.argtypes = [u64, i32, i64, i32, i32, vp]
        L.gen_router_f32.argtypes = [u64, i32, i32, i32, vp]
        L.gen_shared_bf16.argtypes = [u64, i32, i32, i32, vp, vp, vp]
        L.gen_global_scales.argtypes = [u64, i32, i32, vp]
        L.gen_expert_record.argtypes = [u64, i32, i32, i32, i32, i32, vp]
        L.gen_expert_records_mt.argtypes = [u64, i32, vp, i32, i32, i32, i32, vp, i32]
        L.gen_zipf_bias.argtypes = [u64, i32, i32, ctypes.c_double, vp, vp]
        L.gen_expert_prequant_row.argtypes = [u64, i32, i32, i32, i32, i32, i32, vp]
        L.gen_mix64_export.argtypes = [u64]
        L.gen_mix64_export.restype = u64
        L.gen_record_size.argtypes = [i32, i32, i32]
        L.gen_record_size.restype = u64
        _host = L
    return _host


def _lib_cuda():
    global _cuda
    if _cuda is None:
        if not os.path.exists(_CUDA_SO):
            raise RuntimeError("device generator not built (gen.build(cuda=True))")
        L = ctypes.CDLL(_CUDA_SO)
        u64, i32, i64, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        L.gen_dev_expert_record.argtypes = [u64, i32, i32, i32, i32, i32, vp, vp]
        L.gen_dev_x_bf16.argtypes = [u64, i32, i64, i32, i32, vp, vp]
        L.gen_dev_router_f32.argtypes = [u64, i32, i32, i32, vp, vp]
        L.gen_dev_shared_bf16.argtypes = [u64, i32, i32, i32, vp, vp, vp, vp]
        for f in (L.gen_dev_expert_record, L.gen_dev_x_bf16, L.gen_dev_router_f32,
                  L.gen_dev_shared_bf16):
            f.restype = i32
        _cuda = L
    return _cuda


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ------------------------------------------------------------------ host side

# record formats: 0 = NVFP4 (E4M3 scale per 16 values), 1 = MXFP4 (E8M0 per 32)
NVFP4, MXFP4 = 0, 1


def record_bytes(H: int, I: int, fmt: int = NVFP4) -> int:
    return 3 * I * H // 2 + 3 * I * H // (32 if fmt == MXFP4 else 16)


def x_bf16(seed: int, layer: int, draw0: int, T: int, H: int) -> np.ndarray:
    out = np.empty((T, H), np.uint16)
    _lib_host().gen_x_bf16(seed, layer, draw0, T, H, _p(out))
    return out


def router_f32(seed: int, layer: int, E: int, H: int) -> np.ndarray:
    out = np.empty((E, H), np.float32)
    _lib_host().gen_router_f32(seed, layer, E, H, _p(out))
    return out


def shared_bf16(seed: int, layer: int, Is: int, H: int):
    g = np.empty((Is, H), np.uint16)
    u = np.empty((Is, H), np.uint16)
    d = np.empty((H, Is), np.uint16)
    _lib_host().gen_shared_bf16(seed, layer, Is, H, _p(g), _p(u), _p(d))
    return g, u, d


def global_scales(seed: int, layer: int, E: int) -> np.ndarray:
    out = np.empty((E, 3), np.float32)
    _lib_host().gen_global_scales(seed, layer, E, _p(out))
    return out


def expert_records(seed: int, layer: int, experts, H: int, I: int, nthreads: int = 0,
                   fmt: int = NVFP4) -> np.ndarray:
    """Records of the listed experts, [n, record_bytes] uint8 (threaded)."""
    experts = np.ascontiguousarray(np.asarray(experts, np.int32))
    n = len(experts)
    rb = record_bytes(H, I, fmt)
    out = np.empty((n, rb), np.uint8)
    if n == 0:
        return out
    ptrs = (ctypes.c_void_p * n)(*[out.ctypes.data + i * rb for i in range(n)])
    nt = nthreads or min(os.cpu_count() or 1, 64)
    _lib_host().gen_expert_records_mt(seed, layer, _p(experts), n, H, I, fmt, ptrs, nt)
    return out


def expert_prequant_row(seed, layer, expert, H, I, m, r) -> np.ndarray:
    """Integers d of row r of matrix m before quantisation (weight = d * g / 64)."""
    K = I if m == 2 else H
    out = np.empty(K, np.int32)
    _lib_host().gen_expert_prequant_row(seed, layer, expert, H, I, m, r, _p(out))
    return out


def mix64(z: int) -> int:
    return int(_lib_host().gen_mix64_export(z & 0xFFFFFFFFFFFFFFFF))


def zipf_bias(seed: int, layer: int, E: int, alpha: float):
    """Per-layer popularity bias b_e = -alpha ln(rank_e), rank a seeded permutation of 1..E."""
    b = np.empty(E, np.float32)
    rank = np.empty(E, np.int32)
    _lib_host().gen_zipf_bias(seed, layer, E, float(alpha), _p(b), _p(rank))
    return b, rank


# ---------------------------------------------------------------- device side

def dev_expert_record(seed, layer, expert, H, I, dst_ptr: int, stream: int = 0,
                      fmt: int = NVFP4) -> None:
    if _lib_cuda().gen_dev_expert_record(seed, layer, expert, H, I, fmt, dst_ptr, stream):
        raise RuntimeError("gen_dev_expert_record failed")


def dev_x_bf16(seed, layer, draw0, T, H, dst_ptr: int, stream: int = 0) -> None:
    if _lib_cuda().gen_dev_x_bf16(seed, layer, draw0, T, H, dst_ptr, stream):
        raise RuntimeError("gen_dev_x_bf16 failed")


def dev_router_f32(seed, layer, E, H, dst_ptr: int, stream: int = 0) -> None:
    if _lib_cuda().gen_dev_router_f32(seed, layer, E, H, dst_ptr, stream):
        raise RuntimeError("gen_dev_router_f32 failed")


def dev_shared_bf16(seed, layer, Is, H, g_ptr, u_ptr, d_ptr, stream: int = 0) -> None:
    if _lib_cuda().gen_dev_shared_bf16(seed, layer, Is, H, g_ptr, u_ptr, d_ptr, stream):
        raise RuntimeError("gen_dev_shared_bf16 failed")


# ------------------------------------------------------------------ workloads

@dataclass(frozen=True)
class Workload:
    """One synthetic workload: the dimensions and input recipe of a config."""
    name: str
    H: int
    I: int
    E: int
    k: int
    T: int
    layers: int
    Is: int            # shared-expert intermediate size (0 = none)
    seed: int
    zipf_alpha: float = 0.0   # per-layer popularity bias strength (0 = unbiased)
    hot: int = 0              # experts per layer kept in the HBM cache (0 = all)
    hot_rule: str = "all"     # "all" | "zipf" (smallest ranks) | "saliency"
    prefill: bool = False
    group: int = 64           # prefill: experts per staging group
    fmt: int = NVFP4          # routed expert record format
    extra: dict = field(default_factory=dict)


# Zipf strength for the skewed stack: calibrated by gen/calibrate_zipf.py so
# that the hottest 35% of experts take 74% of top-8 picks when logits are
# N(0, (0.05 sqrt(H))^2) per expert, as the unbiased router gives.
ZIPF_ALPHA_STACK = 1.556

WORKLOADS = {
    "tiny": Workload("tiny", H=256, I=128, E=16, k=2, T=4, layers=1, Is=0, seed=0),
    "decode": Workload("decode", H=6144, I=2048, E=288, k=8, T=1, layers=1, Is=2048, seed=1),
    "stack": Workload("stack", H=6144, I=2048, E=288, k=8, T=1, layers=16, Is=2048, seed=2,
                      zipf_alpha=ZIPF_ALPHA_STACK, hot=66, hot_rule="zipf"),
    "prefill": Workload("prefill", H=6144, I=2048, E=288, k=8, T=4096, layers=1, Is=2048,
                        seed=3, prefill=True, group=64),
    "flat": Workload("flat", H=6144, I=2048, E=288, k=8, T=64, layers=8, Is=2048, seed=4,
                     hot=72, hot_rule="saliency"),
}
