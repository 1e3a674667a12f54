"""CPU oracle of the routed MoE layer (plain C, fp64) - TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library under
``routed_expert_layer_router_gb300/`` never does; the two share no code.

This module compiles ``oracle.c`` with gcc and exposes its functions through
ctypes.  Every computation lives in ``oracle.c``; the helpers below only
marshal numpy arrays and, for large layers, generate the expert records a
forward pass needs (through the seeded generator in ``gen``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None
openmp = False


def build(verbose: bool = False) -> None:
    """Compile oracle.c (with OpenMP when the compiler has it)."""
    base = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o", _SO,
            os.path.join(_HERE, "oracle.c"), "-lm"]
    p = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if p.returncode != 0:
        p = subprocess.run(base, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + p.stdout + p.stderr)
    if verbose:
        print(p.stdout + p.stderr)


def lib():
    global _lib, openmp
    if _lib is None:
        if not os.path.exists(_SO):
            build()
        L = ctypes.CDLL(_SO)
        vp, i32, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.oracle_e2m1.argtypes = [ctypes.c_uint]
        L.oracle_e2m1.restype = d
        L.oracle_e4m3.argtypes = [ctypes.c_uint]
        L.oracle_e4m3.restype = d
        L.oracle_bf16.argtypes = [ctypes.c_uint16]
        L.oracle_bf16.restype = d
        L.oracle_weight.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp]
        L.oracle_weight.restype = d
        L.oracle_dequant_matrix.argtypes = [vp, i32, i32, i32, i32, vp, vp]
        L.oracle_e8m0.argtypes = [ctypes.c_uint]
        L.oracle_e8m0.restype = d
        L.oracle_mxfp4_quant.argtypes = [vp, i32, vp, vp]
        L.oracle_route.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]
        L.oracle_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
        L.oracle_permute.restype = i32
        L.oracle_e4m3_rne.argtypes = [ctypes.c_float]
        L.oracle_e4m3_rne.restype = ctypes.c_uint
        L.oracle_e2m1_rne_sat.argtypes = [ctypes.c_float]
        L.oracle_e2m1_rne_sat.restype = ctypes.c_uint
        L.oracle_nvfp4_quant.argtypes = [vp, i32, vp, vp, vp]
        L.oracle_expert.argtypes = [vp, i32, i32, i32, vp, vp, i32, vp]
        L.oracle_shared.argtypes = [vp, vp, vp, i32, i32, vp, i32, vp]
        L.oracle_renorm_skip.argtypes = [vp, vp, i32, i32, vp, d, vp, vp]
        L.oracle_layer_forward.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                           vp, vp, vp, i32, vp, d, vp, vp, vp, vp, vp]
        L.oracle_layer_forward.restype = i32
        L.oracle_set_defect.argtypes = [i32]
        L.oracle_quant_flip_delta.argtypes = [vp, i32, i32, vp]
        L.oracle_bf16_flip_delta.argtypes = [vp, i32, vp]
        L.oracle_set_flip_margins.argtypes = [d, d, d]
        L.oracle_slot_budget.argtypes = [i32, i32, vp, i32, i32, vp, vp]
        L.oracle_slot_budget.restype = i32
        L.oracle_expert_h.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.oracle_prefill_near_boundary.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp]
        L.oracle_cache_policy_step.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                               vp, vp, vp]
        L.oracle_cache_policy_step.restype = i32
        _lib = L
        try:
            openmp = "omp_get_num_threads" in open(_SO, "rb").read().decode("latin1")
        except OSError:
            openmp = False
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "need a C-contiguous array"
    return a.ctypes.data


DEFECTS = {"nibble_swap": 1, "scale_ue8m0": 2, "block_off_by_one": 3, "tie_high_id": 4,
           "scaling_2_5": 5}


class defect:
    """Context manager planting one named defect in the oracle (negative controls)."""

    def __init__(self, name: str):
        self.code = DEFECTS[name]

    def __enter__(self):
        lib().oracle_set_defect(self.code)
        return self

    def __exit__(self, *exc):
        lib().oracle_set_defect(0)
        return False


def e2m1(code: int) -> float:
    return lib().oracle_e2m1(code)


def e4m3(byte: int) -> float:
    return lib().oracle_e4m3(byte)


def bf16(h: int) -> float:
    return lib().oracle_bf16(h)


# record formats (gen.NVFP4, gen.MXFP4)
NVFP4, MXFP4 = 0, 1


def weight(rec, H, I, m, r, c, g3, fmt=NVFP4) -> float:
    return lib().oracle_weight(_p(rec), H, I, fmt, m, r, c,
                               _p(np.ascontiguousarray(g3, np.float32)))


def dequant_matrix(rec, H, I, m, g3, fmt=NVFP4) -> np.ndarray:
    R, K = (H, I) if m == 2 else (I, H)
    out = np.empty((R, K), np.float64)
    lib().oracle_dequant_matrix(_p(rec), H, I, fmt, m, _p(np.ascontiguousarray(g3, np.float32)),
                                _p(out))
    return out


def route(x, Wr, bias, k):
    """Returns ids [T,k] i32, w [T,k], p_sel [T,k], logits [T,E], gap [T] (fp64)."""
    x = np.ascontiguousarray(x, np.uint16)
    Wr = np.ascontiguousarray(Wr, np.float32)
    T, H = x.shape
    E = Wr.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, np.float32)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    p = np.empty((T, k), np.float64)
    logits = np.empty((T, E), np.float64)
    gap = np.empty(T, np.float64)
    lib().oracle_route(_p(x), _p(Wr), _p(b), T, H, E, k, _p(ids), _p(w), _p(p), _p(logits), _p(gap))
    return ids, w, p, logits, gap


def permute(ids, E):
    ids = np.ascontiguousarray(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    if lib().oracle_permute(_p(ids), T, k, E, _p(counts), _p(offsets), _p(perm), _p(inv)):
        raise ValueError("expert id out of range")
    return counts, offsets, perm, inv


def e4m3_rne(t: float) -> int:
    return lib().oracle_e4m3_rne(t)


def e2m1_rne_sat(q: float) -> int:
    return lib().oracle_e2m1_rne_sat(q)


def nvfp4_quant(v):
    v = np.ascontiguousarray(v, np.float32)
    n = v.shape[0]
    codes = np.empty(n // 2, np.uint8)
    scales = np.empty(n // 16, np.uint8)
    G = np.empty(1, np.float32)
    lib().oracle_nvfp4_quant(_p(v), n, _p(codes), _p(scales), _p(G))
    return codes, scales, float(G[0])


def e8m0(b: int) -> float:
    return lib().oracle_e8m0(b)


def mxfp4_quant(v):
    """MXFP4 codes [n/2] and E8M0 scales [n/32] of an fp32 row (OCP MX rule)."""
    v = np.ascontiguousarray(v, np.float32)
    n = v.shape[0]
    codes = np.empty(n // 2, np.uint8)
    scales = np.empty(n // 32, np.uint8)
    lib().oracle_mxfp4_quant(_p(v), n, _p(codes), _p(scales))
    return codes, scales


def quant_flip_delta(v, fmt=NVFP4):
    """Per-element rounding-boundary slack of the NVFP4 (or MXFP4)
    quantisation of v."""
    v = np.ascontiguousarray(v, np.float32)
    out = np.empty(v.shape[0], np.float64)
    lib().oracle_quant_flip_delta(_p(v), v.shape[0], fmt, _p(out))
    return out


# margins of the rounding-boundary slack (oracle.c, orc_quant_flip_delta):
# E2M1 code units, relative E4M3 scale argument, relative bf16 value
FLIP_Q, FLIP_T, FLIP_BF16 = 2e-5, 1e-5, 2e-6


def set_flip_margins(q=FLIP_Q, t=FLIP_T, bf16=FLIP_BF16):
    lib().oracle_set_flip_margins(float(q), float(t), float(bf16))


def expert_h(rec, H, I, g3, x, fmt=NVFP4):
    """h = silu(Wg x) * (Wu x) [I] in fp64 for one routed expert (x fp64 [H])."""
    x = np.ascontiguousarray(x, np.float64)
    h = np.empty(I, np.float64)
    lib().oracle_expert_h(_p(rec), H, I, fmt, _p(np.ascontiguousarray(g3, np.float32)), _p(x),
                          _p(h))
    return h


def prefill_near_boundary(x, H, I, k, ids, records, g, fmt=NVFP4):
    """Per token of x [T,H] (bf16) with routes ids [T,k]: the number of
    elements of its routes' h that lie within the margins of an NVFP4
    rounding boundary (where another implementation may take the
    neighbouring code).  records: expert id -> record (dict or sequence)."""
    x = np.ascontiguousarray(x, np.uint16)
    ids = np.ascontiguousarray(ids, np.int32)
    T = x.shape[0]
    E = int(ids.max()) + 1 if ids.size else 1
    keep = []
    ptrs = (ctypes.c_void_p * E)()
    for e in set(ids.ravel().tolist()):
        r = np.ascontiguousarray(records[e])
        keep.append(r)
        ptrs[e] = r.ctypes.data
    count = np.empty(T, np.int32)
    lib().oracle_prefill_near_boundary(_p(x), T, H, I, fmt, k, _p(ids), ptrs,
                                       _p(np.ascontiguousarray(g, np.float32)), _p(count))
    return count


def bf16_flip_delta(v):
    """Per-element bf16 rounding-boundary slack of fp64 values v: one bf16
    step where v lies within relative FLIP_BF16 of a bf16 rounding midpoint."""
    v = np.ascontiguousarray(v, np.float64)
    out = np.empty(v.shape[0], np.float64)
    lib().oracle_bf16_flip_delta(_p(v), v.shape[0], _p(out))
    return out


def expert(rec, H, I, g3, x, act_quant=False, fmt=NVFP4):
    x = np.ascontiguousarray(x, np.float64)
    o = np.empty(H, np.float64)
    lib().oracle_expert(_p(rec), H, I, fmt, _p(np.ascontiguousarray(g3, np.float32)), _p(x),
                        int(act_quant), _p(o))
    return o


def shared(wg, wu, wd, x, round_h_bf16=False):
    x = np.ascontiguousarray(x, np.float64)
    Is, H = wg.shape
    o = np.empty(H, np.float64)
    lib().oracle_shared(_p(wg), _p(wu), _p(wd), H, Is, _p(x), int(round_h_bf16), _p(o))
    return o


def layer_forward(x, H, I, E, k, Wr, bias, records, g, shared_w=None, mode=0,
                  return_bound=False, resident=None, tau=0.0, fmt=NVFP4):
    """y [T,H] fp64 plus ids, w, p_sel (and, with return_bound, the
    rounding-boundary slack [T,H] of the prefill numerics, zero in mode 0).
    ``records`` maps expert id -> uint8 record array (a dict or a sequence
    with None for absent experts).  resident [E] (bool) and tau: the
    renorm-skip of low-weight misses (None: exact)."""
    x = np.ascontiguousarray(x, np.uint16)
    T = x.shape[0]
    keep = []
    ptrs = (ctypes.c_void_p * E)()
    for e in range(E):
        r = records.get(e) if isinstance(records, dict) else records[e]
        if r is not None:
            r = np.ascontiguousarray(r)
            keep.append(r)
            ptrs[e] = r.ctypes.data
    y = np.empty((T, H), np.float64)
    bound = np.zeros((T, H), np.float64)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    p = np.empty((T, k), np.float64)
    Is = 0 if shared_w is None else shared_w[0].shape[0]
    sg, su, sd = (None, None, None) if shared_w is None else shared_w
    rc = lib().oracle_layer_forward(
        _p(x), T, H, I, fmt, E, k, Is, _p(np.ascontiguousarray(Wr, np.float32)),
        _p(None if bias is None else np.ascontiguousarray(bias, np.float32)), ptrs,
        _p(np.ascontiguousarray(g, np.float32)), _p(sg), _p(su), _p(sd), mode,
        _p(None if resident is None else np.ascontiguousarray(resident, np.uint8)), float(tau),
        _p(y), _p(ids), _p(w), _p(p), _p(bound))
    if rc:
        raise ValueError("oracle_layer_forward: a selected expert has no record")
    return (y, ids, w, p, bound) if return_bound else (y, ids, w, p)


class CachePolicy:
    """The adaptive cache's state for all layers, stepped by the oracle's
    policy (oracle_cache_policy_step): table [L,E] (slot or -1), cnt and last
    [L,E], stamp [L], events, free [n_cache]."""

    def __init__(self, L, E, n_cache, layer_slots, K, table):
        self.L, self.E, self.K = L, E, K
        self.layer_slots = [int(v) for v in layer_slots]
        self.table = np.ascontiguousarray(table, dtype=np.int32).reshape(L, E).copy()
        self.cnt = np.zeros((L, E), np.uint32)
        self.last = np.zeros((L, E), np.uint32)
        self.stamp = np.zeros(L, np.uint32)
        self.events = np.zeros(1, np.uint32)
        self.free = np.zeros(n_cache, np.uint8)
        for l in range(L):
            used = set(int(s) for s in self.table[l] if s >= 0)
            for s in range(self.layer_slots[l], self.layer_slots[l + 1]):
                if s not in used:
                    self.free[s] = 1

    def step(self, layer, counts):
        """One forward of `layer` with routes counts[E]; returns the misses'
        promoted slots (-1 = staged) in ascending expert id."""
        counts = np.ascontiguousarray(counts, dtype=np.int32)
        prom = np.zeros(self.E, np.int32)
        n = lib().oracle_cache_policy_step(
            self.L, self.E, layer, self.layer_slots[layer], self.layer_slots[layer + 1], self.K,
            _p(self.table), _p(self.cnt), _p(self.last), _p(self.stamp), _p(self.events),
            _p(self.free), _p(counts), _p(prom))
        return prom[:n].copy()


def renorm_skip(ids, w, resident, tau):
    """The renorm-skip step alone: (w_eff, keep) for routes ids [T,k] with
    weights w [T,k] (fp64), resident [E] bool."""
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    T, k = ids.shape
    w_eff = np.empty((T, k), np.float64)
    keep = np.empty((T, k), np.uint8)
    lib().oracle_renorm_skip(_p(ids), _p(w), T, k,
                             _p(np.ascontiguousarray(resident, np.uint8)), float(tau),
                             _p(w_eff), _p(keep))
    return w_eff, keep.astype(bool)


def slot_budget(counts, total, floor):
    """Greedy per-layer slot budget from per-layer route counts [L,E]:
    (layer_slots [L+1], order [L,E]) - layer l owns slots [layer_slots[l],
    layer_slots[l+1]) and caches order[l][:n_l].  None when the floor does
    not fit."""
    counts = np.ascontiguousarray(counts, np.uint32)
    L, E = counts.shape
    ls = np.empty(L + 1, np.int32)
    order = np.empty((L, E), np.int32)
    if lib().oracle_slot_budget(L, E, _p(counts), int(total), int(floor), _p(ls), _p(order)):
        return None
    return ls, order
