"""Helpers for the GPU parity tests: seeded token draws with near-tie
rejection (decided by the oracle's fp64 router), oracle forward passes for a
device workload, and the comparison rules."""
from __future__ import annotations

import numpy as np
import torch

import gen
import oracle
from tests.helpers import TOL, PROB_RTOL, bf16_to_f64

GAP_MIN = 1e-4  # adjacent logit gaps among the k+1 best must be at least this


def draw_tokens(wl: gen.Workload, layer: int, T: int, Wr: np.ndarray, bias, draw0: int = 0,
                batch: int = 64, reject: bool = True):
    """T bf16 tokens from consecutive draws of (seed, layer), skipping draws
    whose oracle logits have an adjacent gap < GAP_MIN among the k+1 largest.
    Returns (x [T,H] uint16, draw indices)."""
    xs, idx = [], []
    d = draw0
    while len(idx) < T:
        n = min(batch, max(T - len(idx), 1) * 2)
        cand = gen.x_bf16(wl.seed, layer, d, n, wl.H)
        if reject:
            *_, gap = oracle.route(cand, Wr, bias, wl.k)
            ok = gap >= GAP_MIN
        else:
            ok = np.ones(n, bool)
        for i in range(n):
            if ok[i] and len(idx) < T:
                xs.append(cand[i])
                idx.append(d + i)
        d += n
    return np.stack(xs), idx


def host_inputs(dw, layer: int):
    """Host copies of a device workload layer's router, bias and shared weights."""
    wl = dw.wl
    Wr = gen.router_f32(wl.seed, layer, wl.E, wl.H)
    sh = gen.shared_bf16(wl.seed, layer, wl.Is, wl.H) if wl.Is > 0 else None
    return Wr, dw.bias_host[layer], sh


def oracle_layer(dw, layer: int, x: np.ndarray, mode: int = 0, record_cache=None,
                 return_bound: bool = False):
    """Oracle forward of layer `layer` on tokens x: generates (on the host)
    the records of the experts the oracle's router selects."""
    wl = dw.wl
    Wr, bias, sh = host_inputs(dw, layer)
    ids, w, p, _, _ = oracle.route(x, Wr, bias, wl.k)
    need = sorted(set(ids.ravel().tolist()))
    cache = record_cache if record_cache is not None else {}
    rl = dw.record_layer[layer] if dw.record_layer else layer
    missing = [e for e in need if (rl, e) not in cache]
    if missing:
        recs = gen.expert_records(wl.seed, rl, missing, wl.H, wl.I)
        for e, r in zip(missing, recs):
            cache[(rl, e)] = r
    records = {e: cache[(rl, e)] for e in need}
    y, ids2, w2, p2, bound = oracle.layer_forward(x, wl.H, wl.I, wl.E, wl.k, Wr, bias, records,
                                                  dw.gscale_host[layer], shared_w=sh, mode=mode,
                                                  return_bound=True)
    if return_bound:
        return y, ids2, w2, p2, bound
    return y, ids2, w2, p2


def to_dev_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x.astype(np.int16)).view(torch.bfloat16).cuda()


def y_to_f64(y: torch.Tensor) -> np.ndarray:
    return bf16_to_f64(y.view(torch.int16).cpu().numpy().view(np.uint16))


def check_outputs(y_gpu: np.ndarray, y_ref: np.ndarray, tol: float = TOL, bound=None):
    """max |y_gpu - y_ref| <= tol * rms(y_ref), element by element widened by
    `bound` (the oracle's rounding-boundary slack of the prefill numerics:
    where the two sides' intermediate values straddle a rounding boundary of
    the NVFP4 or bf16 re-quantisation, either neighbour is a correct result)."""
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    assert rms > 0
    excess = np.abs(y_gpu - y_ref) - (0.0 if bound is None else bound)
    err = float(excess.max())
    assert err <= tol * rms, f"max|dy| = {err:.3e} > {tol} * rms {rms:.3e} (ratio {err / rms:.3e})"
    return err / rms


def check_permutation(dbg: dict, ids_ref):
    """The layer's permutation and lookup against their definitions: perm is
    the stable sort of the routes by expert; every selected expert is active
    (hits counted among them) and has a cache or staging slot."""
    flat = np.asarray(ids_ref).ravel()
    perm = dbg["perm"].cpu().numpy()
    assert np.array_equal(perm, np.argsort(flat, kind="stable")), (perm, flat)
    n_act = dbg["n_act"].cpu().numpy()
    assert n_act[0] == len(np.unique(flat)) and 0 <= n_act[1] <= n_act[0], n_act
    src = dbg["src_slot"].cpu().numpy()
    assert np.all(src[np.unique(flat)] >= 0), src


def check_router(dbg: dict, ids_ref, w_ref, p_ref):
    ids = dbg["ids"].cpu().numpy()
    assert np.array_equal(ids, ids_ref), f"ids differ:\n{ids}\nvs\n{ids_ref}"
    w = dbg["w"].cpu().numpy().astype(np.float64)
    p = dbg["p_sel"].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(w - w_ref) <= PROB_RTOL * np.abs(w_ref)), np.abs(w / w_ref - 1).max()
    assert np.all(np.abs(p - p_ref) <= PROB_RTOL * np.abs(p_ref)), np.abs(p / p_ref - 1).max()
