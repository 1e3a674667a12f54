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


# the rounding-boundary slack may widen the tolerance by at most this
# fraction of it anywhere: the slack can never carry a comparison
SLACK_CAP = 0.25


def check_outputs(y_gpu: np.ndarray, y_ref: np.ndarray, tol: float = TOL, bound=None):
    """max |y_gpu - y_ref| <= tol * rms(y_ref), element by element widened by
    `bound` (the oracle's rounding-boundary slack of the prefill numerics:
    where the two sides' intermediate values straddle a rounding boundary of
    the bf16 re-quantisation, either neighbour is a correct result).  The
    slack itself must stay below SLACK_CAP * tol * rms everywhere.  Returns
    max|dy|/rms."""
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    assert rms > 0
    if bound is not None:
        slack = float(np.max(bound)) / (tol * rms)
        assert slack <= SLACK_CAP, f"rounding-boundary slack {slack:.3f} x tol > {SLACK_CAP}"
    dy = np.abs(y_gpu - y_ref)
    excess = dy - (0.0 if bound is None else bound)
    err = float(excess.max())
    assert err <= tol * rms, f"max|dy| = {err:.3e} > {tol} * rms {rms:.3e} (ratio {err / rms:.3e})"
    return float(dy.max()) / rms


def prefill_clean(dw, layer: int, x: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """Mask of the tokens of x (routes ids, from the oracle's router) whose
    routes' h carries no element within the oracle's margins of an NVFP4
    rounding boundary.  Like the router's near-tie rule, this keeps the
    comparison to tokens whose quantised h codes are decided by a clear
    margin, so that both sides must produce the same codes."""
    wl = dw.wl
    rl = dw.record_layer[layer] if dw.record_layer else layer
    need = sorted(set(np.asarray(ids).ravel().tolist()))
    recs = dict(zip(need, gen.expert_records(wl.seed, rl, need, wl.H, wl.I)))
    return oracle.prefill_near_boundary(x, wl.H, wl.I, wl.k, ids, recs,
                                        dw.gscale_host[layer]) == 0


_E2M1 = None


def nvfp4_dequant(codes, scales, G):
    """Values of an NVFP4-quantised row (oracle.nvfp4_quant layout), fp64."""
    global _E2M1
    if _E2M1 is None:
        _E2M1 = (np.array([oracle.e2m1(c) for c in range(16)]),
                 np.array([oracle.e4m3(b) for b in range(256)]))
    c = np.stack([codes & 15, codes >> 4], 1).ravel()
    return _E2M1[0][c] * np.repeat(_E2M1[1][scales], 16) * G


def check_prefill_h(dw, layer: int, x: np.ndarray, h_gpu: np.ndarray, perm: np.ndarray,
                    tokens) -> float:
    """The prefill gate/up GEMM's fp32 h of every route of `tokens` against the
    oracle's fp64 h of the same expert on the same NVFP4-quantised token, in
    units of the block scale s*G that the oracle's re-quantisation of that h
    gives each element (one E2M1 code step is 0.5 to 2 of these units).  The
    difference must stay within a quarter of the oracle's rounding margin
    FLIP_Q: the tokens the comparisons keep (prefill_clean) are then decided
    by a clear margin on both sides.  Returns the largest difference."""
    wl = dw.wl
    k, H, I = wl.k, wl.H, wl.I
    Wr, bias, _ = host_inputs(dw, layer)
    ids, *_ = oracle.route(x[tokens], Wr, bias, k)
    rl = dw.record_layer[layer] if dw.record_layer else layer
    need = sorted(set(ids.ravel().tolist()))
    recs = dict(zip(need, gen.expert_records(wl.seed, rl, need, H, I)))
    pos = np.empty(perm.size, np.int64)
    pos[perm] = np.arange(perm.size)  # route r -> its expert-sorted position
    worst = 0.0
    for i, t in enumerate(tokens):
        xf = bf16_to_f64(x[t]).astype(np.float32)
        xq = nvfp4_dequant(*oracle.nvfp4_quant(xf))
        for j in range(k):
            e = int(ids[i, j])
            h_ref = oracle.expert_h(recs[e], H, I, dw.gscale_host[layer][e], xq)
            hf = h_ref.astype(np.float32)
            _, sc, G = oracle.nvfp4_quant(hf)
            sg = np.repeat(np.array([oracle.e4m3(int(b)) for b in sc]) * G, 16)
            sg[sg == 0] = np.inf
            dq = np.abs(h_gpu[pos[t * k + j]].astype(np.float64) - h_ref) / sg
            worst = max(worst, float(dq.max()))
    assert worst <= oracle.FLIP_Q / 4, f"h differs by {worst:.3e} code units"
    return worst


def draw_prefill_tokens(dw, layer: int, T: int, draw0: int = 0, batch: int = 64):
    """T tokens that pass both the router's near-tie rule and the prefill
    rounding-margin rule (prefill_clean)."""
    wl = dw.wl
    Wr, bias, _ = host_inputs(dw, layer)
    xs, d = [], draw0
    while sum(len(v) for v in xs) < T:
        x, idx = draw_tokens(wl, layer, batch, Wr, bias, draw0=d, batch=batch)
        d = idx[-1] + 1
        ids, *_ = oracle.route(x, Wr, bias, wl.k)
        xs.append(x[prefill_clean(dw, layer, x, ids)])
    return np.concatenate(xs)[:T]


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
