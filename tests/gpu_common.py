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
        recs = gen.expert_records(wl.seed, rl, missing, wl.H, wl.I, fmt=wl.fmt)
        for e, r in zip(missing, recs):
            cache[(rl, e)] = r
    records = {e: cache[(rl, e)] for e in need}
    y, ids2, w2, p2, bound = oracle.layer_forward(x, wl.H, wl.I, wl.E, wl.k, Wr, bias, records,
                                                  dw.gscale_host[layer], shared_w=sh, mode=mode,
                                                  return_bound=True, fmt=wl.fmt)
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
    recs = dict(zip(need, gen.expert_records(wl.seed, rl, need, wl.H, wl.I, fmt=wl.fmt)))
    return oracle.prefill_near_boundary(x, wl.H, wl.I, wl.k, ids, recs,
                                        dw.gscale_host[layer], fmt=wl.fmt) == 0


_E2M1 = None


def nvfp4_dequant(codes, scales, G):
    """Values of an NVFP4-quantised row (oracle.nvfp4_quant layout), fp64."""
    global _E2M1
    if _E2M1 is None:
        _E2M1 = (np.array([oracle.e2m1(c) for c in range(16)]),
                 np.array([oracle.e4m3(b) for b in range(256)]))
    c = np.stack([codes & 15, codes >> 4], 1).ravel()
    return _E2M1[0][c] * np.repeat(_E2M1[1][scales], 16) * G


def mxfp4_dequant(codes, scales):
    """Values of an MXFP4-quantised row (oracle.mxfp4_quant layout), fp64."""
    global _E2M1
    if _E2M1 is None:
        nvfp4_dequant(np.zeros(8, np.uint8), np.zeros(1, np.uint8), 1.0)
    c = np.stack([codes & 15, codes >> 4], 1).ravel()
    return _E2M1[0][c] * np.repeat([oracle.e8m0(int(b)) for b in scales], 32)


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
    recs = dict(zip(need, gen.expert_records(wl.seed, rl, need, H, I, fmt=wl.fmt)))
    pos = np.empty(perm.size, np.int64)
    pos[perm] = np.arange(perm.size)  # route r -> its expert-sorted position
    worst = 0.0
    mx = wl.fmt == oracle.MXFP4
    for i, t in enumerate(tokens):
        xf = bf16_to_f64(x[t]).astype(np.float32)
        xq = mxfp4_dequant(*oracle.mxfp4_quant(xf)) if mx else nvfp4_dequant(*oracle.nvfp4_quant(xf))
        for j in range(k):
            e = int(ids[i, j])
            h_ref = oracle.expert_h(recs[e], H, I, dw.gscale_host[layer][e], xq, fmt=wl.fmt)
            hf = h_ref.astype(np.float32)
            if mx:
                _, sc = oracle.mxfp4_quant(hf)
                sg = np.repeat(np.array([oracle.e8m0(int(b)) for b in sc]), 32)
            else:
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


def ffn_fp32(dw, layer, x):
    """The layer's output before the final bf16 rounding: the individual ABI
    calls (route, permute, lookup, expert FFN) with test-owned buffers, then
    sum_j o_route + o_shared in fp64 on the host (comparison only)."""
    from routed_expert_layer_router_gb300 import moe
    wl = dw.wl
    T, H, I, E, k, Is = x.shape[0], wl.H, wl.I, wl.E, wl.k, wl.Is
    s = torch.cuda.current_stream().cuda_stream
    i32, f32 = torch.int32, torch.float32
    z = {n: torch.zeros(sz, dtype=dt, device="cuda") for n, sz, dt in (
        ("ids", T * k, i32), ("w", T * k, f32), ("p", T * k, f32), ("lg", T * E, f32),
        ("counts", E, i32), ("off", E + 1, i32), ("perm", T * k, i32), ("inv", T * k, i32),
        ("src", E, i32), ("act", E, i32), ("nact", 2, i32), ("miss", E, i32), ("nmiss", 1, i32),
        ("st", 1, i32), ("o", T * k * H, f32), ("os", T * H, f32))}
    xd = to_dev_bf16(x)
    ra = moe.moe_route_args()
    ra.x, ra.w_router = xd.data_ptr(), dw.w_router[layer].data_ptr()
    ra.bias = dw.bias[layer].data_ptr() if dw.bias[layer] is not None else None
    ra.T, ra.H, ra.E, ra.k = T, H, E, k
    ra.ids, ra.w, ra.p_sel, ra.logits = (z[n].data_ptr() for n in ("ids", "w", "p", "lg"))
    moe.moe_route(ra, s)
    moe.moe_permute(z["ids"].data_ptr(), T, k, E, z["counts"].data_ptr(), z["off"].data_ptr(),
                    z["perm"].data_ptr(), z["inv"].data_ptr(), 0, 128, z["st"].data_ptr(), s)
    moe.expcache_lookup(dw.cache.handle, layer, z["counts"].data_ptr(), z["src"].data_ptr(),
                        z["act"].data_ptr(), z["nact"].data_ptr(), z["miss"].data_ptr(),
                        z["nmiss"].data_ptr(), z["st"].data_ptr(), s)
    ws_b = moe.moe_ffn_workspace_bytes(0, T, H, I, E, k, Is)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    fa = moe.moe_ffn_args()
    fa.mode, fa.stages, fa.T, fa.H, fa.I, fa.E, fa.k = 0, 3, T, H, I, E, k
    fa.x, fa.cache, fa.gscale = xd.data_ptr(), dw.cache.handle, dw.gscale[layer].data_ptr()
    fa.src_slot, fa.act_list, fa.n_act = (z[n].data_ptr() for n in ("src", "act", "nact"))
    fa.offsets, fa.perm, fa.w = z["off"].data_ptr(), z["perm"].data_ptr(), z["w"].data_ptr()
    fa.group, fa.n_stage, fa.Is = 0, dw.cache.n_stage, Is
    if Is:
        fa.s_gate, fa.s_up, fa.s_down = (t.data_ptr() for t in dw.shared[layer])
    fa.o_route, fa.o_shared = z["o"].data_ptr(), z["os"].data_ptr() if Is else None
    fa.workspace, fa.workspace_bytes, fa.status = ws.data_ptr(), ws_b, z["st"].data_ptr()
    moe.moe_expert_ffn(fa, s)
    torch.cuda.synchronize()
    assert z["st"].item() == 0
    o = z["o"].double().view(T * k, H).cpu().numpy()
    inv = z["inv"].cpu().numpy()
    y = np.stack([o[inv[t * k:(t + 1) * k]].sum(0) for t in range(T)])
    if Is:
        y += z["os"].double().view(T, H).cpu().numpy()
    return y
