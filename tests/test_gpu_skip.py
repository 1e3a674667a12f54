"""GPU parity of the renorm-skip (moe_layer_desc.skip_tau) against the
oracle's: the routes whose expert misses the cache and whose weight is below
tau are dropped, the rest renormalised; outputs within 2e-2 * rms of the
oracle run with the same residency and tau.  Tokens whose missing routes sit
within 1e-4 of tau are left out (fp32 and fp64 weights may fall on either
side)."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_common import (check_outputs, check_router, draw_tokens, host_inputs,
                              oracle_layer, to_dev_bf16, y_to_f64)

pytestmark = pytest.mark.gpu

MARGIN = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from routed_expert_layer_router_gb300 import moe
    moe.lib()
    gen._lib_cuda()


def _tokens(wl, l, T, Wr, bias, resident, tau, draw0):
    """T tokens none of whose missing routes has |w - tau| < MARGIN."""
    out, d = [], draw0
    while len(out) < T:
        x, _ = draw_tokens(wl, l, 1, Wr, bias, draw0=d)
        d += 1
        ids, w, _, _, _ = oracle.route(x, Wr, bias, wl.k)
        miss = ~resident[ids[0]]
        if np.all(np.abs(w[0][miss] - tau) > MARGIN):
            out.append(x[0])
    return np.stack(out)


def _check_layer(dw, l, x, resident, tau, recs):
    wl = dw.wl
    Wr, bias, sh = host_inputs(dw, l)
    y = y_to_f64(dw.moe_layers[l].forward(to_dev_bf16(x)))
    torch.cuda.synchronize()
    rl = dw.record_layer[l] if dw.record_layer else l
    ids, w, p, _, _ = oracle.route(x, Wr, bias, wl.k)
    _, keep = oracle.renorm_skip(ids, w, resident, tau)
    need = sorted(set(ids[keep].ravel().tolist()))
    missing = [e for e in need if (rl, e) not in recs]
    for e, r in zip(missing, gen.expert_records(wl.seed, rl, missing, wl.H, wl.I)):
        recs[(rl, e)] = r
    y_ref, ids_r, w_r, p_r = oracle.layer_forward(
        x, wl.H, wl.I, wl.E, wl.k, Wr, bias, {e: recs[(rl, e)] for e in need},
        dw.gscale_host[l], shared_w=sh, resident=resident, tau=tau)
    check_router(dw.moe_layers[l].debug(x.shape[0]), ids_r, w_r, p_r)
    check_outputs(y, y_ref)
    assert dw.moe_layers[l].read_status() == 0
    return int((~keep).sum())


def test_stack_renorm_skip():
    """Two stack layers (one token per forward: the fused router kernel)."""
    import gen.device as gd
    wl = gen.WORKLOADS["stack"]
    tau = 0.05
    dw = gd.build(wl, layers=2, T_max=1, alias_host_records=True, skip_tau=tau)
    try:
        recs, dropped = {}, 0
        table = dw.cache.table().cpu().numpy()
        for l in range(2):
            Wr, bias, _ = host_inputs(dw, l)
            resident = table[l] >= 0
            xs = _tokens(wl, l, 3, Wr, bias, resident, tau, draw0=700)
            for t in range(3):
                dropped += _check_layer(dw, l, xs[t:t + 1], resident, tau, recs)
        assert dropped > 0
    finally:
        dw.close()


def test_tiny_renorm_skip_many_tokens():
    """16 tokens (more than the fused kernel takes: the skip runs as a kernel
    of its own before the permutation)."""
    import gen.device as gd
    wl = gen.WORKLOADS["tiny"]
    tau = 0.45  # below 1/k = 0.5
    dw = gd.build(wl, T_max=16, resident=[list(range(0, wl.E, 2))], skip_tau=tau)
    try:
        Wr, bias, _ = host_inputs(dw, 0)
        resident = dw.cache.table().cpu().numpy()[0] >= 0
        x = _tokens(wl, 0, 16, Wr, bias, resident, tau, draw0=900)
        assert _check_layer(dw, 0, x, resident, tau, {}) > 0
    finally:
        dw.close()
