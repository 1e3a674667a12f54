"""GPU parity of the prefill path (NVFP4 activation quantisation + tcgen05
grouped GEMMs) against the oracle's prefill numerics: identity expert exact,
a small layer on every token, the 4096-token layer on sampled tokens."""
import numpy as np
import pytest
import torch

import gen
from tests.gpu_common import (check_outputs, check_router, draw_tokens, host_inputs,
                              oracle_layer, to_dev_bf16, y_to_f64)
from tests.helpers import identity_record, nvfp4_exact_x

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from routed_expert_layer_router_gb300 import moe
    moe.lib()
    gen._lib_cuda()


def test_prefill_identity_expert_exact():
    """Every expert is the identity expert and the tokens are exactly
    representable in NVFP4 (and so is h = 64 x): the tensor-core path must
    return the input bit for bit."""
    from routed_expert_layer_router_gb300.layer import ExpertCache, MoELayer, device_view
    H, I, E, k, T = 512, 256, 8, 3, 160
    rec = identity_record(H, I)
    cache = ExpertCache(1, E, H, I, n_cache_slots=E, n_stage=0, layer_slots=[0, E])
    try:
        dev_rec = torch.from_numpy(rec).cuda()
        for e in range(E):
            device_view(cache.slot_ptr(e), (rec.size,), torch.uint8).copy_(dev_rec)
            cache.set_resident(0, e, e)
        wr = torch.from_numpy(gen.router_f32(41, 0, E, H)).cuda()
        g = torch.ones((E, 3), dtype=torch.float32, device="cuda")
        layer = MoELayer(cache, 0, wr, g, k, T_max=T, prefill_min_tokens=1, prefill_group=3)
        x = nvfp4_exact_x(H, T, seed=42)
        y = layer.forward(to_dev_bf16(x))
        torch.cuda.synchronize()
        yv = y_to_f64(y)  # compared as values: a -0.0 input comes back as +0.0
        xv = y_to_f64(to_dev_bf16(x))
        assert layer.read_status() == 0
        assert np.array_equal(yv[:, 16:16 + I], xv[:, 16:16 + I])
        assert not yv[:, :16].any() and not yv[:, 16 + I:].any()
        layer.close()
    finally:
        cache.close()


SMALL = gen.Workload("prefill-small", H=512, I=256, E=16, k=4, T=300, layers=1, Is=256, seed=5,
                     prefill=True, group=6)


def test_prefill_small_layer_parity():
    import gen.device as gd
    dw = gd.build(SMALL, T_max=SMALL.T)
    try:
        Wr, bias, sh = host_inputs(dw, 0)
        x, _ = draw_tokens(SMALL, 0, SMALL.T, Wr, bias)
        y = dw.moe_layers[0].forward(to_dev_bf16(x))
        torch.cuda.synchronize()
        assert dw.moe_layers[0].read_status() == 0
        y_ref, ids, w, p, bound = oracle_layer(dw, 0, x, mode=1, return_bound=True)
        check_router(dw.moe_layers[0].debug(SMALL.T), ids, w, p)
        check_outputs(y_to_f64(y), y_ref, bound=bound)
    finally:
        dw.close()


def test_prefill_4096_tokens_sampled_parity():
    """The 4096-token prefill layer (288 experts top-8, all resident, groups of
    64) in the launch configuration the bench times; the oracle recomputes
    eight sampled tokens."""
    import gen.device as gd
    wl = gen.WORKLOADS["prefill"]
    dw = gd.build(wl, T_max=wl.T)
    try:
        Wr, bias, sh = host_inputs(dw, 0)
        x, _ = draw_tokens(wl, 0, wl.T, Wr, bias, batch=512)
        y = dw.moe_layers[0].forward(to_dev_bf16(x))
        torch.cuda.synchronize()
        assert dw.moe_layers[0].read_status() == 0
        dbg = dw.moe_layers[0].debug(wl.T)
        ids = dbg["ids"].cpu().numpy()
        assert len(np.unique(ids)) == wl.E  # every expert is hit
        sample = [0, 1, 511, 1024, 2047, 2500, 4000, 4095]
        y_ref, ids_r, w_r, p_r, bound = oracle_layer(dw, 0, x[sample], mode=1, return_bound=True)
        check_router({kk: (v[sample] if kk in ("ids", "w", "p_sel") else v) for kk, v in dbg.items()},
                     ids_r, w_r, p_r)
        check_outputs(y_to_f64(y)[sample], y_ref, bound=bound)
    finally:
        dw.close()
