"""GPU parity of the MXFP4 record format (windlass README: GLM-5.2 in MXFP4,
E2M1 values with an E8M0 scale per 32; OCP Microscaling Formats v1.0)
against the oracle: the bit-built identity expert exact through the decode
and the prefill (tcgen05 kind::mxf4nvf4, scale_vec::2X) paths; the tiny layer
and the 6144 x 2048, 288-expert decode layer; negative controls (flipped
nibble order, scales decoded as the other format) far from the GPU; the
prefill path on a small layer, masked on the 288-expert layer, and on the
4096-token layer (every token's routing; 32 clean tokens' outputs)."""
import dataclasses

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_common import (check_outputs, check_permutation, check_prefill_h, check_router,
                              draw_prefill_tokens, draw_tokens, ffn_fp32, host_inputs,
                              oracle_layer, to_dev_bf16, y_to_f64)
from tests.helpers import identity_record_mx, mxfp4_exact_x

pytestmark = pytest.mark.gpu

TINY_MX = dataclasses.replace(gen.WORKLOADS["tiny"], name="tiny-mx", fmt=gen.MXFP4, seed=10)
DECODE_MX = dataclasses.replace(gen.WORKLOADS["decode"], name="decode-mx", fmt=gen.MXFP4, seed=11)
SMALL_MX = gen.Workload("prefill-small-mx", H=512, I=256, E=16, k=4, T=300, layers=1, Is=256,
                        seed=12, prefill=True, group=6, fmt=gen.MXFP4)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from routed_expert_layer_router_gb300 import moe
    moe.lib()
    gen._lib_cuda()


@pytest.mark.parametrize("prefill", [False, True])
def test_mx_identity_expert_exact(prefill):
    from routed_expert_layer_router_gb300.layer import ExpertCache, MoELayer, device_view
    from routed_expert_layer_router_gb300 import moe
    H, I, E, k, T = 512, 256, 8, 3, 160 if prefill else 5
    rec = identity_record_mx(H, I)
    cache = ExpertCache(1, E, H, I, n_cache_slots=E, n_stage=0, layer_slots=[0, E],
                        fmt=moe.MOE_FMT_MXFP4)
    try:
        assert cache.record_bytes == rec.size
        dev_rec = torch.from_numpy(rec).cuda()
        for e in range(E):
            device_view(cache.slot_ptr(e), (rec.size,), torch.uint8).copy_(dev_rec)
            cache.set_resident(0, e, e)
        wr = torch.from_numpy(gen.router_f32(43, 0, E, H)).cuda()
        g = torch.ones((E, 3), dtype=torch.float32, device="cuda")
        layer = MoELayer(cache, 0, wr, g, k, T_max=T, prefill_min_tokens=1 if prefill else 0,
                         prefill_group=3)
        x = mxfp4_exact_x(H, T, seed=44)
        y = layer.forward(to_dev_bf16(x))
        torch.cuda.synchronize()
        assert layer.read_status() == 0
        yv, xv = y_to_f64(y), y_to_f64(to_dev_bf16(x))
        assert np.array_equal(yv[:, 16:16 + I], xv[:, 16:16 + I])
        assert not yv[:, :16].any() and not yv[:, 16 + I:].any()
        layer.close()
    finally:
        cache.close()


@pytest.mark.parametrize("T", [1, 4, 37])
def test_mx_tiny_layer_parity(T):
    import gen.device as gd
    dw = gd.build(TINY_MX, T_max=T)
    try:
        Wr, bias, _ = host_inputs(dw, 0)
        x, _ = draw_tokens(TINY_MX, 0, T, Wr, bias, draw0=T)
        layer = dw.moe_layers[0]
        y = layer.forward(to_dev_bf16(x))
        torch.cuda.synchronize()
        assert layer.read_status() == 0
        y_ref, ids, w, p = oracle_layer(dw, 0, x)
        dbg = layer.debug(T)
        check_router(dbg, ids, w, p)
        check_permutation(dbg, ids)
        check_outputs(y_to_f64(y), y_ref)
    finally:
        dw.close()


def test_mx_decode_layer_parity_and_negative_controls():
    """The 6144 x 2048, 288-expert decode layer with MXFP4 records: one token
    (two draws) and three tokens against the oracle; then per-substep
    separation: the GPU's fp32 layer output is at least 100x closer to the
    oracle than to an oracle with a flipped MXFP4 nibble order or with its
    scale bytes decoded in the other format."""
    import gen.device as gd
    dw = gd.build(DECODE_MX, T_max=3)
    try:
        Wr, bias, _ = host_inputs(dw, 0)
        layer = dw.moe_layers[0]
        recs = {}
        for T, draw0 in ((1, 0), (1, 50), (3, 100)):
            x, _ = draw_tokens(DECODE_MX, 0, T, Wr, bias, draw0=draw0)
            y = layer.forward(to_dev_bf16(x))
            torch.cuda.synchronize()
            assert layer.read_status() == 0
            y_ref, ids, w, p = oracle_layer(dw, 0, x, record_cache=recs)
            check_router(layer.debug(T), ids, w, p)
            check_outputs(y_to_f64(y), y_ref)
        x, _ = draw_tokens(DECODE_MX, 0, 1, Wr, bias, draw0=500)
        y = ffn_fp32(dw, 0, x)
        y_ref, *_ = oracle_layer(dw, 0, x, record_cache=recs)
        base = np.abs(y - y_ref).max()
        assert base <= 1e-3 * np.sqrt(np.mean(y_ref ** 2))
        for name in ("nibble_swap", "scale_ue8m0"):
            with oracle.defect(name):
                y_bad, *_ = oracle_layer(dw, 0, x, record_cache=recs)
            assert np.abs(y - y_bad).max() >= 100 * base, name
    finally:
        dw.close()


def test_mx_prefill_small_layer_parity():
    import gen.device as gd
    dw = gd.build(SMALL_MX, T_max=SMALL_MX.T)
    try:
        x = draw_prefill_tokens(dw, 0, SMALL_MX.T)
        layer = dw.moe_layers[0]
        y = layer.forward(to_dev_bf16(x))
        torch.cuda.synchronize()
        assert layer.read_status() == 0
        y_ref, ids, w, p, bound = oracle_layer(dw, 0, x, mode=1, return_bound=True)
        dbg = layer.debug(SMALL_MX.T)
        check_router(dbg, ids, w, p)
        check_permutation(dbg, ids)
        check_prefill_h(dw, 0, x, layer.debug_prefill(SMALL_MX.T)["h"].cpu().numpy(),
                        dbg["perm"].cpu().numpy(), list(range(0, SMALL_MX.T, 7)))
        check_outputs(y_to_f64(y), y_ref, bound=bound)
    finally:
        dw.close()


def test_mx_masked_prefill_parity():
    """The 288-expert MXFP4 layer on the prefill path at 20 and 47 tokens
    (most experts unused), groups of 64."""
    import gen.device as gd
    dw = gd.build(DECODE_MX, T_max=47, prefill_min_tokens=8, prefill_group=64)
    try:
        layer = dw.moe_layers[0]
        pool = draw_prefill_tokens(dw, 0, 20 + 47, draw0=7000)
        for T, x in ((20, pool[:20]), (47, pool[20:])):
            y = layer.forward(to_dev_bf16(x))
            torch.cuda.synchronize()
            assert layer.read_status() == 0
            dbg = layer.debug(T)
            y_ref, ids, w, p, bound = oracle_layer(dw, 0, x, mode=1, return_bound=True)
            check_router(dbg, ids, w, p)
            check_permutation(dbg, ids)
            check_prefill_h(dw, 0, x, layer.debug_prefill(T)["h"].cpu().numpy(),
                            dbg["perm"].cpu().numpy(), [0, T - 1])
            check_outputs(y_to_f64(y), y_ref, bound=bound)
    finally:
        dw.close()


PREFILL_MX = dataclasses.replace(gen.WORKLOADS["prefill"], name="prefill-mx", fmt=gen.MXFP4,
                                 seed=13)


def test_mx_prefill_4096_tokens_parity():
    """The 4096-token MXFP4 prefill layer (288 experts top-8, all resident,
    router logits on the tensor cores) in the bench's launch configuration:
    ids, weights and probabilities of every token and the permutation against
    the oracle's router; outputs of 32 clean tokens whose routes reach every
    group of 64 experts."""
    import gen.device as gd
    from tests.gpu_common import prefill_clean
    wl = PREFILL_MX
    dw = gd.build(wl, T_max=wl.T)
    try:
        Wr, bias, sh = host_inputs(dw, 0)
        x, _ = draw_tokens(wl, 0, wl.T, Wr, bias, batch=512)
        layer = dw.moe_layers[0]
        y = layer.forward(to_dev_bf16(x))
        torch.cuda.synchronize()
        assert layer.read_status() == 0
        dbg = layer.debug(wl.T)
        ids_r, w_r, p_r, _, _ = oracle.route(x, Wr, bias, wl.k)
        check_router(dbg, ids_r, w_r, p_r)
        check_permutation(dbg, ids_r)
        order = (np.arange(wl.T) * 1031) % wl.T
        sample = []
        for i0 in range(0, wl.T, 48):
            cand = order[i0:i0 + 48]
            ok = prefill_clean(dw, 0, x[cand], ids_r[cand])
            sample += [int(t) for t in cand[ok]]
            if len(sample) >= 32:
                break
        sample = sorted(sample[:32])
        assert len(sample) == 32
        assert set(ids_r[sample].ravel() // 64) == set(range((wl.E + 63) // 64))
        y_ref, ids_s, _, _, bound = oracle_layer(dw, 0, x[sample], mode=1, return_bound=True)
        assert np.array_equal(ids_s, ids_r[sample])
        check_outputs(y_to_f64(y)[sample], y_ref, bound=bound)
    finally:
        dw.close()
