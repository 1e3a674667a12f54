"""GPU parity of the prefill path (NVFP4 activation quantisation + tcgen05
grouped GEMMs) against the oracle's prefill numerics: the identity expert
exact; a small layer on every token; the 4096-token layer's router outputs
on every token and its outputs on 64 tokens spread over every expert group;
the masked prefill (experts the chunk does not route to are skipped) at 8,
20 and 47 tokens.  The gate/up GEMM's h is compared with the oracle's h
before its re-quantisation.  Output comparisons keep the tokens whose routes'
h is clear of every NVFP4 rounding boundary by the oracle's margin
(prefill_clean), as the router comparisons keep tokens clear of near-ties."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_common import (check_outputs, check_permutation, check_prefill_h, check_router,
                              draw_prefill_tokens, draw_tokens, host_inputs, oracle_layer,
                              prefill_clean, to_dev_bf16, y_to_f64)
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
        x = draw_prefill_tokens(dw, 0, SMALL.T)
        layer = dw.moe_layers[0]
        y = layer.forward(to_dev_bf16(x))
        torch.cuda.synchronize()
        assert layer.read_status() == 0
        y_ref, ids, w, p, bound = oracle_layer(dw, 0, x, mode=1, return_bound=True)
        dbg = layer.debug(SMALL.T)
        check_router(dbg, ids, w, p)
        check_permutation(dbg, ids)
        check_prefill_h(dw, 0, x, layer.debug_prefill(SMALL.T)["h"].cpu().numpy(),
                        dbg["perm"].cpu().numpy(), list(range(0, SMALL.T, 7)))
        check_outputs(y_to_f64(y), y_ref, bound=bound)
    finally:
        dw.close()


def test_prefill_4096_tokens_parity():
    """The 4096-token prefill layer (288 experts top-8, all resident) in the
    launch configuration the bench times: ids, weights and probabilities of
    all 4096 tokens and the permutation against the oracle's router; outputs
    of 64 tokens spread over the chunk whose routes reach every group of 64
    experts (the order the GEMMs walk them), and the h of 8 of them."""
    import gen.device as gd
    wl = gen.WORKLOADS["prefill"]
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
        assert len(np.unique(ids_r)) == wl.E  # every expert is hit
        # 64 clean tokens, taken in a stride over the chunk
        order = (np.arange(wl.T) * 1031) % wl.T
        sample = []
        for i0 in range(0, wl.T, 48):
            cand = order[i0:i0 + 48]
            ok = prefill_clean(dw, 0, x[cand], ids_r[cand])
            sample += [int(t) for t in cand[ok]]
            if len(sample) >= 64:
                break
        sample = sorted(sample[:64])
        assert len(sample) == 64
        assert set(ids_r[sample].ravel() // 64) == set(range((wl.E + 63) // 64))
        y_ref, ids_s, w_s, p_s, bound = oracle_layer(dw, 0, x[sample], mode=1, return_bound=True)
        assert np.array_equal(ids_s, ids_r[sample])
        check_outputs(y_to_f64(y)[sample], y_ref, bound=bound)
        check_prefill_h(dw, 0, x, layer.debug_prefill(wl.T)["h"].cpu().numpy(),
                        dbg["perm"].cpu().numpy(), sample[::8])
    finally:
        dw.close()


_POOL = {}


@pytest.mark.parametrize("group", [0, 64])
def test_masked_prefill_parity(group):
    """The masked grouped prefill (the tile plan walks only the experts the
    chunk routes to) on the 6144 x 2048, 288-expert layer switched to the
    prefill path from 8 tokens: at 8, 20 and 47 tokens most experts are
    unused.  Router, permutation, h and every output against the oracle."""
    import gen.device as gd
    wl = gen.WORKLOADS["decode"]
    dw = gd.build(wl, T_max=47, prefill_min_tokens=8, prefill_group=group)
    try:
        layer = dw.moe_layers[0]
        if "decode" not in _POOL:  # the same tokens for both groupings
            _POOL["decode"] = draw_prefill_tokens(dw, 0, 8 + 20 + 47, draw0=5000)
        pool = _POOL["decode"]
        i0 = 0
        for T in (8, 20, 47):
            x = pool[i0:i0 + T]
            i0 += T
            y = layer.forward(to_dev_bf16(x))
            torch.cuda.synchronize()
            assert layer.read_status() == 0
            dbg = layer.debug(T)
            y_ref, ids, w, p, bound = oracle_layer(dw, 0, x, mode=1, return_bound=True)
            check_router(dbg, ids, w, p)
            check_permutation(dbg, ids)
            n_act = int(dbg["n_act"][0])
            assert n_act == len(np.unique(ids)) < wl.E  # experts left out
            check_prefill_h(dw, 0, x, layer.debug_prefill(T)["h"].cpu().numpy(),
                            dbg["perm"].cpu().numpy(), [0, T - 1])
            check_outputs(y_to_f64(y), y_ref, bound=bound)
    finally:
        dw.close()


def test_prefill_public_calls_match_the_layer():
    """The PREFILL expert FFN through the individual ABI calls (route, padded
    permutation, lookup, moe_expert_ffn adding into a caller-zeroed y_acc,
    moe_combine) against the oracle, beside the layer's own sequence (which
    clears its sum in the token quantisation and lets the shared expert's
    down GEMM write y): both within the tolerance on the same tokens."""
    from routed_expert_layer_router_gb300 import moe
    import gen.device as gd
    dw = gd.build(SMALL, T_max=SMALL.T)
    try:
        wl = SMALL
        T, H, I, E, k, Is = wl.T, wl.H, wl.I, wl.E, wl.k, wl.Is
        x = draw_prefill_tokens(dw, 0, T)
        y_layer = dw.moe_layers[0].forward(to_dev_bf16(x))
        s = torch.cuda.current_stream().cuda_stream
        i32, f32 = torch.int32, torch.float32
        z = {n: torch.zeros(sz, dtype=dt, device="cuda") for n, sz, dt in (
            ("ids", T * k, i32), ("w", T * k, f32), ("p", T * k, f32), ("lg", T * E, f32),
            ("counts", E, i32), ("off", E + 1, i32), ("pad", E + 1, i32), ("perm", T * k, i32),
            ("inv", T * k, i32), ("src", E, i32), ("act", E, i32), ("nact", 2, i32),
            ("miss", E, i32), ("nmiss", 1, i32), ("st", 1, i32), ("os", T * H, f32),
            ("yacc", T * H, f32))}
        xd = to_dev_bf16(x)
        ra = moe.moe_route_args()
        ra.x, ra.w_router = xd.data_ptr(), dw.w_router[0].data_ptr()
        ra.T, ra.H, ra.E, ra.k = T, H, E, k
        ra.ids, ra.w, ra.p_sel, ra.logits = (z[n].data_ptr() for n in ("ids", "w", "p", "lg"))
        moe.moe_route(ra, s)
        moe.moe_permute(z["ids"].data_ptr(), T, k, E, z["counts"].data_ptr(), z["off"].data_ptr(),
                        z["perm"].data_ptr(), z["inv"].data_ptr(), z["pad"].data_ptr(), 128,
                        z["st"].data_ptr(), s)
        moe.expcache_lookup(dw.cache.handle, 0, z["counts"].data_ptr(), z["src"].data_ptr(),
                            z["act"].data_ptr(), z["nact"].data_ptr(), z["miss"].data_ptr(),
                            z["nmiss"].data_ptr(), z["st"].data_ptr(), s)
        ws_b = moe.moe_ffn_workspace_bytes(1, T, H, I, E, k, Is)
        ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
        fa = moe.moe_ffn_args()
        fa.mode, fa.stages, fa.T, fa.H, fa.I, fa.E, fa.k = 1, 3, T, H, I, E, k
        fa.x, fa.cache, fa.gscale = xd.data_ptr(), dw.cache.handle, dw.gscale[0].data_ptr()
        fa.src_slot, fa.act_list, fa.n_act = (z[n].data_ptr() for n in ("src", "act", "nact"))
        fa.offsets, fa.pad_offsets = z["off"].data_ptr(), z["pad"].data_ptr()
        fa.perm, fa.inv, fa.w = z["perm"].data_ptr(), z["inv"].data_ptr(), z["w"].data_ptr()
        fa.group, fa.n_stage, fa.prefill_group, fa.Is = 0, 0, wl.group, Is
        fa.s_gate, fa.s_up, fa.s_down = (t.data_ptr() for t in dw.shared[0])
        fa.o_shared, fa.y_acc = z["os"].data_ptr(), z["yacc"].data_ptr()
        fa.workspace, fa.workspace_bytes, fa.status = ws.data_ptr(), ws_b, z["st"].data_ptr()
        moe.moe_expert_ffn(fa, s)
        y_pub = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        ca = moe.moe_combine_args()
        ca.T, ca.H, ca.k = T, H, k
        ca.y_acc, ca.inv, ca.y = z["yacc"].data_ptr(), z["inv"].data_ptr(), y_pub.data_ptr()
        moe.moe_combine(ca, s)
        torch.cuda.synchronize()
        assert z["st"].item() == 0 and dw.moe_layers[0].read_status() == 0
        y_ref, _, _, _, bound = oracle_layer(dw, 0, x, mode=1, return_bound=True)
        check_outputs(y_to_f64(y_pub), y_ref, bound=bound)
        check_outputs(y_to_f64(y_layer), y_ref, bound=bound)
        # the two orders of adding the shared expert differ by bf16 rounding at most
        d = np.abs(y_to_f64(y_pub) - y_to_f64(y_layer))
        assert d.max() <= 2.0 ** -7 * np.abs(y_to_f64(y_layer)).max()
    finally:
        dw.close()


def test_prefill_tokens_and_output_in_pinned_host_memory():
    """The prefill layer called on pinned host buffers (the layer copies x in
    with its first kernel; the shared expert's down GEMM stores y into host
    memory) against the same call on device buffers.  The down GEMMs' L2
    reductions add in any order, so the two may differ by a bf16 rounding."""
    import gen.device as gd
    dw = gd.build(SMALL, T_max=SMALL.T)
    try:
        layer = dw.moe_layers[0]
        x = draw_prefill_tokens(dw, 0, SMALL.T)
        xd = to_dev_bf16(x)
        yd = layer.forward(xd)
        xh = xd.cpu().pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        layer.forward(xh, yh)
        torch.cuda.synchronize()
        assert layer.read_status() == 0
        a, b = y_to_f64(yd), y_to_f64(yh)
        assert np.abs(a - b).max() <= 2.0 ** -7 * np.abs(a).max()
        y_ref, _, _, _, bound = oracle_layer(dw, 0, x, mode=1, return_bound=True)
        check_outputs(b, y_ref, bound=bound)
    finally:
        dw.close()
