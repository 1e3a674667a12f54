"""GPU parity of whole layers (moe_layer_forward through the C ABI) against
the oracle on seeded inputs: ids bit-exact, router probabilities within 1e-5
relative, outputs within 2e-2 * rms; identity expert exact; residency
invariance bitwise; negative controls separated from the GPU-vs-oracle error."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_common import (check_outputs, check_permutation, check_router, draw_tokens, ffn_fp32,
                              host_inputs, oracle_layer, to_dev_bf16, y_to_f64)
from tests.helpers import TOL, identity_record, identity_x, bf16_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from routed_expert_layer_router_gb300 import moe
    moe.lib()
    gen._lib_cuda()


def _run(dw, layer, x):
    y = dw.moe_layers[layer].forward(to_dev_bf16(x))
    torch.cuda.synchronize()
    return y_to_f64(y)


@pytest.fixture(scope="module")
def tiny():
    import gen.device as gd
    dw = gd.build(gen.WORKLOADS["tiny"], T_max=64)
    yield dw
    dw.close()


@pytest.mark.parametrize("T", [1, 4, 37])
def test_tiny_layer_parity(tiny, T):
    dw = tiny
    Wr, bias, sh = host_inputs(dw, 0)
    x, _ = draw_tokens(dw.wl, 0, T, Wr, bias, draw0=100 * T)
    y = _run(dw, 0, x)
    y_ref, ids_r, w_r, p_r = oracle_layer(dw, 0, x)
    check_router(dw.moe_layers[0].debug(T), ids_r, w_r, p_r)
    check_permutation(dw.moe_layers[0].debug(T), ids_r)  # T <= 8: inside the router kernel
    check_outputs(y, y_ref)
    assert dw.moe_layers[0].read_status() == 0


@pytest.fixture(scope="module")
def decode():
    import gen.device as gd
    dw = gd.build(gen.WORKLOADS["decode"], T_max=8)
    yield dw
    dw.close()


def test_decode_layer_parity(decode):
    dw = decode
    Wr, bias, sh = host_inputs(dw, 0)
    x, _ = draw_tokens(dw.wl, 0, 3, Wr, bias)
    recs = {}
    for t in range(3):  # the decode workload: one token per forward
        y = _run(dw, 0, x[t:t + 1])
        y_ref, ids_r, w_r, p_r = oracle_layer(dw, 0, x[t:t + 1], record_cache=recs)
        check_router(dw.moe_layers[0].debug(1), ids_r, w_r, p_r)
        check_permutation(dw.moe_layers[0].debug(1), ids_r)
        check_outputs(y, y_ref)
    # a few tokens per forward as well (two-token staging path)
    y = _run(dw, 0, x)
    y_ref, ids_r, w_r, p_r = oracle_layer(dw, 0, x, record_cache=recs)
    check_router(dw.moe_layers[0].debug(3), ids_r, w_r, p_r)
    check_permutation(dw.moe_layers[0].debug(3), ids_r)
    check_outputs(y, y_ref)
    assert dw.moe_layers[0].read_status() == 0


def test_decode_negative_controls_are_far_from_gpu(decode):
    """Per-substep separation: the GPU's fp32 layer output (before the bf16
    rounding) is at least 100x closer to the oracle than to an oracle with a
    planted defect (nibble order, scale format, block offset, scaling 2.5)."""
    dw = decode
    Wr, bias, sh = host_inputs(dw, 0)
    x, _ = draw_tokens(dw.wl, 0, 1, Wr, bias, draw0=500)
    y = ffn_fp32(dw, 0, x)
    recs = {}
    y_ref, *_ = oracle_layer(dw, 0, x, record_cache=recs)
    base = np.abs(y - y_ref).max()
    assert base <= 1e-3 * np.sqrt(np.mean(y_ref ** 2))
    for name in ("nibble_swap", "scale_ue8m0", "block_off_by_one", "scaling_2_5"):
        with oracle.defect(name):
            y_bad, *_ = oracle_layer(dw, 0, x, record_cache=recs)
        assert np.abs(y - y_bad).max() >= 100 * base, name


def _identity_workload(H, I, E, k, T_max, n_cache, n_stage, hot):
    """A layer whose experts are all the identity expert; `hot` of them cached."""
    from routed_expert_layer_router_gb300.layer import ExpertCache, HostArena, MoELayer
    rec = identity_record(H, I)
    rb = rec.size
    arena = HostArena(E, rb)
    arena.array[:] = rec
    arena.register()
    host_index = np.arange(E, dtype=np.int64)[None, :]
    cache = ExpertCache(1, E, H, I, n_cache_slots=n_cache, n_stage=n_stage,
                        layer_slots=[0, n_cache], host_arena=arena, host_index=host_index)
    dev_rec = torch.from_numpy(rec).cuda()
    from routed_expert_layer_router_gb300.layer import device_view
    for j, e in enumerate(hot):
        device_view(cache.slot_ptr(j), (rb,), torch.uint8).copy_(dev_rec)
        cache.set_resident(0, e, j)
    wr = torch.from_numpy(gen.router_f32(31, 0, E, H)).cuda()
    g = torch.ones((E, 3), dtype=torch.float32, device="cuda")
    layer = MoELayer(cache, 0, wr, g, k, T_max=T_max)
    return layer, cache, arena


@pytest.mark.parametrize("hot", ["all", "none", "half"])
def test_identity_expert_exact_and_residency_invariant(hot):
    H, I, E, k, T = 256, 128, 16, 4, 6
    hot_list = {"all": list(range(E)), "none": [], "half": list(range(0, E, 2))}[hot]
    n_cache = max(len(hot_list), 1)
    layer, cache, arena = _identity_workload(H, I, E, k, T, n_cache, n_stage=5, hot=hot_list)
    try:
        x = identity_x(H, T, seed=7)
        y = layer.forward(to_dev_bf16(x))
        torch.cuda.synchronize()
        yb = y.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(yb[:, 16:16 + I], x[:, 16:16 + I])
        assert not yb[:, :16].any() and not yb[:, 16 + I:].any()
        assert layer.read_status() == 0
    finally:
        layer.close()
        cache.close()
        arena.close()


def test_residency_invariance_bitwise():
    """Same records served from cache slots, from staging (gathered from the
    host arena) or a mix: identical output bits."""
    import gen.device as gd
    wl = gen.WORKLOADS["tiny"]
    outs = []
    for resident in (list(range(wl.E)), [], list(range(0, wl.E, 2))):
        dw = gd.build(wl, T_max=8, resident=[resident], n_stage=3)
        Wr, bias, sh = host_inputs(dw, 0)
        x, _ = draw_tokens(wl, 0, 8, Wr, bias, draw0=777)
        outs.append(dw.moe_layers[0].forward(to_dev_bf16(x)).view(torch.int16).cpu().numpy())
        assert dw.moe_layers[0].read_status() == 0
        dw.close()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_stack_layers_parity():
    """Decode stack: all 16 layers, Zipf-skewed routing, 66 hot experts per
    layer in HBM, the rest gathered from pinned host memory; each layer vs the
    oracle."""
    import gen.device as gd
    wl = gen.WORKLOADS["stack"]
    layers = wl.layers
    dw = gd.build(wl, layers=layers, T_max=1, alias_host_records=True)
    try:
        recs = {}
        hits = misses = 0
        for l in range(layers):
            Wr, bias, sh = host_inputs(dw, l)
            x, _ = draw_tokens(wl, l, 1, Wr, bias, draw0=3)
            y = _run(dw, l, x)
            y_ref, ids_r, w_r, p_r = oracle_layer(dw, l, x, record_cache=recs)
            dbg = dw.moe_layers[l].debug(1)
            check_router(dbg, ids_r, w_r, p_r)
            check_outputs(y, y_ref)
            n_act, n_hit = dbg["n_act"].cpu().tolist()
            hits += n_hit
            misses += n_act - n_hit
            assert dw.moe_layers[l].read_status() == 0
        assert misses > 0 and hits > 0
    finally:
        dw.close()


def test_flat_batched_parity():
    """Batched flat routing: 64 tokens, 72 experts per layer cached by
    saliency, the rest gathered in groups through the staging slots."""
    import gen.device as gd
    wl = gen.WORKLOADS["flat"]
    order = [list(np.random.default_rng(l).permutation(wl.E)) for l in range(1)]
    dw = gd.build(wl, layers=1, T_max=64, saliency_order=order, n_stage=64)
    try:
        Wr, bias, sh = host_inputs(dw, 0)
        x, _ = draw_tokens(wl, 0, 64, Wr, bias, draw0=11)
        y = _run(dw, 0, x)
        y_ref, ids_r, w_r, p_r = oracle_layer(dw, 0, x)  # every token
        dbg = dw.moe_layers[0].debug(64)
        check_router(dbg, ids_r, w_r, p_r)
        check_permutation(dbg, ids_r)
        n_act, n_hit = dbg["n_act"].cpu().tolist()
        assert n_act - n_hit > 64  # several staging groups
        check_outputs(y, y_ref)
        assert dw.moe_layers[0].read_status() == 0
    finally:
        dw.close()


def test_decode_flags_activation_beyond_f16():
    """The decode path holds activations in f16: a token with an element of
    magnitude above 65504 is reported as MOE_ERR_UNSUPPORTED in the status
    word (not silently turned into inf), and an in-range call after it is
    clean again."""
    import gen.device as gd
    from routed_expert_layer_router_gb300 import moe
    wl = gen.WORKLOADS["tiny"]
    dw = gd.build(wl, T_max=wl.T)
    try:
        Wr, bias, _ = host_inputs(dw, 0)
        x, _ = draw_tokens(wl, 0, wl.T, Wr, bias)
        layer = dw.moe_layers[0]
        layer.forward(to_dev_bf16(x))
        assert layer.read_status() == 0
        xb = x.copy()
        xb[1, 37] = 0x4880  # bf16 262144 = 2^18
        layer.forward(to_dev_bf16(xb))
        assert layer.read_status() == moe.MOE_ERR_UNSUPPORTED
        layer.forward(to_dev_bf16(x))
        assert layer.read_status() == 0
    finally:
        dw.close()


def test_decode_tokens_and_output_in_pinned_host_memory():
    """moe_layer_forward with y in pinned host memory (the decode path's last
    kernel stores it there), and with x in pinned host memory too (the layer
    copies it in with its first kernel): bit for bit the device-memory call."""
    import gen.device as gd
    wl = gen.WORKLOADS["decode"]
    dw = gd.build(wl, T_max=1)
    try:
        layer = dw.moe_layers[0]
        x = torch.empty((3, wl.H), dtype=torch.bfloat16, device="cuda")
        gen.dev_x_bf16(wl.seed, 0, 9000, 3, wl.H, x.data_ptr(), torch.cuda.current_stream().cuda_stream)
        yd = torch.empty((3, wl.H), dtype=torch.bfloat16, device="cuda")
        yh = torch.empty((3, wl.H), dtype=torch.bfloat16, pin_memory=True)
        xh = x.cpu().pin_memory()
        yhh = torch.empty((3, wl.H), dtype=torch.bfloat16, pin_memory=True)
        for t in range(3):
            layer.forward(x[t:t + 1], yd[t:t + 1])
            layer.forward(x[t:t + 1], yh[t:t + 1])
            layer.forward(xh[t:t + 1], yhh[t:t + 1])
        torch.cuda.synchronize()
        assert layer.read_status() == 0
        assert torch.equal(yd.cpu().view(torch.int16), yh.view(torch.int16))
        assert torch.equal(yd.cpu().view(torch.int16), yhh.view(torch.int16))
    finally:
        dw.close()
