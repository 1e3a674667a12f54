"""GPU parity of the individual ABI calls against the oracle (bit-exact for
ids, permutations, slots and gathered bytes; 1e-5 relative for router
probabilities)."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_common import draw_tokens, to_dev_bf16
from tests.helpers import PROB_RTOL, bf16_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import routed_expert_layer_router_gb300 as pkg
    from routed_expert_layer_router_gb300 import moe
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.lib()
    gen._lib_cuda()
    yield pkg


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("H,I", [(256, 128), (512, 256), (6144, 2048)])
def test_device_generator_matches_host(H, I):
    n = 2 if H < 6144 else 1
    recs = gen.expert_records(9, 3, list(range(n)), H, I)
    rb = gen.record_bytes(H, I)
    buf = torch.empty((n, rb), dtype=torch.uint8, device="cuda")
    for e in range(n):
        gen.dev_expert_record(9, 3, e, H, I, buf[e].data_ptr(), _stream())
    assert np.array_equal(buf.cpu().numpy(), recs)
    x = torch.empty((5, H), dtype=torch.int16, device="cuda")
    gen.dev_x_bf16(9, 3, 7, 5, H, x.data_ptr(), _stream())
    assert np.array_equal(x.cpu().numpy().view(np.uint16), gen.x_bf16(9, 3, 7, 5, H))
    wr = torch.empty((16, H), dtype=torch.float32, device="cuda")
    gen.dev_router_f32(9, 3, 16, H, wr.data_ptr(), _stream())
    assert np.array_equal(wr.cpu().numpy(), gen.router_f32(9, 3, 16, H))
    sg = torch.empty((128, H), dtype=torch.int16, device="cuda")
    su = torch.empty((128, H), dtype=torch.int16, device="cuda")
    sd = torch.empty((H, 128), dtype=torch.int16, device="cuda")
    gen.dev_shared_bf16(9, 3, 128, H, sg.data_ptr(), su.data_ptr(), sd.data_ptr(), _stream())
    hg, hu, hd = gen.shared_bf16(9, 3, 128, H)
    assert np.array_equal(sg.cpu().numpy().view(np.uint16), hg)
    assert np.array_equal(sd.cpu().numpy().view(np.uint16), hd)


def _route_gpu(x, Wr, bias, k, ctl=None, split=None):
    """moe_route; with `ctl` (a zeroed device buffer) the call gets a workspace
    control area, which lets up to 8 tokens run as one kernel; with `split`
    (a device buffer of moe_route_split_bytes) more than 1024 tokens take the
    tensor-core logits."""
    from routed_expert_layer_router_gb300 import moe
    T, H = x.shape
    E = Wr.shape[0]
    xd = to_dev_bf16(x)
    wd = torch.from_numpy(Wr).cuda()
    bd = torch.from_numpy(bias).cuda() if bias is not None else None
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    p = torch.empty((T, k), dtype=torch.float32, device="cuda")
    lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
    a = moe.moe_route_args()
    a.x, a.w_router, a.bias = xd.data_ptr(), wd.data_ptr(), bd.data_ptr() if bd is not None else None
    a.T, a.H, a.E, a.k = T, H, E, k
    a.ids, a.w, a.p_sel, a.logits = ids.data_ptr(), w.data_ptr(), p.data_ptr(), lg.data_ptr()
    if ctl is not None:
        a.workspace, a.workspace_bytes = ctl.data_ptr(), ctl.numel()
    if split is not None:
        a.w_split, a.w_split_bytes = split.data_ptr(), split.numel()
    moe.moe_route(a, _stream())
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), p.cpu().numpy(), lg.cpu().numpy()


@pytest.mark.parametrize("name,T,one_kernel", [
    ("tiny", 4, False), ("tiny", 37, False), ("decode", 1, False), ("decode", 8, False),
    ("decode", 64, False), ("decode", 300, False), ("decode", 1100, False),
    ("tiny", 4, True), ("decode", 1, True), ("decode", 8, True), ("decode", 64, True)])
def test_route_parity(name, T, one_kernel):
    wl = gen.WORKLOADS[name]
    Wr = gen.router_f32(wl.seed, 0, wl.E, wl.H)
    bias = gen.zipf_bias(wl.seed, 0, wl.E, 1.556)[0] if T == 8 else None
    x, _ = draw_tokens(wl, 0, T, Wr, bias)
    ids_r, w_r, p_r, lg_r, _ = oracle.route(x, Wr, bias, wl.k)
    ctl = torch.zeros(256, dtype=torch.uint8, device="cuda") if one_kernel else None
    for _ in range(2 if one_kernel else 1):  # the control area is reset by each call
        ids, w, p, lg = _route_gpu(x, Wr, bias, wl.k, ctl)
        assert np.array_equal(ids, ids_r)
        assert np.all(np.abs(w - w_r) <= PROB_RTOL * w_r)
        assert np.all(np.abs(p - p_r) <= PROB_RTOL * p_r)
        assert np.abs(lg - lg_r).max() <= 1e-5 * np.abs(lg_r).max()
    if one_kernel:
        assert int(ctl.view(torch.int32)[0].item()) == 0


ODD = gen.Workload("tc-odd", H=512, I=128, E=100, k=6, T=1300, layers=1, Is=0, seed=11)
WIDE = gen.Workload("tc-wide", H=512, I=128, E=1000, k=8, T=1100, layers=1, Is=0, seed=12)


@pytest.mark.parametrize("wl,T,with_bias", [(gen.WORKLOADS["tiny"], 1100, False),
                                            (ODD, 1300, True),
                                            (gen.WORKLOADS["decode"], 1100, False),
                                            (gen.WORKLOADS["decode"], 2200, True),
                                            (WIDE, 1100, True)])
def test_route_tensor_core_parity(wl, T, with_bias):
    """More than 1024 tokens with the weight-piece scratch: the logits run on
    the tensor cores from the three bf16 pieces of the fp32 router weights.
    The pieces must add up to the weights exactly (padding rows zero), and
    ids, weights, probabilities and logits must meet the router's bar.  The
    shapes cover a padded expert tile (16 and 100 experts) and a ragged last
    token tile (1100 and 1300 tokens), and two token tiles per CTA (2200
    tokens: more 128-token tiles than SMs), the second tile of the last pair
    holding 24 tokens; and 1000 experts (32 expert tiles, the last padded),
    paired at 1100 tokens."""
    from routed_expert_layer_router_gb300 import moe
    Wr = gen.router_f32(wl.seed, 0, wl.E, wl.H)
    bias = gen.zipf_bias(wl.seed, 0, wl.E, 1.556)[0] if with_bias else None
    x, _ = draw_tokens(wl, 0, T, Wr, bias, batch=512)
    ids_r, w_r, p_r, lg_r, _ = oracle.route(x, Wr, bias, wl.k)
    split = torch.zeros(moe.moe_route_split_bytes(wl.E, wl.H), dtype=torch.uint8, device="cuda")
    ids, w, p, lg = _route_gpu(x, Wr, bias, wl.k, split=split)
    E_pad = (wl.E + 31) // 32 * 32
    pieces = split.cpu().numpy().view(np.uint16).reshape(3, E_pad, wl.H)
    total = sum(bf16_to_f64(pieces[i]) for i in range(3))
    assert np.array_equal(total[:wl.E], Wr.astype(np.float64))
    assert not total[wl.E:].any()
    assert np.array_equal(ids, ids_r)
    assert np.all(np.abs(w - w_r) <= PROB_RTOL * w_r)
    assert np.all(np.abs(p - p_r) <= PROB_RTOL * p_r)
    err = np.abs(lg - lg_r).max()
    print(f"max logit error {err:.3g} (max |logit| {np.abs(lg_r).max():.3g})")
    assert err <= 1e-5 * np.abs(lg_r).max()


@pytest.mark.parametrize("T,k,E", [(1, 8, 288), (4, 2, 16), (64, 8, 288), (4096, 8, 288),
                                   (1000, 3, 1000), (0, 8, 288)])
def test_permute_parity(T, k, E):
    from routed_expert_layer_router_gb300 import moe
    rng = np.random.default_rng(T + k + E)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32) \
        if T else np.zeros((0, k), np.int32)
    d_ids = torch.from_numpy(ids).cuda()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pad = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(max(T * k, 1), dtype=torch.int32, device="cuda")
    inv = torch.empty(max(T * k, 1), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_permute(d_ids.data_ptr(), T, k, E, counts.data_ptr(), offsets.data_ptr(),
                    perm.data_ptr(), inv.data_ptr(), pad.data_ptr(), 128, status.data_ptr(),
                    _stream())
    torch.cuda.synchronize()
    c_r, o_r, p_r, i_r = oracle.permute(ids, E)
    assert np.array_equal(counts.cpu().numpy(), c_r)
    assert np.array_equal(offsets.cpu().numpy(), o_r)
    assert np.array_equal(perm.cpu().numpy()[:T * k], p_r)
    assert np.array_equal(inv.cpu().numpy()[:T * k], i_r)
    pc = ((c_r + 127) // 128) * 128
    assert np.array_equal(pad.cpu().numpy(), np.concatenate([[0], np.cumsum(pc)]))
    assert status.item() == 0


def test_permute_flags_bad_ids():
    from routed_expert_layer_router_gb300 import moe
    ids = torch.tensor([[0, 5], [3, 16]], dtype=torch.int32, device="cuda")  # 16 out of range
    E = 16
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    inv = torch.empty(4, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_permute(ids.data_ptr(), 2, 2, E, counts.data_ptr(), offsets.data_ptr(),
                    perm.data_ptr(), inv.data_ptr(), 0, 128, status.data_ptr(), _stream())
    torch.cuda.synchronize()
    assert status.item() == moe.MOE_ERR_DEVICE
    assert counts.sum().item() == 3 and inv[3].item() == -1


def test_lookup_and_gather():
    """Lookup classifies hits/misses (ascending ids, staging slot i mod S) and
    the gather copies host records into staging slots byte for byte."""
    from routed_expert_layer_router_gb300 import moe
    from routed_expert_layer_router_gb300.layer import ExpertCache, HostArena
    H, I, E, L = 256, 128, 16, 2
    rb = gen.record_bytes(H, I)
    host_recs = gen.expert_records(5, 1, list(range(E)), H, I)
    arena = HostArena(E, rb)
    arena.array[:] = host_recs
    arena.register()
    host_index = np.full((L, E), -1, np.int64)
    host_index[1] = np.arange(E)
    cache = ExpertCache(L, E, H, I, n_cache_slots=6, n_stage=3,
                        layer_slots=[0, 2, 6], host_arena=arena, host_index=host_index)
    try:
        s = _stream()
        for j, e in enumerate([2, 9, 11, 14]):  # layer 1 owns slots 2..5
            torch.from_numpy(host_recs[e]).cuda()  # warm
            slot_t = torch.from_numpy(host_recs[e]).cuda()
            moe_ptr = cache.slot_ptr(2 + j)
            torch.cuda.synchronize()
            from routed_expert_layer_router_gb300.layer import device_view
            device_view(moe_ptr, (rb,), torch.uint8).copy_(slot_t)
            cache.set_resident(1, e, 2 + j)
        counts = torch.zeros(E, dtype=torch.int32, device="cuda")
        active = [0, 2, 3, 9, 10, 14, 15]
        counts[active] = 1
        src = torch.empty(E, dtype=torch.int32, device="cuda")
        act = torch.empty(E, dtype=torch.int32, device="cuda")
        n_act = torch.empty(2, dtype=torch.int32, device="cuda")
        miss = torch.empty(E, dtype=torch.int32, device="cuda")
        n_miss = torch.empty(1, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.expcache_lookup(cache.handle, 1, counts.data_ptr(), src.data_ptr(), act.data_ptr(),
                            n_act.data_ptr(), miss.data_ptr(), n_miss.data_ptr(), st.data_ptr(), s)
        torch.cuda.synchronize()
        hits, misses = [2, 9, 14], [0, 3, 10, 15]
        assert n_act.cpu().tolist() == [7, 3] and n_miss.item() == 4
        assert act[:7].cpu().tolist() == hits + misses
        assert miss[:4].cpu().tolist() == misses
        srcs = src.cpu().numpy()
        assert srcs[2] == 2 and srcs[9] == 3 and srcs[14] == 5
        assert [srcs[e] for e in misses] == [6, 7, 8, 6]
        assert all(srcs[e] == -1 for e in range(E) if e not in active)
        # group 0 gathers misses 0..2, group 1 miss 3
        for g in range(2):
            moe.expcache_fill(cache.handle, 1, miss.data_ptr(), n_miss.data_ptr(), 3 * g, 3, 0,
                              st.data_ptr(), s)
            torch.cuda.synchronize()
            from routed_expert_layer_router_gb300.layer import device_view
            for i in range(3 * g, min(3 * g + 3, 4)):
                got = device_view(cache.slot_ptr(6 + i % 3), (rb,), torch.uint8).cpu().numpy()
                assert np.array_equal(got, host_recs[misses[i]])
        assert st.item() == 0
        # a fill into cache slots marks them resident
        ids = torch.tensor([3], dtype=torch.int32, device="cuda")
        one = torch.tensor([1], dtype=torch.int32, device="cuda")
        dst = torch.tensor([5], dtype=torch.int32, device="cuda")
        moe.expcache_fill(cache.handle, 1, ids.data_ptr(), one.data_ptr(), 0, 1, dst.data_ptr(),
                          st.data_ptr(), s)
        tab = cache.table().cpu().numpy()
        assert tab[1, 3] == 5 and tab[0].max() == -1
        # a slot outside layer 0's partition is refused on the device
        moe.expcache_fill(cache.handle, 0, ids.data_ptr(), one.data_ptr(), 0, 1, dst.data_ptr(),
                          st.data_ptr(), s)
        torch.cuda.synchronize()
        assert st.item() == moe.MOE_ERR_DEVICE
    finally:
        cache.close()
        arena.close()
