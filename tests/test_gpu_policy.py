"""GPU parity of the adaptive expert cache (expcache_set_policy /
expcache_policy_step through the C ABI) against the oracle's policy: after
every forward the slot table, the promoted slots, the decayed counts, the
latest-forward numbers, the event counter and the free slots are bit-exact;
and whole layers with the policy on give the oracle's outputs (the cache only
changes where the bytes come from)."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_common import (check_outputs, check_router, draw_tokens, host_inputs,
                              oracle_layer, to_dev_bf16, y_to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from routed_expert_layer_router_gb300 import moe
    moe.lib()
    gen._lib_cuda()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _compare_state(cache, ref):
    st = cache.policy_state()
    tab = cache.table().cpu().numpy()
    assert np.array_equal(tab, ref.table)
    assert np.array_equal(st["cnt"], ref.cnt)
    assert np.array_equal(st["last"], ref.last)
    assert np.array_equal(st["stamp"], ref.stamp)
    assert st["events"] == int(ref.events[0])
    assert np.array_equal(st["free"], ref.free)


@pytest.mark.parametrize("K", [0, 1, 3])
def test_policy_step_matches_oracle(K):
    from routed_expert_layer_router_gb300 import moe
    from routed_expert_layer_router_gb300.layer import ExpertCache
    L, E, per, n_stage = 3, 40, 10, 8
    ls = [0, per, 2 * per, 3 * per]
    cache = ExpertCache(L, E, 256, 128, n_cache_slots=3 * per, n_stage=n_stage, layer_slots=ls)
    try:
        table0 = -np.ones((L, E), np.int32)
        for l in range(L):
            for i in range(per - K):
                cache.set_resident(l, 3 * i + l, ls[l] + i)
                table0[l, 3 * i + l] = ls[l] + i
        cache.set_policy(K)
        ref = oracle.CachePolicy(L, E, 3 * per, ls, K, table0)
        _compare_state(cache, ref)
        dev = torch.device("cuda")
        src = torch.empty(E, dtype=torch.int32, device=dev)
        act = torch.empty(E, dtype=torch.int32, device=dev)
        n_act = torch.empty(2, dtype=torch.int32, device=dev)
        miss = torch.empty(E, dtype=torch.int32, device=dev)
        n_miss = torch.empty(1, dtype=torch.int32, device=dev)
        dst = torch.empty(E, dtype=torch.int32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        rng = np.random.default_rng(11 + K)
        for step in range(120):
            l = int(rng.integers(0, L))
            c = np.zeros(E, np.int32)
            ids = rng.choice(E, size=int(rng.integers(1, 9)), replace=False)
            c[ids] = rng.integers(1, 4, size=len(ids))
            if step % 40 == 39:
                c[ids[0]] = 12000  # crosses a halving
            counts = torch.from_numpy(c).to(dev)
            s = _stream()
            moe.expcache_lookup(cache.handle, l, counts.data_ptr(), src.data_ptr(), act.data_ptr(),
                                n_act.data_ptr(), miss.data_ptr(), n_miss.data_ptr(),
                                status.data_ptr(), s)
            moe.expcache_policy_step(cache.handle, l, counts.data_ptr(), src.data_ptr(),
                                     n_act.data_ptr(), miss.data_ptr(), n_miss.data_ptr(),
                                     dst.data_ptr(), 0, s)
            prom = ref.step(l, c)
            torch.cuda.synchronize()
            nm = int(n_miss.item())
            assert nm == len(prom)
            got = dst[:nm].cpu().numpy()
            srcs = src.cpu().numpy()
            for i, e in enumerate(miss[:nm].cpu().numpy()):
                if prom[i] >= 0:
                    assert got[i] == prom[i] and srcs[e] == prom[i]
                else:  # staged: the lookup's staging slot
                    assert got[i] == 3 * per + i % n_stage and srcs[e] == got[i]
            _compare_state(cache, ref)
        assert int(status.item()) == 0
    finally:
        cache.close()


@pytest.mark.parametrize("T", [4, 12])
def test_layer_forward_with_adaptive_cache(T):
    """Two tiny layers with 3 residents + 2 spares each; every forward's
    outputs match the oracle and the slot table follows the oracle's policy
    fed the oracle's routing.  4 tokens: the step runs in the router kernel;
    12: as a kernel of its own after the permutation."""
    import gen.device as gd
    wl = gen.WORKLOADS["tiny"]
    L, K = 2, 2
    resident = [[0, 5, 9], [1, 2, 3]]
    dw = gd.build(wl, layers=L, T_max=T, resident=resident, spares=K)
    try:
        cache = dw.cache
        table0 = cache.table().cpu().numpy()
        ref = oracle.CachePolicy(L, wl.E, cache.n_cache_slots,
                                 [0, 3 + K, 6 + 2 * K], K, table0)
        recs = {}
        promoted = 0
        for step in range(10):
            for l in range(L):
                Wr, bias, sh = host_inputs(dw, l)
                x, _ = draw_tokens(wl, l, T, Wr, bias, draw0=5000 + 97 * step)
                y = y_to_f64(dw.moe_layers[l].forward(to_dev_bf16(x)))
                torch.cuda.synchronize()
                y_ref, ids_r, w_r, p_r = oracle_layer(dw, l, x, record_cache=recs)
                check_router(dw.moe_layers[l].debug(T), ids_r, w_r, p_r)
                check_outputs(y, y_ref)
                c = np.bincount(ids_r.ravel(), minlength=wl.E).astype(np.int32)
                promoted += int((ref.step(l, c) >= 0).sum())
                assert np.array_equal(cache.table().cpu().numpy(), ref.table)
                assert dw.moe_layers[l].read_status() == 0
        assert promoted > 0
        st = cache.policy_state()
        assert np.array_equal(st["cnt"], ref.cnt) and np.array_equal(st["free"], ref.free)
    finally:
        dw.close()
