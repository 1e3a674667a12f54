"""The library's device slot planner (expcache_plan_slots) against the
oracle's greedy per-layer slot budget ("Project Maya" page, section "VRAM:
one partition per layer, sized by what the layer routes"): partition and
per-layer expert order identical, on hand-worked, tied, saturated and
random count matrices, including the stack workload's shape (16 layers x
288 experts, Zipf-skewed counts)."""
import numpy as np
import pytest
import torch

import gen
import oracle

pytestmark = pytest.mark.gpu


def _plan_gpu(counts, total, floor):
    from routed_expert_layer_router_gb300 import moe
    c = torch.from_numpy(np.ascontiguousarray(counts, np.uint32).view(np.int32)).cuda()
    L, E = counts.shape
    ls = torch.full((L + 1,), -7, dtype=torch.int32, device="cuda")
    order = torch.full((L, E), -7, dtype=torch.int32, device="cuda")
    moe.expcache_plan_slots(c.data_ptr(), L, E, total, floor, ls.data_ptr(), order.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return ls.cpu().numpy(), order.cpu().numpy()


def _cases():
    yield np.array([[8, 4, 2, 2], [10, 1, 1, 0]]), 5, 1
    yield np.array([[3, 3, 3, 3]] * 3), 7, 1
    yield np.array([[0, 0, 0], [5, 4, 1]]), 5, 1
    yield np.array([[1, 2], [3, 4]]), 10, 0
    rng = np.random.default_rng(3)
    for _ in range(40):
        L, E = int(rng.integers(1, 9)), int(rng.integers(1, 40))
        c = rng.integers(0, int(rng.choice([3, 50, 100000])), (L, E))
        floor = int(rng.integers(0, E + 1))
        yield c, int(rng.integers(L * floor, L * E + 5)), floor
    # the stack's shape: per-layer Zipf-skewed route counts of 512 tokens
    wl = gen.WORKLOADS["stack"]
    c = np.zeros((wl.layers, wl.E), np.int64)
    for l in range(wl.layers):
        _, rank = gen.zipf_bias(wl.seed, l, wl.E, wl.zipf_alpha)
        p = rank.astype(np.float64) ** -1.3 * (1 + 0.5 * (l % 3))
        c[l] = rng.multinomial(512 * wl.k, p / p.sum())
    yield c, wl.layers * wl.hot, 32


def test_device_planner_matches_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    for counts, total, floor in _cases():
        counts = np.asarray(counts, np.uint32)
        ref = oracle.slot_budget(counts, total, floor)
        got = _plan_gpu(counts, total, floor)
        assert np.array_equal(got[0], ref[0]), (counts, total, floor, got[0], ref[0])
        assert np.array_equal(got[1], ref[1])
