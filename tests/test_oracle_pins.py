"""Pins of the CPU oracle against what mathematics and independent libraries
fix: invariants of the router, a library stable sort for the permutation,
brute-force numpy matmuls for the expert FFN, a bit-constructed identity
expert whose output equals its input exactly, the combine rule, and negative
controls that must fail the parity gate by a wide margin."""
import numpy as np
import pytest
import scipy.special
import torch

import gen
import oracle
from tests.helpers import identity_record, identity_x, nvfp4_exact_x, TOL


def _bf16_to_f64(x):
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.fixture(scope="module")
def tiny():
    wl = gen.WORKLOADS["tiny"]
    x = gen.x_bf16(wl.seed, 0, 0, 16, wl.H)
    Wr = gen.router_f32(wl.seed, 0, wl.E, wl.H)
    return wl, x, Wr


def test_router_logits_match_numpy(tiny):
    wl, x, Wr = tiny
    bias = np.linspace(-1, 1, wl.E).astype(np.float32)
    ids, w, p, logits, gap = oracle.route(x, Wr, bias, wl.k)
    ref = _bf16_to_f64(x) @ Wr.astype(np.float64).T + bias.astype(np.float64)
    assert np.allclose(logits, ref, rtol=1e-12, atol=1e-12)


def test_router_selection_weights_invariants(tiny):
    wl, x, Wr = tiny
    ids, w, p, logits, gap = oracle.route(x, Wr, None, wl.k)
    T = x.shape[0]
    for t in range(T):
        order = np.lexsort((np.arange(wl.E), -logits[t]))  # (logit desc, id asc)
        assert ids[t].tolist() == order[:wl.k].tolist()
        assert len(set(ids[t].tolist())) == wl.k
        sm = scipy.special.softmax(logits[t])
        assert np.allclose(p[t], sm[ids[t]], rtol=1e-12)
        assert abs(w[t].sum() - 1.0) < 1e-12
        l = logits[t][ids[t]]
        assert np.allclose(w[t][0] / w[t][1:], np.exp(l[0] - l[1:]), rtol=1e-12)
        srt = np.sort(logits[t])[::-1]
        assert gap[t] == pytest.approx(np.min(srt[:wl.k] - srt[1:wl.k + 1]), rel=1e-12)
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    assert counts.sum() == T * wl.k


def test_router_ties_go_to_lower_id():
    H, E, k = 32, 6, 2
    Wr = np.zeros((E, H), np.float32)
    Wr[1, 0] = Wr[4, 0] = 1.0  # experts 1 and 4 tie, both above the rest
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80  # 1.0
    ids, w, p, logits, gap = oracle.route(x, Wr, None, k)
    assert ids[0].tolist() == [1, 4] and gap[0] == 0.0
    Wr[4, 0] = 1.0
    Wr[1, 0] = 0.5
    ids, *_ = oracle.route(x, Wr, None, 1)
    assert ids[0].tolist() == [4]


def test_permute_equals_library_stable_sort():
    rng = np.random.default_rng(5)
    for T, k, E in ((1, 8, 288), (4, 2, 16), (64, 8, 288), (513, 8, 32)):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        counts, offsets, perm, inv = oracle.permute(ids, E)
        assert np.array_equal(perm, np.argsort(ids.ravel(), kind="stable"))
        assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        assert np.array_equal(inv[perm], np.arange(T * k))
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 16]], np.int32), 16)


def test_expert_matches_bruteforce_numpy():
    H, I = 256, 128
    rec = gen.expert_records(21, 0, [3], H, I)[0]
    g = gen.global_scales(21, 0, 4)[3]
    x = _bf16_to_f64(gen.x_bf16(21, 0, 0, 1, H))[0]
    Wg, Wu, Wd = (oracle.dequant_matrix(rec, H, I, m, g) for m in range(3))
    gg, uu = Wg @ x, Wu @ x
    h = gg * scipy.special.expit(gg) * uu
    ref = Wd @ h
    got = oracle.expert(rec, H, I, g, x)
    assert np.allclose(got, ref, rtol=1e-11, atol=1e-13)


def test_shared_expert_matches_numpy():
    H, Is = 256, 128
    sg, su, sd = gen.shared_bf16(22, 0, Is, H)
    x = _bf16_to_f64(gen.x_bf16(22, 0, 0, 1, H))[0]

    def f(a):
        return torch.from_numpy(a.astype(np.int16)).view(torch.bfloat16).double().numpy()

    gg, uu = f(sg) @ x, f(su) @ x
    h = gg * scipy.special.expit(gg) * uu
    ref = f(sd) @ h
    assert np.allclose(oracle.shared(sg, su, sd, x), ref, rtol=1e-11, atol=1e-14)
    hb = torch.from_numpy(h).float().bfloat16().double().numpy()
    assert np.allclose(oracle.shared(sg, su, sd, x, round_h_bf16=True), f(sd) @ hb,
                       rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("mode", [0, 1])
def test_identity_expert_returns_its_input(mode):
    H, I, E, k = 256, 128, 4, 2
    rec = identity_record(H, I)
    g = np.ones((E, 3), np.float32)
    Wr = gen.router_f32(23, 0, E, H)
    x = identity_x(H, 3, seed=23) if mode == 0 else nvfp4_exact_x(H, 3, seed=23)
    y, ids, w, p = oracle.layer_forward(x, H, I, E, k, Wr, None, [rec] * E, g, mode=mode)
    xf = _bf16_to_f64(x)
    want = np.zeros_like(xf)
    want[:, 16:16 + I] = xf[:, 16:16 + I]
    assert np.allclose(y, want, rtol=1e-14, atol=0)


def test_combine_of_identical_experts_is_that_expert():
    H, I, E, k, Is = 256, 128, 8, 3, 128
    rec = gen.expert_records(24, 0, [0], H, I)[0]
    g = np.tile(gen.global_scales(24, 0, 1), (E, 1))
    Wr = gen.router_f32(24, 0, E, H)
    sh = gen.shared_bf16(24, 0, Is, H)
    x = gen.x_bf16(24, 0, 0, 2, H)
    y, *_ = oracle.layer_forward(x, H, I, E, k, Wr, None, [rec] * E, g, shared_w=sh)
    for t in range(2):
        xf = _bf16_to_f64(x[t:t + 1])[0]
        ref = oracle.expert(rec, H, I, g[0], xf) + oracle.shared(*sh, xf)
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-15)


def test_layer_is_independent_of_where_records_live():
    wl = gen.WORKLOADS["tiny"]
    recs = gen.expert_records(wl.seed, 0, range(wl.E), wl.H, wl.I)
    g = gen.global_scales(wl.seed, 0, wl.E)
    Wr = gen.router_f32(wl.seed, 0, wl.E, wl.H)
    x = gen.x_bf16(wl.seed, 0, 0, wl.T, wl.H)
    y1, *_ = oracle.layer_forward(x, wl.H, wl.I, wl.E, wl.k, Wr, None, list(recs), g)
    copies = {e: recs[e].copy() for e in range(wl.E)}
    y2, *_ = oracle.layer_forward(x, wl.H, wl.I, wl.E, wl.k, Wr, None, copies, g)
    assert np.array_equal(y1, y2)


@pytest.mark.parametrize("defect", ["nibble_swap", "scale_ue8m0", "block_off_by_one",
                                    "scaling_2_5"])
def test_negative_controls_fail_the_parity_gate(defect):
    wl = gen.WORKLOADS["tiny"]
    recs = gen.expert_records(wl.seed, 0, range(wl.E), wl.H, wl.I)
    g = gen.global_scales(wl.seed, 0, wl.E)
    Wr = gen.router_f32(wl.seed, 0, wl.E, wl.H)
    x = gen.x_bf16(wl.seed, 0, 0, wl.T, wl.H)
    y, *_ = oracle.layer_forward(x, wl.H, wl.I, wl.E, wl.k, Wr, None, list(recs), g)
    with oracle.defect(defect):
        yd, *_ = oracle.layer_forward(x, wl.H, wl.I, wl.E, wl.k, Wr, None, list(recs), g)
    tol = TOL * np.sqrt(np.mean(y ** 2))
    assert np.abs(yd - y).max() > 5 * tol


def test_negative_control_tie_rule():
    H, E, k = 32, 6, 2
    Wr = np.zeros((E, H), np.float32)
    Wr[1, 0] = Wr[4, 0] = 1.0
    Wr[2, 0] = 2.0
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80
    ids, *_ = oracle.route(x, Wr, None, k)
    with oracle.defect("tie_high_id"):
        ids_d, *_ = oracle.route(x, Wr, None, k)
    assert ids[0].tolist() == [2, 1] and ids_d[0].tolist() == [2, 4]


def test_renorm_skip_drops_low_weight_misses_and_renormalises(tiny):
    """The renorm-skip step: only misses below tau drop, the kept weights sum
    to 1 and keep their ratios; tau = 0 (or every expert resident) changes
    nothing; with one route dropped the layer equals the kept experts' own
    outputs weighted by the renormalised weights (brute force)."""
    wl, x, Wr = tiny
    ids, w, p, logits, gap = oracle.route(x, Wr, None, wl.k)
    T, k = ids.shape
    resident = np.zeros(wl.E, bool)
    resident[::2] = True
    for tau in (0.0, 0.3, 0.45, 0.49):
        w_eff, keep = oracle.renorm_skip(ids, w, resident, tau)
        drop = (~resident[ids]) & (w < tau)
        assert np.array_equal(~keep, drop)
        assert np.allclose(w_eff.sum(1), 1.0, atol=1e-14)
        assert np.all(w_eff[~keep] == 0.0)
        for t in range(T):
            kk = keep[t]
            assert np.allclose(w_eff[t, kk], w[t, kk] / w[t, kk].sum(), rtol=1e-15)
    w_eff, keep = oracle.renorm_skip(ids, w, np.ones(wl.E, bool), 0.49)
    assert keep.all() and np.allclose(w_eff, w, rtol=1e-15)
    # layer level: records for every expert, one token whose lower route misses
    recs = gen.expert_records(wl.seed, 0, list(range(wl.E)), wl.H, wl.I)
    g = gen.global_scales(wl.seed, 0, wl.E)
    t = int(np.argmax(w[:, 1] < 0.45))
    assert w[t, 1] < 0.45
    xt = x[t:t + 1]
    res = np.ones(wl.E, bool)
    res[ids[t, 1]] = False
    y_skip = oracle.layer_forward(xt, wl.H, wl.I, wl.E, wl.k, Wr, None, recs, g,
                                  resident=res, tau=0.45)[0]
    xd = _bf16_to_f64(xt[0])
    o0 = oracle.expert(recs[ids[t, 0]], wl.H, wl.I, g[ids[t, 0]], xd)
    assert np.allclose(y_skip[0], o0, rtol=1e-12, atol=1e-12)  # the kept route alone, weight 1
    y_exact = oracle.layer_forward(xt, wl.H, wl.I, wl.E, wl.k, Wr, None, recs, g)[0]
    y_res = oracle.layer_forward(xt, wl.H, wl.I, wl.E, wl.k, Wr, None, recs, g,
                                 resident=np.ones(wl.E, bool), tau=0.45)[0]
    assert np.array_equal(y_exact, y_res)
