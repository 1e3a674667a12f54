"""Pins of the seeded input generator (host side) and of the oracle's record
decode against the generator's pre-quantisation values."""
import os

import numpy as np

import gen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_splitmix64_published_vector():
    x = 0
    for (want,) in _golden("splitmix64.txt"):
        x = (x + gen.GOLDEN) & 0xFFFFFFFFFFFFFFFF
        assert gen.mix64(x) == int(want, 16)


def test_record_sizes_golden():
    for H, I, n in _golden("record_sizes.txt"):
        assert gen.record_bytes(int(H), int(I)) == int(n)
        assert gen._lib_host().gen_record_size(int(H), int(I), gen.NVFP4) == int(n)
        # MXFP4: the same codes, one E8M0 byte per 32 values instead of an E4M3 per 16
        mx = int(n) - 3 * int(H) * int(I) // 32
        assert gen.record_bytes(int(H), int(I), gen.MXFP4) == mx
        assert gen._lib_host().gen_record_size(int(H), int(I), gen.MXFP4) == mx


def test_activation_and_router_moments():
    x = gen.x_bf16(7, 0, 0, 64, 6144)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(xf.mean()) < 0.01 and abs(xf.std() - 1.0) < 0.01
    assert np.abs(xf).max() <= 3.47
    w = gen.router_f32(7, 0, 32, 6144).astype(np.float64)
    assert abs(w.std() - 0.05) < 0.001
    # different draws and layers differ; same draw repeats
    assert not np.array_equal(gen.x_bf16(7, 0, 0, 1, 64), gen.x_bf16(7, 0, 1, 1, 64))
    assert not np.array_equal(gen.x_bf16(7, 0, 0, 1, 64), gen.x_bf16(7, 1, 0, 1, 64))
    assert np.array_equal(gen.x_bf16(7, 0, 3, 1, 64), gen.x_bf16(7, 0, 0, 4, 64)[3:4])


def _half_step(mag):
    # half the distance to the neighbouring E2M1 magnitudes
    return np.where(mag <= 2.0, 0.25, np.where(mag <= 4.0, 0.5, 1.0))


def test_oracle_decode_reproduces_prequant_weights():
    """Every represented weight e2m1 * e4m3 * g sits within half a code step of
    the generator's pre-quantisation weight d * g / 64 (the generator writes
    the record, the oracle reads it; they were written independently)."""
    H, I = 512, 256
    rec = gen.expert_records(11, 2, [5], H, I)[0]
    g = gen.global_scales(11, 2, 8)[5]
    for m, rows in ((0, [0, 1, 31, 32, 127, 128, 255]), (1, [3, 200]), (2, [0, 77, 128, 511])):
        W = oracle.dequant_matrix(rec, H, I, m, g)
        for r in rows:
            d = gen.expert_prequant_row(11, 2, 5, H, I, m, r).astype(np.float64)
            target = d * g[m] / 64.0
            K = W.shape[1]
            for kb in range(K // 16):
                blk = slice(16 * kb, 16 * kb + 16)
                # the block scale (in weight units) lies in [amax/6, 1.125 amax/6]
                # (smallest E4M3 value not below amax/6; E4M3 normals are spaced
                # at most 1/8 apart); the code is the nearest E2M1 magnitude
                amax = np.abs(target[blk]).max()
                s_lo, s_hi = amax / 6.0, 1.125 * amax / 6.0
                mag = np.minimum(np.abs(target[blk]) / s_lo, 6.0)
                err = np.abs(W[r, blk] - target[blk])
                assert np.all(err <= _half_step(mag) * s_hi * (1 + 1e-9)), (m, r, kb)


def test_weight_statistics():
    rec = gen.expert_records(12, 0, [0], 1024, 512)[0]
    g = gen.global_scales(12, 0, 1)[0]
    W = oracle.dequant_matrix(rec, 1024, 512, 0, g)
    # N(0, (0.02 f)^2) before quantisation, f in [0.875, 1.125)
    assert 0.017 < W.std() < 0.023


def test_zipf_bias_is_a_permutation():
    b, rank = gen.zipf_bias(2, 3, 288, 1.55)
    assert sorted(rank.tolist()) == list(range(1, 289))
    assert np.allclose(b, -1.55 * np.log(rank), rtol=1e-6, atol=1e-6)
    b2, rank2 = gen.zipf_bias(2, 4, 288, 1.55)
    assert not np.array_equal(rank, rank2)
