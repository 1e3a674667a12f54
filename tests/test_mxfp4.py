"""Pins of the oracle's MXFP4 format (windlass README: GLM-5.2 runs in MXFP4;
its correctness list names "MXFP4 dequant, 8 seeds x 2 shapes" and a flipped
MXFP4 nibble order as a negative control).  Definitions from OCP
Microscaling Formats (MX) v1.0: E2M1 elements, blocks of 32, one E8M0 scale
per block (2^(b - 127), 0xFF NaN); the conversion takes the shared exponent
floor(log2 max|v|) - 2 and rounds each v / 2^X to E2M1, ties to even,
saturating at 6."""
import numpy as np
import pytest
import torch

import gen
import oracle


def _e2m1(c):
    return oracle.e2m1(int(c))


def test_e8m0_all_256_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    got = np.array([oracle.e8m0(b) for b in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def _dequant_mx(codes, scales):
    c = np.stack([codes & 15, codes >> 4], 1).ravel()
    return np.array([_e2m1(v) for v in c]) * np.repeat([oracle.e8m0(int(b)) for b in scales], 32)


def test_mxfp4_quant_hand_worked_blocks():
    v = np.zeros(96, np.float32)
    # block 0: max 6.0 -> floor(log2 6) = 2, X = 0 (byte 127); 0.3 -> 0.5,
    # 0.25 -> 0 (tie, even), 0.75 -> 1.0 (tie, even code 2), -2.6 -> -3, 5.0 -> 4 (tie)
    v[0:6] = [6.0, 0.3, 0.25, 0.75, -2.6, 5.0]
    # block 1: max 7.0 -> X = 0 as well: 7 saturates to 6 (the MX rule's clamp)
    v[32:34] = [7.0, 1.0]
    # block 2: max exactly 2^-3 -> X = -5, q = 4 for the max; 2^-6 -> q = 0.5
    v[64:66] = [0.125, -0.015625]
    codes, scales = oracle.mxfp4_quant(v)
    assert scales.tolist() == [127, 127, 122]
    deq = _dequant_mx(codes, scales)
    assert deq[0:6].tolist() == [6.0, 0.5, 0.0, 1.0, -3.0, 4.0]
    assert deq[32:34].tolist() == [6.0, 1.0]
    assert deq[64:66].tolist() == [0.125, -0.015625]
    assert not deq[6:32].any() and not deq[34:64].any() and not deq[66:].any()


def _nearest_code(q):
    """E2M1 code (magnitude index 0..7 and sign bit) nearest q, ties to the
    even code, saturating at 6 - written from the definition with numpy."""
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    a = np.abs(q)
    dist = np.abs(a[:, None] - mags[None, :])
    best = dist.min(1, keepdims=True)
    cand = dist == best
    # of the nearest magnitudes take the even index (ties), else the only one
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    idx = np.where(even.any(1), even.argmax(1), cand.argmax(1))
    idx = np.where(a > 6, 7, idx)
    return idx | np.where(np.signbit(q), 8, 0)


def test_mxfp4_quant_matches_its_definition_on_random_rows():
    """For random rows over many magnitudes: each block's scale byte is 127 +
    floor(log2 amax) - 2 and each code is the E2M1 code nearest v / 2^X
    (ties to even, saturating at 6, sign from v); grid values survive
    exactly; an all-zero block gets byte 0 and codes 0."""
    rng = np.random.default_rng(5)
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    for trial in range(60):
        v = (rng.standard_normal(256) * 10.0 ** rng.uniform(-6, 6)).astype(np.float32)
        if trial % 5 == 0:
            b0 = int(rng.integers(8))
            v[32 * b0:32 * b0 + 32] = 0.0
        codes, scales = oracle.mxfp4_quant(v)
        c = np.stack([codes & 15, codes >> 4], 1).ravel()
        for b in range(8):
            blk = v[32 * b:32 * b + 32].astype(np.float64)
            amax = np.abs(blk).max()
            if amax == 0:
                assert scales[b] == 0 and not c[32 * b:32 * b + 32].any()
                continue
            X = int(np.floor(np.log2(amax))) - 2
            assert scales[b] == 127 + X
            assert np.array_equal(c[32 * b:32 * b + 32], _nearest_code(blk / 2.0 ** X))
    # exact grid values survive
    X = -3
    blk = rng.choice(mags, 32) * rng.choice([-1, 1], 32) * 2.0 ** X
    blk[0] = 6.0 * 2.0 ** X
    codes, scales = oracle.mxfp4_quant(blk.astype(np.float32))
    assert np.array_equal(_dequant_mx(codes, scales), blk)


@pytest.mark.parametrize("shape", [(512, 256), (1024, 512)])
@pytest.mark.parametrize("seed", range(8))
def test_mx_record_decode_reproduces_prequant_weights(seed, shape):
    """MXFP4 records from the generator, decoded by the oracle: every weight is
    the E2M1 value nearest the pre-quantisation weight d g / 64 in units of
    its block's E8M0 scale 2^(floor(log2 max|d g / 64|) - 2) (saturating at
    6), times that scale.  8 seeds x 2 shapes."""
    H, I = shape
    rec = gen.expert_records(seed, 1, [3], H, I, fmt=gen.MXFP4)[0]
    assert rec.size == gen.record_bytes(H, I, gen.MXFP4)
    g = gen.global_scales(seed, 1, 4)[3]
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    for m, rows in ((0, [0, 31, 127, 128]), (1, [5, I - 1]), (2, [0, 129, H - 1])):
        W = oracle.dequant_matrix(rec, H, I, m, g, fmt=oracle.MXFP4)
        for r in rows:
            d = gen.expert_prequant_row(seed, 1, 3, H, I, m, r).astype(np.float64)
            for kb in range(W.shape[1] // 32):
                blk = d[32 * kb:32 * kb + 32] / 64.0  # weight / g
                amax = np.abs(blk).max()
                X = int(np.floor(np.log2(amax))) - 2
                code = _nearest_code(blk / 2.0 ** X)
                want = np.where(code & 8, -1.0, 1.0) * mags[code & 7] * 2.0 ** X * g[m]
                got = W[r, 32 * kb:32 * kb + 32]
                assert np.array_equal(got, want), (m, r, kb)


def test_mx_flip_slack_covers_nearby_inputs():
    """The MXFP4 rounding-boundary slack covers every change of the quantised
    value that moving elements by up to half the code margin causes, and a
    block whose max sits on a power of two is flagged on every element."""
    rng = np.random.default_rng(23)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    hits = 0
    for trial in range(200):
        v = (rng.standard_normal(256) * rng.uniform(0.01, 100)).astype(np.float32)
        codes, scales = oracle.mxfp4_quant(v)
        sx = np.repeat([oracle.e8m0(int(b)) for b in scales], 32)
        amax_i = [32 * b + int(np.argmax(np.abs(v[32 * b:32 * b + 32]))) for b in range(8)]
        for i in rng.choice(256, 24, replace=False):
            if i not in amax_i:
                v[i] = np.float32(np.sign(v[i]) * (rng.choice(mids) + rng.uniform(-.3, .3) *
                                                   oracle.FLIP_Q) * sx[i])
        codes, scales = oracle.mxfp4_quant(v)
        base = _dequant_mx(codes, scales)
        delta = oracle.quant_flip_delta(v, fmt=oracle.MXFP4)
        for sign in (1.0, -1.0):
            vp = v.astype(np.float64) + sign * 0.5 * oracle.FLIP_Q * sx * np.sign(v)
            vp[amax_i] = v[amax_i]
            c2, s2 = oracle.mxfp4_quant(vp.astype(np.float32))
            moved = np.abs(_dequant_mx(c2, s2) - base)
            assert np.all(moved <= delta + 1e-30)
            hits += int((moved > 0).sum())
    assert hits > 100
    # a block max just below 2^3: the shared exponent may be 0 or 1
    v = np.zeros(32, np.float32)
    v[0] = np.float32(8.0 * (1 - 1e-7))
    v[1:] = rng.uniform(-5, 5, 31)
    d = oracle.quant_flip_delta(v, fmt=oracle.MXFP4)
    assert np.all(d == 2.0 * 2.0 ** 1)
    base = _dequant_mx(*oracle.mxfp4_quant(v))
    v2 = v.copy()
    v2[0] = np.float32(8.0)
    assert np.all(np.abs(_dequant_mx(*oracle.mxfp4_quant(v2)) - base) <= d)


def test_mx_nibble_order_negative_control():
    """A flipped MXFP4 nibble order in the decoder changes an expert's output
    by far more than the parity tolerance."""
    H, I = 512, 256
    rec = gen.expert_records(3, 0, [1], H, I, fmt=gen.MXFP4)[0]
    g = gen.global_scales(3, 0, 2)[1]
    x = (gen.x_bf16(3, 0, 0, 1, H)[0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    o = oracle.expert(rec, H, I, g, x, fmt=oracle.MXFP4)
    try:
        oracle.lib().oracle_set_defect(1)  # nibble swap
        o_bad = oracle.expert(rec, H, I, g, x, fmt=oracle.MXFP4)
    finally:
        oracle.lib().oracle_set_defect(0)
    rms = np.sqrt(np.mean(o ** 2))
    assert np.abs(o_bad - o).max() > 100 * 2e-2 * rms


@pytest.mark.parametrize("act_quant", [False, True])
def test_mx_identity_expert_returns_its_input(act_quant):
    """The bit-built MXFP4 identity expert maps x to y[16+i] = x[16+i] exactly,
    in the decode numerics and in the prefill numerics (MXFP4 activations)."""
    from tests.helpers import bf16_to_f64, identity_record_mx, mxfp4_exact_x
    H, I = 512, 256
    rec = identity_record_mx(H, I)
    for xv in bf16_to_f64(mxfp4_exact_x(H, 4, seed=3)):
        o = oracle.expert(rec, H, I, np.ones(3, np.float32), xv, act_quant=act_quant,
                          fmt=oracle.MXFP4)
        assert np.array_equal(o[16:16 + I], xv[16:16 + I])
        assert not o[:16].any() and not o[16 + I:].any()
