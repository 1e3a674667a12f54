"""Pins of the oracle's number formats against the format definitions and an
independent library (torch's float8_e4m3fn / bfloat16 conversions)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _same(a, b):
    if math.isnan(b):
        return math.isnan(a)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


def test_e2m1_all_codes_match_spec_table():
    for code, val in _rows("e2m1_values.txt"):
        assert _same(oracle.e2m1(int(code)), float(val)), code


def test_e4m3_landmarks_match_spec():
    for code, val in _rows("e4m3_landmarks.txt"):
        assert _same(oracle.e4m3(int(code, 16)), float(val)), code


def test_e4m3_all_256_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    for b in range(256):
        assert _same(oracle.e4m3(b), ref[b]), hex(b)


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, 4096, dtype=np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # finite only
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64)
    got = np.array([oracle.bf16(int(b)) for b in bits])
    assert np.array_equal(got, ref.numpy())


def test_e4m3_rne_matches_torch_on_grid_midpoints_and_random():
    vals = []
    pos = [oracle.e4m3(b) for b in range(0x7F)]
    for a, b in zip(pos[:-1], pos[1:]):
        vals += [a, b, (a + b) / 2, a + (b - a) * 0.3, a + (b - a) * 0.7]
    rng = np.random.default_rng(1)
    vals += list(rng.uniform(0, 448, 2000)) + list(np.exp(rng.uniform(-12, 6, 2000)))
    v32 = np.array(vals, np.float32)
    v32 = v32[v32 <= 448]
    ref = torch.from_numpy(v32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_rne(float(t)) for t in v32], np.uint8)
    assert np.array_equal(got, ref)
    assert oracle.e4m3_rne(1000.0) == 0x7E  # saturates


@pytest.mark.parametrize("q,code", [
    (0.0, 0), (0.25, 0), (0.2500001, 1), (0.75, 2), (0.7499999, 1), (1.25, 2), (1.75, 4),
    (2.5, 4), (2.5000002, 5), (3.5, 6), (5.0, 6), (5.0000005, 7), (6.0, 7), (100.0, 7),
    (-0.5, 9), (-6.5, 15), (-0.1, 8), (-0.0, 8)])
def test_e2m1_rne_sat_closed_forms(q, code):
    assert oracle.e2m1_rne_sat(q) == code


def _dequant_row(codes, scales, G):
    n = 2 * len(codes)
    out = np.empty(n)
    for i in range(n):
        c = (codes[i // 2] >> 4) if i & 1 else (codes[i // 2] & 15)
        out[i] = oracle.e2m1(int(c)) * oracle.e4m3(int(scales[i // 16])) * G
    return out


def test_nvfp4_quant_global_scale_and_error_bound():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(256).astype(np.float32) * 3.0
    codes, scales, G = oracle.nvfp4_quant(v)
    amax = np.abs(v).max()
    assert G == np.float32(amax) / np.float32(2688.0)
    deq = _dequant_row(codes, scales, G)
    for b in range(16):
        blk = v[b * 16:(b + 1) * 16].astype(np.float64)
        s = oracle.e4m3(int(scales[b])) * G
        # every value lands within half of the largest E2M1 step (1.0) times the
        # scale, plus saturation at 6 s when the scale rounded down
        err = np.abs(deq[b * 16:(b + 1) * 16] - blk)
        assert np.all(err <= 1.0 * s + 1e-12 + np.maximum(0, np.abs(blk) - 6 * s))
        # the block scale is the E4M3 rounding of amax_b / (6 G)
        t = np.float32(np.abs(blk).max()) / np.float32(np.float32(6.0) * np.float32(G))
        assert scales[b] == oracle.e4m3_rne(float(t))


def test_nvfp4_quant_of_exact_values_is_exact():
    # values already on the grid (codes x E4M3 scale x G) survive the round
    # trip; the row amax is 2688 * 2^-10 so that G = 2^-10 exactly, and the
    # block scales come out as 56, 112, 224, 448 (exact E4M3 values)
    rng = np.random.default_rng(3)
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    v = np.empty(64)
    for b in range(4):
        blk = rng.choice(mags, 16) * rng.choice([-1, 1], 16)
        blk[rng.integers(16)] = 6.0  # each block reaches its amax code
        v[b * 16:(b + 1) * 16] = blk * 2.0 ** (b - 2) * (7.0 / 32.0)
    v32 = v.astype(np.float32)
    codes, scales, G = oracle.nvfp4_quant(v32)
    assert np.array_equal(_dequant_row(codes, scales, G), v32.astype(np.float64))


def test_nvfp4_quant_zero_row():
    codes, scales, G = oracle.nvfp4_quant(np.zeros(32, np.float32))
    assert G == 1.0 and not codes.any() and not scales.any()


def _blocks_sg(v):
    """Per element: the dequantised block scale s*G of v's NVFP4 quantisation."""
    codes, scales, G = oracle.nvfp4_quant(v)
    return np.repeat([oracle.e4m3(int(b)) * G for b in scales], 16)


def test_quant_flip_slack_covers_nearby_inputs():
    """The NVFP4 rounding-boundary slack covers every change of the quantised
    value that moving each element by up to half the code margin (in units of
    its block scale) can cause; the row amax element is left alone, so G does
    not move, and the block scales move by far less than their margin."""
    rng = np.random.default_rng(9)
    hits = 0
    for trial in range(200):
        v = (rng.standard_normal(256) * rng.uniform(0.1, 10)).astype(np.float32)
        amax_i = int(np.argmax(np.abs(v)))
        codes, scales, G = oracle.nvfp4_quant(v)
        base = _dequant_row(codes, scales, G)
        delta = oracle.quant_flip_delta(v)
        sg = _blocks_sg(v)
        # plant elements right next to E2M1 midpoints so that flips do happen
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
        for i in rng.choice(256, 24, replace=False):
            if i != amax_i and abs(v[i]) < np.abs(v[(i // 16) * 16:(i // 16 + 1) * 16]).max():
                q = rng.choice(mids) + rng.uniform(-0.3, 0.3) * oracle.FLIP_Q
                v[i] = np.float32(np.sign(v[i]) * q * sg[i])
        codes, scales, G = oracle.nvfp4_quant(v)
        base = _dequant_row(codes, scales, G)
        delta = oracle.quant_flip_delta(v)
        sg = _blocks_sg(v)
        for sign in (1.0, -1.0):
            vp = v.astype(np.float64) + sign * 0.5 * oracle.FLIP_Q * sg * np.sign(v)
            vp[amax_i] = v[amax_i]
            vp = vp.astype(np.float32)
            c2, s2, G2 = oracle.nvfp4_quant(vp)
            assert G2 == G
            moved = np.abs(_dequant_row(c2, s2, G2) - base)
            assert np.all(moved <= delta + 1e-12)
            hits += int((moved > 0).sum())
    assert hits > 100  # the planted elements did flip
    # an element exactly on an E2M1 midpoint (1.25 of its block scale) is
    # flagged with one code step; one at twice the margin from it is not
    v = np.zeros(16, np.float32)
    v[0] = 6.0
    v[1] = 1.25
    v[2] = 1.25 + 2 * oracle.FLIP_Q
    d = oracle.quant_flip_delta(v)
    codes, scales, G = oracle.nvfp4_quant(v)
    s = oracle.e4m3(int(scales[0])) * G
    assert d[1] == pytest.approx(0.5 * s) and d[2] == 0.0 and d[3] == 0.0


def test_quant_flip_slack_of_block_scales():
    """A block whose scale argument amax_b/(6G) sits on an E4M3 midpoint is
    flagged on every element with 4 x the upper scale x G, and that covers the
    requantisation under either neighbouring scale; a block whose argument is
    clear of every midpoint carries no scale slack."""
    rng = np.random.default_rng(21)
    checked = 0
    for c in range(9, 0x7E):  # normal E4M3 scales
        s1, s2 = oracle.e4m3(c - 1), oracle.e4m3(c)
        v = np.zeros(32, np.float32)
        v[16] = 2688.0  # row amax: G = 1 exactly
        v[17:32] = rng.uniform(-2688, 2688, 15)
        blk = rng.uniform(-1, 1, 16) * 3 * (s1 + s2)
        blk[0] = 3.0 * (s1 + s2)  # block amax on the midpoint: t = (s1 + s2) / 2
        v[:16] = blk
        if np.float32(v[0]) / np.float32(6.0) != np.float32(0.5 * (s1 + s2)):
            continue  # midpoint not representable at this magnitude
        d = oracle.quant_flip_delta(v)
        assert np.all(d[:16] == 4 * s2), (c, d[:16])
        # requantise the block under each neighbouring scale (nudging its max)
        base = _dequant_row(*oracle.nvfp4_quant(v))
        for nudge in (1 - 1e-6, 1 + 1e-6):
            vp = v.copy()
            vp[0] = np.float32(v[0] * nudge)
            moved = np.abs(_dequant_row(*oracle.nvfp4_quant(vp)) - base)
            assert np.all(moved[:16] <= d[:16])
        checked += 1
        # clear of the midpoint by 10x the margin: no scale slack in the block
        vq = v.copy()
        vq[0] = np.float32(v[0] * (1 + 10 * oracle.FLIP_T))
        assert np.all(oracle.quant_flip_delta(vq)[:16] != 4 * s2)
    assert checked > 60


def test_bf16_flip_slack_pins():
    """The bf16 rounding-boundary slack (the shared expert's h before its
    bf16 down GEMM): one bf16 step exactly where a value sits within relative
    FLIP_BF16 of a round-to-nearest-even midpoint, zero elsewhere.  Checked against
    numpy's RNE rounding of perturbed values and against midpoints built bit
    by bit."""
    from tests.helpers import bf16_to_f64, f32_to_bf16
    rng = np.random.default_rng(11)
    v = rng.standard_normal(50000) * 10.0 ** rng.uniform(-4, 4, 50000)
    d = oracle.bf16_flip_delta(v)

    def rne(a):
        return bf16_to_f64(f32_to_bf16(np.asarray(a, np.float64).astype(np.float32)))

    base = rne(v)
    # every change of the bf16 value that a relative perturbation of 5e-5 can
    # cause is covered, and is exactly one bf16 step
    for rel in (0.5 * oracle.FLIP_BF16, -0.5 * oracle.FLIP_BF16):
        moved = np.abs(rne(v * (1 + rel)) - base)
        assert np.all(moved <= d)
        flipped = moved > 0
        assert np.all(d[flipped] == moved[flipped])
    # values further than twice the margin from every midpoint carry no slack
    m = 2 * oracle.FLIP_BF16
    far = np.abs(rne(v * (1 + m)) - rne(v * (1 - m))) == 0
    assert far.sum() > 45000 and not d[far].any()
    # exact midpoints between two adjacent bf16 values (both signs, across
    # binades): flagged with the distance between the two
    bits = rng.integers(0x0080, 0x7F7F, 2000).astype(np.uint16)
    bits[:4] = [0x3F7F, 0x3F80, 0x0080, 0x7F7E]  # mantissa carry, 1.0, smallest normal, near max
    lo = bf16_to_f64(bits)
    hi = bf16_to_f64(bits + 1)
    mid = 0.5 * (lo + hi)
    for sgn in (1.0, -1.0):
        assert np.array_equal(oracle.bf16_flip_delta(sgn * mid), hi - lo)
        # a quarter step either side of the midpoint, and the grid values themselves
        assert not oracle.bf16_flip_delta(sgn * (0.75 * lo + 0.25 * hi)).any()
        assert not oracle.bf16_flip_delta(sgn * (0.25 * lo + 0.75 * hi)).any()
        assert not oracle.bf16_flip_delta(sgn * lo).any()
