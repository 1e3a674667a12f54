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


def test_quant_flip_slack_covers_nearby_inputs():
    """The rounding-boundary slack is zero away from boundaries and covers
    every change of the quantised value that a relative perturbation of
    5e-5 of one element can cause (the row amax element is left alone, so G
    does not move)."""
    rng = np.random.default_rng(9)
    for trial in range(40):
        v = (rng.standard_normal(256) * rng.uniform(0.1, 10)).astype(np.float32)
        amax_i = int(np.argmax(np.abs(v)))
        codes, scales, G = oracle.nvfp4_quant(v)
        base = _dequant_row(codes, scales, G)
        delta = oracle.quant_flip_delta(v)
        for rel in (5e-5, -5e-5):
            vp = v.copy()
            mask = np.ones(256, bool)
            mask[amax_i] = False
            vp[mask] = (vp[mask].astype(np.float64) * (1 + rel)).astype(np.float32)
            c2, s2, G2 = oracle.nvfp4_quant(vp)
            assert G2 == G
            moved = np.abs(_dequant_row(c2, s2, G2) - base)
            assert np.all(moved <= delta + 1e-12)
    # an element exactly on an E2M1 midpoint (1.25 of its block scale) is flagged
    v = np.zeros(16, np.float32)
    v[0] = 6.0
    v[1] = 1.25
    d = oracle.quant_flip_delta(v)
    codes, scales, G = oracle.nvfp4_quant(v)
    s = oracle.e4m3(int(scales[0])) * G
    assert d[1] == pytest.approx(0.5 * s) and d[2] == 0.0
