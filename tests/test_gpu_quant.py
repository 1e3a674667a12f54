"""GPU parity of the NVFP4 activation quantiser of the prefill path
(moe_nvfp4_quantize) against the oracle's quantiser: codes, scale bytes and
global scales bit-exact.  Rows: random values over a wide range of
magnitudes, rows of zeros and of one value, rows whose values sit exactly on
the E2M1 rounding ties (and one ulp either side of them) for exactly known
scales, rows tiny and huge enough to leave the fast quotient's range, and a
ragged last 128-row tile."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import _scale_pos, f32_to_bf16

pytestmark = pytest.mark.gpu

TIES = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.5, 1.0, 1.5, 3.0])
E4M3_VALS = np.array([1.0, 1.125, 1.5, 1.75, 2.0, 2.5, 3.25, 6.0, 7.5, 0.75])


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from routed_expert_layer_router_gb300 import moe
    moe.lib()


def _tie_row(rng, K, e, nudge):
    """Row with G = 2^-e exactly (its max is 2688 G) whose blocks have max
    6 G s for an E4M3 value s, so that the block's dequantised scale is s G
    exactly; the other values are boundaries b * s G, moved `nudge` ulps."""
    G = np.float32(2.0 ** -e)
    v = np.zeros(K, np.float32)
    for b in range(K // 16):
        s = np.float32(448.0) if b == 0 else np.float32(rng.choice(E4M3_VALS))
        sdq = np.float32(s * G)
        blk = (rng.choice(TIES, 16) * sdq).astype(np.float32)
        blk *= rng.choice([-1.0, 1.0], 16).astype(np.float32)
        if nudge:
            u = blk.view(np.int32) + rng.integers(-nudge, nudge + 1, 16).astype(np.int32)
            blk = u.view(np.float32)
        blk[rng.integers(16)] = np.float32(6.0) * sdq  # the block max
        v[b * 16:(b + 1) * 16] = blk
    return v


def _rows(K, T, seed, bf16):
    rng = np.random.default_rng(seed)
    X = np.empty((T, K), np.float32)
    for t in range(T):
        kind = t % 8
        if kind == 0:
            X[t] = 0.0
            X[t, rng.integers(K)] = np.float32(rng.normal() * 3.0)
        elif kind == 1:
            X[t] = _tie_row(rng, K, int(rng.integers(-6, 20)), 0)
        elif kind == 2:
            X[t] = _tie_row(rng, K, int(rng.integers(-6, 20)), 1 if bf16 else 3)
        elif kind == 3:
            X[t] = rng.normal(size=K) * np.float32(10.0 ** rng.uniform(-30, -25))  # tiny
        elif kind == 4:
            X[t] = rng.normal(size=K) * np.float32(10.0 ** rng.uniform(25, 30))  # huge
        else:
            X[t] = rng.normal(size=K) * np.float32(2.0 ** rng.uniform(-20, 20))
    X[T // 2] = 0.0  # a zero row
    if bf16:
        xb = f32_to_bf16(X)
        for t in range(2, T, 8):  # nudged tie rows: move by one bf16 ulp instead
            d = np.random.default_rng(seed + t).integers(-1, 2, K).astype(np.int32)
            xb[t] = (xb[t].astype(np.int32) + d).astype(np.uint16)
        return xb, (xb.astype(np.uint32) << 16).view(np.float32)
    return X, X


def _unswizzle(scales, T, K):
    KB = K // 16
    t = np.arange(T)[:, None]
    b = np.arange(KB)[None, :]
    return scales[_scale_pos(t, b, KB)]


@pytest.mark.parametrize("dtype,K,T", [(0, 6144, 300), (0, 256, 130), (0, 8192, 40),
                                       (0, 4096, 64), (1, 2048, 300), (1, 4096, 72),
                                       (1, 256, 129)])
def test_quantize_matches_oracle_bit_exact(dtype, K, T):
    from routed_expert_layer_router_gb300 import moe
    xh, xf = _rows(K, T, seed=7 + K + T, bf16=(dtype == 0))
    dev = torch.from_numpy(xh.view(np.int16) if dtype == 0 else xh).cuda()
    tiles = (T + 127) // 128
    codes = torch.full((T, K // 2), 0xEE, dtype=torch.uint8, device="cuda")
    scales = torch.full((tiles * 128 * K // 16,), 0xEE, dtype=torch.uint8, device="cuda")
    G = torch.full((T,), -1.0, dtype=torch.float32, device="cuda")
    moe.moe_nvfp4_quantize(dev.data_ptr(), dtype, T, K, codes.data_ptr(), scales.data_ptr(),
                           G.data_ptr())
    torch.cuda.synchronize()
    codes, scales, G = codes.cpu().numpy(), scales.cpu().numpy(), G.cpu().numpy()
    sc = _unswizzle(scales, T, K)
    for t in range(T):
        oc, os_, oG = oracle.nvfp4_quant(xf[t])
        assert np.float32(oG) == G[t], (t, oG, G[t])
        assert np.array_equal(os_, sc[t]), (t, np.flatnonzero(os_ != sc[t])[:8])
        bad = np.flatnonzero(oc != codes[t])
        assert bad.size == 0, (t, bad[:8], oc[bad[:8]], codes[t][bad[:8]])


def test_quantize_of_no_rows_is_a_no_op():
    from routed_expert_layer_router_gb300 import moe
    moe.moe_nvfp4_quantize(0, 0, 0, 256, 0, 0, 0)
