"""Shared test helpers: tolerances, bit-constructed records and inputs."""
import numpy as np

# layer outputs: max |y - y_oracle| <= TOL * rms(y_oracle) over the whole output
TOL = 2e-2
# router probabilities (p_sel and renormalised w): relative error
PROB_RTOL = 1e-5

E4M3_ONE = 0x38      # 1.0
E4M3_SIXTEEN = 0x58  # 16.0
E4M3_2M6 = 0x08      # 2^-6
E2M1_ONE = 2         # code of 1.0
E2M1_FOUR = 6        # code of 4.0


def bf16_to_f64(x):
    return (np.asarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16(v):
    u = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _scale_pos(r, kb, KB):
    return ((r // 128) * (KB // 4) + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4


def identity_record(H, I):
    """Record whose expert maps x to y with y[16+i] = x[16+i] (i < I), y = 0
    elsewhere, provided x[0] = 1 and g = (1, 1, 1):
      gate row i = 64 e_0 (code 4.0, block scale 16), so g_i = 64 and silu(64) = 64
      up row i   = e_{16+i} (code 1.0, scale 1),       so h_i = 64 x[16+i]
      down row 16+i = e_i / 64 (code 1.0, scale 2^-6), so y[16+i] = x[16+i]."""
    assert I <= H - 16
    rb = 3 * I * H // 2 + 3 * I * H // 16
    rec = np.zeros(rb, np.uint8)
    codes = [0, I * H // 2, I * H]
    scales = [3 * I * H // 2 + m * (I * H // 16) for m in range(3)]
    KBh, KBi = H // 16, I // 16
    for m, R, KB, s in ((0, I, KBh, E4M3_ONE), (1, I, KBh, E4M3_ONE), (2, H, KBi, E4M3_2M6)):
        for r in range(R):
            for kb in range(KB):
                rec[scales[m] + _scale_pos(r, kb, KB)] = s

    def put(m, r, c, code, K):
        b = codes[m] + r * (K // 2) + c // 2
        rec[b] |= (code << 4) if (c & 1) else code

    for i in range(I):
        put(0, i, 0, E2M1_FOUR, H)
        rec[scales[0] + _scale_pos(i, 0, KBh)] = E4M3_SIXTEEN
        put(1, i, 16 + i, E2M1_ONE, H)
        put(2, 16 + i, i, E2M1_ONE, I)
    return rec


def identity_x(H, T, seed=0):
    """bf16 activations with x[0] = 1 (the identity expert's constant input)."""
    rng = np.random.default_rng(seed)
    x = f32_to_bf16(rng.standard_normal((T, H)).astype(np.float32))
    x[:, 0] = 0x3F80
    return x


_E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])


def nvfp4_exact_x(H, T, seed=0):
    """bf16 activations that NVFP4 quantisation reproduces exactly and whose
    x[16:] shifted by one block also does (the identity expert's h): row amax
    2.625 (G = 2^-10), block 0 on the grid 0.25*code with x[0] = 1 and a 1.5,
    later blocks on grids s*2^-10*code, s in {448, 224, 112}, each with a +-6."""
    rng = np.random.default_rng(seed)
    out = np.empty((T, H), np.float32)
    for t in range(T):
        for b in range(H // 16):
            s = 256.0 if b == 0 else float(rng.choice([448.0, 224.0, 112.0]))
            if b == 1:
                s = 448.0
            mags = rng.choice(_E2M1[:7], 16) * rng.choice([-1, 1], 16)
            mags[rng.integers(16)] = 6.0 * rng.choice([-1, 1])
            blk = mags * s * 2.0 ** -10
            if b == 0:
                blk[0] = 1.0
                blk[1] = 1.5
            out[t, b * 16:(b + 1) * 16] = blk
    return f32_to_bf16(out)


E8M0_ONE = 127        # 2^0
E8M0_SIXTEEN = 131    # 2^4
E8M0_2M6 = 121        # 2^-6


def identity_record_mx(H, I):
    """The identity expert in MXFP4 (blocks of 32, E8M0 scales): the same
    construction as identity_record - gate row i = 64 e_0 (code 4.0, block
    scale 16), up row i = e_{16+i} (code 1.0, scale 1), down row 16+i = e_i / 64
    (code 1.0, scale 2^-6) - so that y[16+i] = x[16+i] when x[0] = 1 and
    g = (1, 1, 1)."""
    assert I <= H - 16
    rb = 3 * I * H // 2 + 3 * I * H // 32
    rec = np.zeros(rb, np.uint8)
    codes = [0, I * H // 2, I * H]
    scales = [3 * I * H // 2 + m * (I * H // 32) for m in range(3)]
    KBh, KBi = H // 32, I // 32
    for m, R, KB, sc in ((0, I, KBh, E8M0_ONE), (1, I, KBh, E8M0_ONE), (2, H, KBi, E8M0_2M6)):
        for r in range(R):
            for kb in range(KB):
                rec[scales[m] + _scale_pos(r, kb, KB)] = sc

    def put(m, r, c, code, K):
        b = codes[m] + r * (K // 2) + c // 2
        rec[b] |= (code << 4) if (c & 1) else code

    for i in range(I):
        put(0, i, 0, E2M1_FOUR, H)
        rec[scales[0] + _scale_pos(i, 0, KBh)] = E8M0_SIXTEEN
        put(1, i, 16 + i, E2M1_ONE, H)
        put(2, 16 + i, i, E2M1_ONE, I)
    return rec


def mxfp4_exact_x(H, T, seed=0):
    """bf16 activations that MXFP4 quantisation reproduces exactly, and whose
    shift by 16 values (the identity expert's h = 64 x[16:]) does too: every
    value is an E2M1 magnitude times 2^-1 and every run of 16 values holds a
    +-3 (= 6 x 2^-1), so each block of 32 at any 16-value offset has the
    shared exponent -1; x[0] = 1."""
    rng = np.random.default_rng(seed)
    out = np.empty((T, H), np.float32)
    for t in range(T):
        for h in range(H // 16):
            mags = rng.choice(_E2M1[:7], 16) * rng.choice([-1, 1], 16)
            mags[rng.integers(16)] = 6.0 * rng.choice([-1, 1])
            out[t, h * 16:(h + 1) * 16] = mags * 0.5
        out[t, 0] = 1.0
        if not np.any(np.abs(out[t, :16]) == 3.0):
            out[t, 1] = 3.0
    return f32_to_bf16(out)
