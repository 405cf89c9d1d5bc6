"""Pins of the oracle's MXFP4 quantizer / dequantizer and of the two FP8 conversions.

MX rule ("Pretraining LLMs with MXFP4 on Native FP4 Hardware", MX section):
X ~ 2^E * Q_FP4(X / 2^E), E the block's shared exponent, Q_FP4 round to nearest.
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1_SET = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def unpack(q: np.ndarray) -> np.ndarray:
    """[R, C/2] packed -> [R, C] codes (even element = low nibble)."""
    out = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = q & 0xF
    out[:, 1::2] = q >> 4
    return out


def _read_blocks():
    blocks = []
    with open(os.path.join(GOLDEN, "mx_blocks.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            name, xs, sb, cs = [t.strip() for t in line.split("|")]
            x = np.zeros(32, dtype=np.float64)
            for tok in xs.split():
                i, v = tok.split("=")
                x[int(i)] = float(eval(v))
            codes = np.zeros(32, dtype=np.uint8)
            for tok in cs.split():
                i, c = tok.split("=")
                codes[int(i)] = int(c)
            blocks.append((name, x, int(sb), codes))
    return blocks


@pytest.mark.parametrize("blk", _read_blocks(), ids=lambda b: b[0])
def test_mx_golden_blocks(oracle, blk):
    name, x, sbyte, codes = blk
    x32 = x.astype(np.float32)     # decimal literals are taken at their FP32 rounding
    q, s = oracle.mx_quantize(x32[None, :])
    assert s[0, 0] == sbyte
    assert np.array_equal(unpack(q)[0], codes)


def _ref_quantize_f64(x: np.ndarray):
    """Independent restatement for the sweep: E from log2 of the block amax,
    rounding by the threshold table of round-to-nearest-even."""
    R, C = x.shape
    xb = x.reshape(R, C // 32, 32).astype(np.float64)
    amax = np.abs(xb).max(axis=2)
    with np.errstate(divide="ignore"):
        e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, -127)
    e = np.clip(e, -127, 127).astype(np.int64)
    v = xb * np.exp2(-e.astype(np.float64))[:, :, None]
    a = np.abs(v)
    mag = np.select([a <= 0.25, a < 0.75, a <= 1.25, a < 1.75, a <= 2.5, a < 3.5, a <= 5.0],
                    [0, 1, 2, 3, 4, 5, 6], default=7)
    codes = (mag | (np.signbit(v).astype(np.int64) << 3)).reshape(R, C).astype(np.uint8)
    return codes, (e + 127).astype(np.uint8)


def _all_finite_bf16():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = (b.astype(np.uint32) << 16).view(np.float32)
    return b[np.isfinite(f)]


@pytest.mark.parametrize("placement", ["alone", "uniform", "next_to_one"])
def test_mx_bruteforce_every_bf16(oracle, placement):
    b = _all_finite_bf16()
    n = b.size
    x = np.zeros((n, 32), dtype=np.uint16)
    if placement == "alone":
        x[:, 7] = b
    elif placement == "uniform":
        x[:, :] = b[:, None]
    else:
        x[:, 0] = b
        x[:, 1] = 0x3F80          # 1.0
    q, s = oracle.mx_quantize(x)
    codes, sref = _ref_quantize_f64(oracle.bf16_bits_to_f32(x))
    assert np.array_equal(s[:, 0], sref[:, 0])
    assert np.array_equal(unpack(q), codes)


def test_mx_invariants_random(oracle):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 512)) * np.exp2(rng.integers(-20, 20, (64, 1)))).astype(np.float32)
    x[3, 64:96] = 0.0
    x[5, :] *= 1e-38          # subnormal block amax
    q, s = oracle.mx_quantize(x)
    codes = unpack(q)
    vals = oracle.e2m1_values()[codes]
    e = s.astype(np.int64) - 127
    scale = np.repeat(np.exp2(e.astype(np.float64)), 32, axis=1)
    # codes confined to the E2M1 set
    assert set(np.unique(np.abs(vals))) <= set(E2M1_SET)
    # reconstruction = 2^E * Q(x / 2^E) with Q nearest on the grid
    yf, _ = oracle.mx_dequantize(q, s)
    assert np.array_equal(yf.astype(np.float64), vals * scale)
    # |dequantized| <= 6 * 2^E ; for non-zero blocks the dequantized block max is 4 or 6 times 2^E
    assert np.all(np.abs(vals * scale) <= 6 * scale)
    qmax = np.abs(vals).reshape(64, -1, 32).max(axis=2)
    nz = np.abs(x).reshape(64, -1, 32).max(axis=2) > 0
    big = e > -127       # blocks whose exponent was not clamped
    assert set(np.unique(qmax[nz & big])) <= {4.0, 6.0}
    # the error against the source is at most half a grid step at that magnitude
    v = x.astype(np.float64) / scale
    step = np.where(np.abs(v) < 2, 0.5, np.where(np.abs(v) < 4, 1.0, 2.0))
    err = np.abs(vals - np.clip(v, -6, 6))
    assert np.all(err <= step / 2 + 1e-12)
    # idempotence: quantize(dequantize(q)) == q
    q2, s2 = oracle.mx_quantize(yf)
    assert np.array_equal(q2, q) and np.array_equal(s2, s)


def test_mx_dequantize_bf16_is_the_exact_value(oracle):
    rng = np.random.default_rng(1)
    q = rng.integers(0, 256, (8, 64), dtype=np.uint8)
    s = rng.integers(1, 250, (8, 4), dtype=np.uint8)
    yf, yb = oracle.mx_dequantize(q, s)
    assert np.array_equal(oracle.bf16_bits_to_f32(yb), yf)    # 2-bit significands fit BF16
    s[:] = 0                                                  # 2^-127: FP32/BF16 subnormal range
    yf, yb = oracle.mx_dequantize(q, s)
    ref = oracle.e2m1_values()[unpack(q)] * 2.0 ** -127
    assert np.array_equal(yf.astype(np.float64), ref)


# ---------------------------------------------------------------------------
# Direct FP8 -> MXFP4
# ---------------------------------------------------------------------------
def test_fp8_to_mx_equals_mx_of_the_fp32_products(oracle):
    rng = np.random.default_rng(2)
    R, C = 16, 512
    x8 = rng.integers(0, 256, (R, C), dtype=np.uint8)
    x8[(x8 & 0x7F) == 0x7F] = 0x3C        # no NaN codes
    ts = (rng.uniform(0.5, 2, (R, C // 128)) * np.exp2(rng.integers(-30, 30, (R, C // 128)))).astype(np.float32)
    ts[0, 0] = -ts[0, 0]                   # a negative tile scale is allowed
    q, s = oracle.fp8_to_mx(x8, ts)
    dec = oracle.e4m3_values()[x8].astype(np.float32)          # exact
    prod = dec * np.repeat(ts, 128, axis=1)                   # one FP32 RN multiply
    q2, s2 = oracle.mx_quantize(prod.astype(np.float32))
    assert np.array_equal(q, q2) and np.array_equal(s, s2)


def test_fp8_block_amax_from_magnitude_bytes(oracle):
    # the FP32 products are monotone in the E4M3 magnitude, so the block amax is
    # reached at the largest magnitude byte (for every scale tried)
    vals = oracle.e4m3_values()[:0x7f].astype(np.float32)
    rng = np.random.default_rng(3)
    for sc in np.concatenate([rng.uniform(1e-3, 1e3, 200), [1.0, 2.0 ** -100, 3.3e-38]]).astype(np.float32):
        p = vals * sc
        assert np.all(np.diff(p) >= 0)


# ---------------------------------------------------------------------------
# Scaled MXFP4 -> FP8
# ---------------------------------------------------------------------------
def _bit_remap(code: int, d: int) -> int:
    """Independent bit-level restatement: E2M1 (k, m) fields rebased by d into E4M3."""
    sign = 0x80 if code & 8 else 0
    c = code & 7
    if c == 0:
        return sign
    k, m = (-1, 0) if c == 1 else ((c >> 1) - 1, c & 1)
    t = k + d                      # value = (1 + m/2) * 2^t
    if t >= -6:
        return sign | ((t + 7) << 3) | (m << 2)
    units = (2 + m) * 2.0 ** (t + 9 - 1)     # value in units of 2^-9
    if units < 1:
        return sign
    f = math.floor(units)
    r = units - f
    n = f + (1 if (r > 0.5 or (r == 0.5 and f % 2 == 1)) else 0)
    return sign | n if n < 8 else sign | 0x08


def test_mx_to_fp8_element_rule_all_codes_all_shifts(oracle):
    for code in range(16):
        for d in range(-254, 1):
            assert oracle.fp8_from_e2m1_shifted(code, d) == _bit_remap(code, d), (code, d)


def test_mx_to_fp8_golden(oracle):
    with open(os.path.join(GOLDEN, "mx_to_fp8_tiles.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, d, b = line.split()
                assert oracle.fp8_from_e2m1_shifted(int(c), int(d)) == int(b, 16), line


def test_mx_to_fp8_tiles_lossless(oracle):
    rng = np.random.default_rng(4)
    R, C = 32, 1024
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    base = rng.integers(100, 150, (R, C // 128))
    s = (np.repeat(base, 4, axis=1) - rng.integers(0, 7, (R, C // 32))).astype(np.uint8)
    y, ts = oracle.mx_to_fp8(q, s)
    # tile scale = 2^max(E_i) over the 4 blocks of the tile
    emax = (s.reshape(R, -1, 4).astype(np.int64) - 127).max(axis=2)
    assert np.array_equal(ts.astype(np.float64), np.exp2(emax.astype(np.float64)))
    # lossless: FP8 value * tile scale == MXFP4 value (in-row exponent spread <= 6 -> no flush)
    e8 = oracle.e4m3_values()[y] * np.repeat(ts.astype(np.float64), 128, axis=1)
    mx = oracle.mx_dequantize_f64(q, s)
    assert np.array_equal(e8, mx)


def test_mx_to_fp8_flush_counts_only_deep_shifts(oracle):
    q = np.full((1, 64), 0x77, dtype=np.uint8)            # all codes 6.0
    s = np.array([[127, 127 - 12, 127 - 10, 127 - 9]], dtype=np.uint8)
    y, ts = oracle.mx_to_fp8(q, s)
    assert ts[0, 0] == 1.0
    assert np.all(y[0, 32:64] == 0)                        # 6 * 2^-12 < 2^-9 -> flushed
    assert np.all(y[0, 64:96] == 0x03)                     # 6 * 2^-10 = 3 * 2^-9
    assert np.all(y[0, 96:128] == 0x06)                    # 6 * 2^-9


def test_mx_shared_exponent_edges(oracle):
    """E = floor(log2 amax) - 2 (E2M1's largest exponent), -127 for a zero
    block, clamped to the E8M0 range [-127, 127]."""
    assert oracle.mx_shared_exponent(6.0) == 0
    assert oracle.mx_shared_exponent(4.0) == 0
    assert oracle.mx_shared_exponent(3.999) == -1
    assert oracle.mx_shared_exponent(1.5 * 2.0 ** 100) == 98
    assert oracle.mx_shared_exponent(0.0) == -127
    assert oracle.mx_shared_exponent(2.0 ** -126) == -127          # -128 clamped
    assert oracle.mx_shared_exponent(2.0 ** -140) == -127
    assert oracle.mx_shared_exponent(2.0 ** 200) == 127


def test_mx_quantize_col_hand_derived(oracle):
    """Blocks of 32 run down the columns and the result is laid out by column:
    column 0 holds 4.0, 0.5, -1.5 and zeros (amax 4: E = 0, codes 6, 1, 0xB
    and 0), column 1 is all 1.0 (amax 1: E = -2, 1 / 2^-2 = 4 -> code 6)."""
    x = np.zeros((32, 2), dtype=np.float32)
    x[0, 0], x[1, 0], x[2, 0] = 4.0, 0.5, -1.5
    x[:, 1] = 1.0
    q, s = oracle.mx_quantize_col(x)
    assert q.shape == (2, 16) and s.shape == (2, 1)
    assert s[0, 0] == 127 and s[1, 0] == 125
    codes = np.empty((2, 32), dtype=np.uint8)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    assert list(codes[0, :3]) == [6, 1, 0xB] and np.all(codes[0, 3:] == 0)
    assert np.all(codes[1] == 6)
