"""Pins of the oracle's 16-point random Hadamard transform and NVFP4 quantizer.

"Pretraining Large Language Models with NVFP4", technical summary 2.A (format:
16-element E2M1 blocks, E4M3 block scale, FP32 tensor scale) and 2.B (random
Hadamard transform on the weight-gradient inputs, stochastic rounding).
"""
import math

import numpy as np
import pytest

E2M1_SET = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _sylvester(n=16):
    i = np.arange(n)
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


def _rht_with_signs(oracle, x, d):
    import ctypes
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = np.ascontiguousarray(d, dtype=np.float32)
    y = np.empty(16, dtype=np.float32)
    oracle._L().or_rht16(oracle._p(x), oracle._p(d), oracle._p(y))
    return y


def test_rht_columns_are_the_sylvester_matrix(oracle):
    H = _sylvester()
    assert np.array_equal(H @ H.T, 16 * np.eye(16))           # closed form H H^T = 16 I
    ones = np.ones(16)
    cols = np.stack([_rht_with_signs(oracle, np.eye(16)[j], ones) for j in range(16)], axis=1)
    assert np.array_equal(cols.astype(np.float64), H / 4)


def test_rht_matches_matrix_product(oracle):
    H = _sylvester()
    rng = np.random.default_rng(0)
    d = np.where(rng.random(16) < 0.5, -1.0, 1.0)
    for trial in range(200):
        x = rng.integers(-1000, 1000, 16).astype(np.float64)  # small integers: exact
        y = _rht_with_signs(oracle, x, d)
        assert np.array_equal(y.astype(np.float64), (H @ (d * x)) / 4)
    for trial in range(200):
        x = rng.standard_normal(16).astype(np.float32)
        y = _rht_with_signs(oracle, x, d).astype(np.float64)
        ref = (H @ (d * x.astype(np.float64))) / 4
        assert np.all(np.abs(y - ref) <= 4 * np.spacing(np.float32(np.abs(x).max() * 4)))


def test_rht_is_orthogonal(oracle):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 16)).astype(np.float32)
    y = oracle.rht16(x, 7).astype(np.float64)
    xn = np.linalg.norm(x.astype(np.float64), axis=1)
    assert np.allclose(np.linalg.norm(y, axis=1), xn, rtol=1e-6)
    # inverse: x = D (H/4)^T y
    d = oracle.rht16_signs(7).astype(np.float64)
    H = _sylvester()
    back = (y @ (H / 4)) * d
    assert np.allclose(back, x, atol=1e-6)


def test_rht_signs_from_philox_word(oracle):
    d = oracle.rht16_signs(7)
    w = oracle.philox4x32_10([0, 0, 0, 0], [7, 0])[0]
    assert set(np.unique(d)) <= {-1.0, 1.0}
    assert [int(x < 0) for x in d] == [(int(w) >> j) & 1 for j in range(16)]


def test_rht_cancels_in_the_contraction(oracle):
    # the rotation applied to both operands along K drops out of A . B^T
    rng = np.random.default_rng(2)
    a = rng.standard_normal((8, 64)).astype(np.float32)
    b = rng.standard_normal((8, 64)).astype(np.float32)
    ya = oracle.rht16(a, 7).astype(np.float64)
    yb = oracle.rht16(b, 7).astype(np.float64)
    assert np.allclose(ya @ yb.T, a.astype(np.float64) @ b.astype(np.float64).T, atol=1e-4)


def _bf16(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def unpack(q):
    out = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = q & 0xF
    out[:, 1::2] = q >> 4
    return out


def test_nv_golden_single_block(oracle):
    # one 16-element block, no rotation, amax 3: s_t = 3/2688, the block ratio is
    # 3 / (6 s_t) ~ 448 -> E4M3 0x7e; sf = 448 s_t ~ 0.5 -> codes 3->6 (7), 1->2 (4),
    # 0.5->1 (2), -0.25 -> -0.5 (9), 0.125 -> 0.25 tie -> 0 (0)
    x = np.zeros((1, 16), dtype=np.float32)
    x[0, :5] = [3.0, 1.0, 0.5, -0.25, 0.125]
    r = oracle.nv_quantize(_bf16(x))
    assert r["amax"] == np.float32(3.0)
    assert r["s_t"] == np.float32(3.0) / np.float32(2688.0)
    assert r["s"][0, 0] == 0x7E
    assert list(unpack(r["q"])[0, :5]) == [7, 4, 2, 9, 0]


def test_nv_invariants(oracle):
    rng = np.random.default_rng(3)
    x = (rng.standard_t(3, (64, 256)) * 1e-3).astype(np.float32)
    x[2, 16:32] = 0.0
    xb = _bf16(x)
    for rht in (False, True):
        r = oracle.nv_quantize(xb, rht=rht, rht_seed=7)
        y = oracle.rht16(oracle.bf16_bits_to_f32(xb), 7) if rht else oracle.bf16_bits_to_f32(xb)
        assert r["amax"] == np.abs(y).max()
        s_t = np.float32(r["s_t"])
        codes = unpack(r["q"])
        vals = oracle.e2m1_values()[codes]
        sb = oracle.e4m3_values()[r["s"]]
        assert set(np.unique(np.abs(vals))) <= set(E2M1_SET)
        assert np.all(sb <= 448) and np.all(sb >= 0)
        # per-block scaled amax lies in [6/(1+2^-4), 6/(1-2^-4)] when s_b is a
        # normal, unsaturated E4M3 value
        sf = (sb.astype(np.float32) * s_t).astype(np.float32)
        ab = np.abs(y).reshape(64, -1, 16).max(axis=2)
        normal = (sb >= 2.0 ** -6) & (sb < 448)
        ratio = ab[normal] / sf[normal]
        assert np.all(ratio >= 6 / (1 + 2 ** -4) - 1e-5) and np.all(ratio <= 6 / (1 - 2 ** -4) + 1e-5)
        # RNE error <= half a grid step (with saturation above 6)
        with np.errstate(divide="ignore", invalid="ignore"):     # zero blocks (sf = 0) are masked below
            v = y.astype(np.float64) / np.repeat(sf, 16, axis=1)
        step = np.where(np.abs(v) < 2, 0.5, np.where(np.abs(v) < 4, 1.0, 2.0))
        ok = np.repeat(sb, 16, axis=1) > 0
        err = np.abs(vals - np.clip(v, -6, 6))[ok]
        assert np.all(err <= step[ok] / 2 * (1 + 1e-6))
        # zero block -> zero scale, signed-zero codes
        if not rht:
            assert r["s"][2, 1] == 0 and np.all(codes[2, 16:32] & 7 == 0)
        # idempotence with the scales held fixed
        with np.errstate(divide="ignore", invalid="ignore"):
            rcp = (np.float32(1.0) / sf).astype(np.float32)
            v2 = (vals.astype(np.float32) * np.repeat(sf, 16, axis=1)).astype(np.float32) * np.repeat(rcp, 16, axis=1)
        q2 = oracle.e2m1_rne(v2.astype(np.float32))
        assert np.array_equal(q2[ok], codes[ok])


def test_nv_bruteforce_every_bf16_under_fixed_tensor_scale(oracle):
    # each finite BF16 value as the single non-zero element of a block, with the
    # tensor amax held at 1.0; reference: the same FP32 steps written in NumPy
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_bits_to_f32(b)
    keep = np.isfinite(f) & (np.abs(f) <= 1.0)
    b, f = b[keep], f[keep]
    x = np.zeros((b.size, 16), dtype=np.uint16)
    x[:, 3] = b
    r = oracle.nv_quantize(x, amax=1.0)
    s_t = np.float32(1.0) / np.float32(2688.0)
    ratio = (np.abs(f) / (np.float32(6.0) * s_t)).astype(np.float32)
    sb = oracle.e4m3_rn_satfinite(ratio)
    assert np.array_equal(r["s"][:, 0], sb)
    sbv = oracle.e4m3_values()[sb].astype(np.float32)
    sf = (sbv * s_t).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        rcp = (np.float32(1.0) / sf).astype(np.float32)
        v = (f * rcp).astype(np.float32)
    expect = np.where(sb > 0, oracle.e2m1_rne(np.where(sb > 0, v, 0).astype(np.float32)),
                      np.signbit(f).astype(np.uint8) << 3)
    assert np.array_equal(unpack(r["q"])[:, 3], expect)


def test_nv_sr_uses_the_linear_index_stream(oracle):
    rng = np.random.default_rng(4)
    x = _bf16(rng.standard_normal((8, 64)).astype(np.float32))
    r = oracle.nv_quantize(x, rounding="sr", sr_seed=1234)
    s_t = np.float32(r["s_t"])
    sb = oracle.e4m3_values()[r["s"]].astype(np.float32)
    sf = (sb * s_t).astype(np.float32)
    rcp = (np.float32(1.0) / sf).astype(np.float32)
    v = (oracle.bf16_bits_to_f32(x) * np.repeat(rcp, 16, axis=1)).astype(np.float32)
    words = oracle.sr_words(1234, 0, x.size).reshape(x.shape)
    assert np.array_equal(unpack(r["q"]), oracle.e2m1_sr(v, words))


def test_nv_sr_unbiased_in_the_mean(oracle):
    # averaged over many independent seeds, SR dequantizes to the input (scales fixed)
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((4, 64)).astype(np.float32))
    acc = np.zeros((4, 64))
    n = 400
    for k in range(n):
        r = oracle.nv_quantize(x, rounding="sr", sr_seed=1000 + k)
        acc += oracle.nv_dequantize_f64(r["q"], r["s"], r["s_t"])
    mean = acc / n
    xf = oracle.bf16_bits_to_f32(x).astype(np.float64)
    r0 = oracle.nv_quantize(x)
    sf = np.repeat(oracle.e4m3_values()[r0["s"]] * float(r0["s_t"]), 16, axis=1)
    # per-element sd of one draw is <= step/2 * sf <= sf; 6 sigma bound on the mean
    assert np.all(np.abs(mean - xf) <= 6 * sf / math.sqrt(n) + 1e-12)


def test_nv_quantize_col_runs_down_the_columns(oracle):
    """Column-wise NVFP4 of a matrix whose columns are constant: every 16-row
    block of column c sees the same 16 values, so row c of the transposed
    result repeats one scale byte and one code, and the dequantized value is
    the column's value within the E4M3 scale's rounding (2^-4 relative); a
    reduction along the wrong axis would mix the columns' magnitudes."""
    R, C = 64, 16
    v = (np.linspace(0.25, 3.0, C) * np.where(np.arange(C) % 2, -1.0, 1.0)).astype(np.float32)
    x = _bf16(np.tile(v, (R, 1)))
    r = oracle.nv_quantize_col(x)
    q, s = r["q"], r["s"]
    assert q.shape == (C, R // 2) and s.shape == (C, R // 16)
    assert np.all(s == s[:, :1]) and np.all(q == q[:, :1])
    y = oracle.nv_dequantize_f64(q, s, r["s_t"])
    vb = oracle.bf16_bits_to_f32(_bf16(v)).astype(np.float64)
    assert np.all(np.abs(y - vb[:, None]) <= np.abs(vb[:, None]) * 2.0 ** -4)
    assert len(np.unique(s[:, 0])) > 4                 # the columns' scales differ
