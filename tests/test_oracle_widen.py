"""Pins of the oracle's column-path, 2D-scaling and deterministic-Hadamard steps.

"Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs" (French
summary 2.C, Spanish summary 2): FP4RowToFP8Col, one kernel that dequantizes,
transposes and re-quantizes the weight-gradient operand.  "Pretraining Large
Language Models with NVFP4" (2.B): 16x16 block scaling of the weights, so the
forward pass and the transposed backward read identical values.  "Pretraining
large language models with MXFP4 on Native FP4 Hardware" (Wgrad section): the
deterministic Hadamard rotation H16, the same at every step.
"""
import numpy as np
import pytest
import scipy.linalg


def _bf16(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# deterministic H16 (rht = 2)
# ---------------------------------------------------------------------------
def test_deterministic_h16_is_the_scaled_sylvester_matrix(oracle):
    """rht=2 rotates each 16-tile by H16/4 with no sign flips: for a BF16 tile
    of small integers (exact in FP32) the rotated values are the product with
    the Sylvester matrix from scipy, so the amax is known in closed form."""
    H = scipy.linalg.hadamard(16).astype(np.float64)
    rng = np.random.default_rng(11)
    x = rng.integers(-8, 9, (4, 64)).astype(np.float32)
    y = np.concatenate([(H @ x[:, 16 * t:16 * t + 16].T).T / 4 for t in range(4)], axis=1)
    assert oracle.nv_amax(_bf16(x), 2, 0) == np.abs(y).max()
    # and it is an involution: (H/4)(H/4) = I
    assert np.array_equal((H / 4) @ (H / 4), np.eye(16))


def test_deterministic_h16_ignores_the_seed_and_differs_from_rht(oracle):
    rng = np.random.default_rng(12)
    xb = _bf16((rng.standard_t(3, (32, 128)) * 1e-3).astype(np.float32))
    a = oracle.nv_quantize(xb, rht=2, rht_seed=1)
    b = oracle.nv_quantize(xb, rht=2, rht_seed=99)
    c = oracle.nv_quantize(xb, rht=1, rht_seed=7)
    assert np.array_equal(a["q"], b["q"]) and np.array_equal(a["s"], b["s"])
    assert not np.array_equal(a["q"], c["q"])


def test_deterministic_h16_cancels_in_the_contraction(oracle):
    """The same rotation on both GEMM operands along K leaves A.B^T unchanged:
    (A H/4)(B H/4)^T = A B^T, checked on exactly representable integers."""
    H = scipy.linalg.hadamard(16).astype(np.float64) / 4
    rng = np.random.default_rng(13)
    A = rng.integers(-4, 5, (8, 16)).astype(np.float64)
    B = rng.integers(-4, 5, (8, 16)).astype(np.float64)
    assert np.array_equal((A @ H) @ (B @ H).T, A @ B.T)


# ---------------------------------------------------------------------------
# 2D (16 x 16) NVFP4
# ---------------------------------------------------------------------------
def test_2d_scaling_is_transpose_invariant(oracle):
    """The dequantized 16x16-scaled tensor of W^T is the transpose of that of W
    (the property the 2D scaling exists for); the 1D scaling does not have it."""
    rng = np.random.default_rng(14)
    w = (rng.standard_normal((64, 96)) * 0.02).astype(np.float32)
    w[:, 5] *= 30.0                                           # one outlier column
    wb = _bf16(w)
    a = oracle.nv_quantize_2d(wb)
    b = oracle.nv_quantize_2d(np.ascontiguousarray(wb.T))
    assert a["amax"] == b["amax"]
    da = oracle.nv_dequantize_f64(a["q"], a["s"], a["s_t"])
    db = oracle.nv_dequantize_f64(b["q"], b["s"], b["s_t"])
    assert np.array_equal(da, db.T)
    a1 = oracle.nv_quantize(wb)
    b1 = oracle.nv_quantize(np.ascontiguousarray(wb.T))
    assert not np.array_equal(oracle.nv_dequantize_f64(a1["q"], a1["s"], a1["s_t"]),
                              oracle.nv_dequantize_f64(b1["q"], b1["s"], b1["s_t"]).T)


def test_2d_scaling_reduces_to_1d_when_rows_share_the_block_amax(oracle):
    """If every row of every 16x16 tile has the same 16-element block amax, the
    2D and 1D scales coincide, hence so do all codes."""
    rng = np.random.default_rng(15)
    base = (rng.standard_normal((16, 64)) * 0.1).astype(np.float32)
    w = np.concatenate([base[rng.permutation(16)] for _ in range(4)], axis=0)   # 64 rows
    # make each row's block amax equal within a tile: put the tile's max in every row
    w = w.reshape(4, 16, 4, 16)
    m = np.abs(w).max(axis=(1, 3), keepdims=True)
    w[:, :, :, 0:1] = np.broadcast_to(m[:, :, :, 0:1] * 1.0, (4, 16, 4, 1))
    w = w.reshape(64, 64)
    wb = _bf16(w)
    a = oracle.nv_quantize_2d(wb)
    b = oracle.nv_quantize(wb)
    assert np.array_equal(a["s"], b["s"]) and np.array_equal(a["q"], b["q"])


def test_2d_scales_repeat_over_the_tile_rows(oracle):
    rng = np.random.default_rng(16)
    wb = _bf16((rng.standard_normal((48, 32)) * 0.05).astype(np.float32))
    r = oracle.nv_quantize_2d(wb)
    s = r["s"].reshape(3, 16, 2)
    assert np.all(s == s[:, :1, :])
    # the tile scale is the E4M3 rounding of tile amax / (6 s_t)
    x = oracle.bf16_bits_to_f32(wb).reshape(3, 16, 2, 16)
    ab = np.abs(x).max(axis=(1, 3)).astype(np.float32)
    want = oracle.e4m3_rn_satfinite((ab / (np.float32(6.0) * r["s_t"])).astype(np.float32))
    assert np.array_equal(s[:, 0, :], want)


def _tile_reciprocals(oracle, x, s_t):
    """1 / (E4M3(tile amax / (6 s_t)) * s_t) per 16x16 tile, in FP32, repeated
    over the tile's elements (the 2D scale rule restated here)."""
    R, C = x.shape
    ab = np.abs(x).reshape(R // 16, 16, C // 16, 16).max(axis=(1, 3)).astype(np.float32)
    sb = oracle.e4m3_values()[oracle.e4m3_rn_satfinite((ab / (np.float32(6.0) * s_t)).astype(np.float32))]
    sf = (sb.astype(np.float32) * s_t).astype(np.float32)
    rcp = (np.float32(1.0) / sf).astype(np.float32)
    return np.repeat(np.repeat(rcp, 16, axis=0), 16, axis=1)


def test_2d_sr_takes_the_word_of_each_elements_linear_index(oracle):
    """SR in the 2D form: element (r, c) of an R x C weight is rounded with word
    r * C + c of the Philox stream (the index is the element's, not its tile's
    or the transpose's), over the same scales as the RNE pass.  The shape is not
    square and spans several tiles in both directions, so a tile-wise or
    transposed index, or scales that depend on the rounding, fail."""
    from _helpers import unpack
    rng = np.random.default_rng(18)
    R, C = 48, 80
    w = (rng.standard_normal((R, C)) * 0.02).astype(np.float32)
    w[7, :] *= 25.0
    wb = _bf16(w)
    sr = oracle.nv_quantize_2d(wb, rounding="sr", sr_seed=1234)
    rne = oracle.nv_quantize_2d(wb)
    assert np.array_equal(sr["s"], rne["s"]) and sr["s_t"] == rne["s_t"]
    x = oracle.bf16_bits_to_f32(wb)
    s_t = (np.float32(np.abs(x).max()) / np.float32(2688.0)).astype(np.float32)
    assert s_t == sr["s_t"]
    v = (x * _tile_reciprocals(oracle, x, s_t)).astype(np.float32)
    words = oracle.sr_words(1234, 0, R * C)
    assert np.array_equal(unpack(sr["q"]), oracle.e2m1_sr(v, words.reshape(R, C)))
    # the plausible wrong indexings give other codes on this input
    assert not np.array_equal(unpack(sr["q"]), oracle.e2m1_sr(v, words.reshape(C, R).T))
    tile_major = words.reshape(R // 16, C // 16, 16, 16).transpose(0, 2, 1, 3).reshape(R, C)
    assert not np.array_equal(unpack(sr["q"]), oracle.e2m1_sr(v, tile_major))
    # a different seed draws a different stream
    assert not np.array_equal(sr["q"], oracle.nv_quantize_2d(wb, rounding="sr", sr_seed=1235)["q"])


def test_2d_sr_is_unbiased_in_the_mean(oracle):
    """Averaged over many seeds, the 2D SR result dequantizes to the input
    (scales are fixed by the tile amax): per element within 6 sigma, sigma of
    one draw being at most half a grid step times the scale (<= the scale)."""
    rng = np.random.default_rng(19)
    R, C = 32, 48
    wb = _bf16((rng.standard_normal((R, C)) * 0.05).astype(np.float32))
    n = 400
    acc = np.zeros((R, C))
    for k in range(n):
        r = oracle.nv_quantize_2d(wb, rounding="sr", sr_seed=2000 + k)
        acc += oracle.nv_dequantize_f64(r["q"], r["s"], r["s_t"])
    x = oracle.bf16_bits_to_f32(wb).astype(np.float64)
    r0 = oracle.nv_quantize_2d(wb)
    sf = np.repeat(oracle.e4m3_values()[r0["s"]] * float(r0["s_t"]), 16, axis=1)
    err = np.abs(acc / n - x)
    assert np.all(err <= 6 * sf / np.sqrt(n) + 1e-12)
    # and RNE is biased somewhere on the same input (the test can tell the two apart)
    assert np.abs(oracle.nv_dequantize_f64(r0["q"], r0["s"], r0["s_t"]) - x).max() > 6 * sf.max() / np.sqrt(n)


# ---------------------------------------------------------------------------
# FP4RowToFP8Col
# ---------------------------------------------------------------------------
def test_fp4_row_to_fp8_col_is_lossless_and_transposed(oracle):
    """With block exponents within 6 of each other down every 128-row tile, the
    FP8 copy (times its tile scale) is exactly the transpose of the MXFP4 value,
    and the tile scale is 2^(largest block exponent of the tile)."""
    rng = np.random.default_rng(17)
    R, C = 256, 96
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    base = rng.integers(110, 140, (R // 128, C // 32))
    s = (np.repeat(base, 128, axis=0) - rng.integers(0, 7, (R, C // 32))).astype(np.uint8)
    y, ts = oracle.mx_to_fp8_col(q, s)
    assert y.shape == (C, R) and ts.shape == (C, R // 128)
    e = s.astype(np.int64) - 127
    emax = e.reshape(R // 128, 128, C // 32).max(axis=1)                 # [tiles, blocks]
    assert np.array_equal(ts.astype(np.float64), np.exp2(np.repeat(emax.T, 32, axis=0)))
    e8 = oracle.e4m3_values()[y] * np.repeat(ts.astype(np.float64), 128, axis=1)
    assert np.array_equal(e8, oracle.mx_dequantize_f64(q, s).T)


def test_fp4_row_to_fp8_col_flushes_only_deep_shifts(oracle):
    R, C = 128, 32
    q = np.full((R, C // 2), 0x77, dtype=np.uint8)            # all codes 6.0
    s = np.full((R, 1), 127, dtype=np.uint8)
    s[1:32] = 127 - 12                                        # 6 * 2^-12 < 2^-9: flushed
    s[32:64] = 127 - 10                                       # 6 * 2^-10 = 3 * 2^-9
    s[64:] = 127 - 9                                          # 6 * 2^-9
    y, ts = oracle.mx_to_fp8_col(q, s)
    assert np.all(ts == 1.0)
    assert np.all(y[:, 0] == 0x4C)                            # 6.0 = 1.5 * 2^2 in E4M3
    assert np.all(y[:, 1:32] == 0) and np.all(y[:, 32:64] == 0x03) and np.all(y[:, 64:] == 0x06)


def test_fp4_row_to_fp8_col_agrees_with_the_row_kernel_on_a_transposed_tile(oracle):
    """When each block exponent is constant along the rows of a 128x128 tile and
    the codes form a symmetric pattern, the column conversion of the tile equals
    the row conversion (a different code path of the oracle)."""
    rng = np.random.default_rng(18)
    codes = rng.integers(0, 16, (128, 128), dtype=np.uint8)
    codes = np.triu(codes) + np.triu(codes, 1).T               # symmetric
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    s = np.full((128, 4), 120, dtype=np.uint8)
    yc, tc = oracle.mx_to_fp8_col(q, s)
    yr, tr = oracle.mx_to_fp8(q, s)
    assert np.array_equal(yc, yr) and np.array_equal(tc, tr)


def test_fp4_row_to_fp8_col_grouped_equals_the_dense_rule_on_tile_aligned_groups(oracle):
    """Groups whose sizes are multiples of 128 are laid out back to back with no
    padding, so the grouped form is the dense form of the whole tensor."""
    rng = np.random.default_rng(19)
    R, C = 512, 64
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    s = rng.integers(110, 140, (R, C // 32), dtype=np.uint8)
    y, ts = oracle.mx_to_fp8_col_grouped(q, s, [0, 128, 128, 384, 512])
    yd, tsd = oracle.mx_to_fp8_col(q, s)
    assert np.array_equal(y, yd) and np.array_equal(ts, tsd)


def test_fp4_row_to_fp8_col_grouped_partial_tile_by_hand(oracle):
    """Groups of 3 and 2 rows, one 32-column block: each group is one tile whose
    scale is 2^(max E of its own rows), with its rows at the start of the tile
    and zeros after them; the second group's large exponent does not reach the
    first group's tile."""
    q = np.zeros((5, 16), dtype=np.uint8)
    q[:, 0] = [0x77, 0x22, 0x11, 0x77, 0x44]          # element 0 codes 7, 2, 1, 7, 4
    s = np.array([[127], [126], [125], [140], [127]], dtype=np.uint8)
    y, ts = oracle.mx_to_fp8_col_grouped(q, s, [0, 3, 5])
    assert y.shape == (32, 256) and ts.shape == (32, 2)
    assert np.all(ts[:, 0] == 1.0) and np.all(ts[:, 1] == np.float32(2.0 ** 13))
    # group 0 (Emax 0): 6.0 -> 0x4C; 1.0 * 2^-1 = 0.5 -> 0x30; 0.5 * 2^-2 = 2^-3 -> 0x20
    assert list(y[0, :3]) == [0x4C, 0x30, 0x20] and list(y[1, :3]) == [0x4C, 0x30, 0x20]
    # group 1 (Emax 13): 6.0 -> 0x4C; 2.0 * 2^-13 -> 2^-12 < 2^-9: flushed to zero
    assert list(y[0, 128:130]) == [0x4C, 0x00]
    assert np.all(y[:, 3:128] == 0) and np.all(y[:, 130:] == 0)


def test_fp4_row_to_fp8_col_grouped_element_brute_force(oracle):
    """Element by element from the definition: output (c, 128 T_g + j) is the
    E4M3 of code (off_g + j, c) shifted by its block exponent minus the maximum
    block exponent of its 128-row tile within the group."""
    rng = np.random.default_rng(20)
    offs = [0, 0, 1, 130, 258, 300]
    R, C = 300, 64
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    s = rng.integers(100, 140, (R, C // 32), dtype=np.uint8)
    y, ts = oracle.mx_to_fp8_col_grouped(q, s, offs)
    codes = np.empty((R, C), dtype=np.int64)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    e = s.astype(np.int64) - 127
    t0 = 0
    for g in range(len(offs) - 1):
        n = offs[g + 1] - offs[g]
        for t in range((n + 127) // 128):
            lo, hi = offs[g] + 128 * t, min(offs[g] + 128 * (t + 1), offs[g + 1])
            for c in range(0, C, 7):
                emax = e[lo:hi, c // 32].max()
                assert ts[c, t0 + t] == np.float32(2.0 ** emax)
                for r in range(lo, hi):
                    want = oracle.fp8_from_e2m1_shifted(codes[r, c], e[r, c // 32] - emax)
                    assert y[c, 128 * (t0 + t) + (r - lo)] == want
            assert np.all(y[:, 128 * (t0 + t) + (hi - lo): 128 * (t0 + t + 1)] == 0)
        t0 += (n + 127) // 128
    assert y.shape[1] == 128 * t0


# ---------------------------------------------------------------------------
# FP8 GEMM reference (the FP8 consumer of the FP4 -> FP8 conversions)
# ---------------------------------------------------------------------------
def test_fp8_gemm_ref_against_exact_rationals(oracle):
    from fractions import Fraction
    rng = np.random.default_rng(19)
    lut = oracle.e4m3_values()
    ok = np.flatnonzero(np.isfinite(lut) & (np.abs(lut) <= 8))
    M, N, K = 3, 4, 256
    ya = rng.choice(ok, (M, K)).astype(np.uint8)
    yb = rng.choice(ok, (N, K)).astype(np.uint8)
    tsa = np.exp2(rng.integers(-3, 4, (M, K // 128))).astype(np.float32)
    tsb = np.exp2(rng.integers(-3, 4, (N, K // 128))).astype(np.float32)
    d = oracle.fp8_gemm_ref(ya, tsa, yb, tsb)
    for i in range(M):
        for j in range(N):
            acc = sum(Fraction(float(lut[ya[i, k]])) * Fraction(float(tsa[i, k // 128])) *
                      Fraction(float(lut[yb[j, k]])) * Fraction(float(tsb[j, k // 128])) for k in range(K))
            assert Fraction(d[i, j]) == acc
