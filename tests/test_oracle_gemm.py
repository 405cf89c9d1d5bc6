"""Pins of the GEMM and MoE oracles (float64 NumPy on dequantized operands)."""
from fractions import Fraction

import numpy as np


def test_gemm_ref_against_exact_rationals(oracle):
    # Y = A . B^T: every product of E2M1 values and power-of-two scales is exact,
    # so an exact rational triple loop pins the float64 matmul to 1 ulp-ish.
    rng = np.random.default_rng(0)
    M, N, K = 6, 5, 64
    qa = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(120, 135, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(120, 135, (N, K // 32), dtype=np.uint8)
    y = oracle.mx_gemm_ref(qa, sa, qb, sb)
    a = oracle.mx_dequantize_f64(qa, sa)
    b = oracle.mx_dequantize_f64(qb, sb)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(a[m, k])) * Fraction(float(b[n, k])) for k in range(K))
            assert abs(Fraction(float(y[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 48) + Fraction(1, 2 ** 200)


def test_nv_dequant_products_exact(oracle):
    # value(q) * s_b * s_t has at most 2 + 4 + 24 significant bits: exact in float64
    q = np.array([[0x7F, 0x21] + [0] * 6], dtype=np.uint8)
    s = np.array([[0x7E]], dtype=np.uint8)
    s_t = np.float32(3.0) / np.float32(2688.0)
    y = oracle.nv_dequantize_f64(q, s, s_t)
    # byte 0x7F: element 0 = low nibble 0xF (-6), element 1 = high nibble 0x7 (6)
    assert y[0, 0] == -6.0 * 448.0 * float(s_t) and y[0, 1] == 6.0 * 448.0 * float(s_t)
    # byte 0x21: element 2 = 0x1 (0.5), element 3 = 0x2 (1.0)
    assert y[0, 2] == 0.5 * 448.0 * float(s_t) and y[0, 3] == 1.0 * 448.0 * float(s_t)


def test_rel_frobenius(oracle):
    ref = np.array([[3.0, 4.0]])
    assert oracle.rel_frobenius(ref, ref) == 0.0
    assert abs(oracle.rel_frobenius(ref * 1.001, ref) - 1e-3) < 1e-12


def test_moe_dispatch_brute_force(oracle):
    rng = np.random.default_rng(1)
    T, k, E = 37, 3, 5
    topk = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    rows, offs = oracle.moe_dispatch(topk, E)
    # brute force: for every expert, the tokens that chose it, in ascending order
    expect = []
    eoffs = [0]
    for e in range(E):
        toks = [t for t in range(T) if e in topk[t]]
        expect += toks
        eoffs.append(eoffs[-1] + len(toks))
    assert list(rows) == expect and list(offs) == eoffs


def test_silu_closed_forms(oracle):
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0])
    s = oracle.silu(g)
    assert s[0] == 0.0
    assert abs(s[1] - 1.0 / (1.0 + np.exp(-1.0))) < 1e-16
    assert abs(s[1] - s[2] - 1.0) < 1e-15          # silu(x) - silu(-x) = x
    assert abs(s[3] - 30.0) < 1e-11 and abs(s[4]) < 1e-11


def test_mx_rebase_hand_derived_rows(oracle):
    # Row bytes 127, 119, 110, 109, 0 -> E = 0, -8, -17, -18, -127; B = max E - 8 = -8.
    # E - B = 8, 0, -9, -10, -119: UE4M3 0x78 (2^8), 0x38 (1.0), 0x01 (2^-9, the
    # smallest subnormal), then two unrepresentable blocks (byte 0, counted).
    ue, f, v = oracle.mx_rebase_scales(np.array([[127, 119, 110, 109, 0]], dtype=np.uint8))
    assert list(ue[0]) == [0x78, 0x78, 0x38, 0x38, 0x01, 0x01, 0, 0, 0, 0]
    assert f[0] == np.float32(2.0 ** -8) and v == 2
    # all-zero bytes (E = -127 everywhere): B = -135, an FP32 subnormal factor,
    # and every block is the top UE4M3 power 2^8
    ue, f, v = oracle.mx_rebase_scales(np.zeros((1, 3), dtype=np.uint8))
    assert np.all(ue == 0x78) and f[0] == np.float32(2.0 ** -135) and f[0] > 0 and v == 0
    # the largest finite E8M0 byte (254, E = 127): B = 119
    ue, f, v = oracle.mx_rebase_scales(np.array([[254, 238, 240, 233]], dtype=np.uint8))
    assert f[0] == np.float32(2.0 ** 119)
    # E - B: 8, -8, -6, -13 -> 0x78, 0x02 (2^-8), 0x08 (2^-6, the smallest normal), 0 (violation)
    assert list(ue[0]) == [0x78, 0x78, 0x02, 0x02, 0x08, 0x08, 0, 0] and v == 1


def test_mx_rebase_reconstructs_every_representable_block(oracle):
    # e4m3_value(byte) * 2^B == 2^E exactly where E - B >= -9, byte 0 elsewhere,
    # and the violation count is the number of blocks below B - 9
    rng = np.random.default_rng(11)
    s = rng.integers(0, 255, (64, 40), dtype=np.uint8)
    s[:32] = rng.integers(100, 140, (32, 40), dtype=np.uint8)     # rows with few violations
    ue, f, v = oracle.mx_rebase_scales(s)
    e = s.astype(np.int64) - 127
    B = e.max(axis=1) - 8
    ok = (e - B[:, None]) >= -9
    vals = oracle.e4m3_values()[ue[:, 0::2]] * f.astype(np.float64)[:, None]
    assert np.array_equal(vals[ok], np.exp2(e[ok].astype(np.float64)))
    assert np.all(ue[:, 0::2][~ok] == 0) and v == int((~ok).sum()) and v > 0
    assert np.array_equal(ue[:, 0::2], ue[:, 1::2])
    assert np.array_equal(f.astype(np.float64), np.exp2(B.astype(np.float64)))


def test_nv_gemm_ref_against_exact_rationals(oracle):
    """Y = s_tA s_tB sum_k (qA sA)(qB sB): an exact rational triple loop pins the
    float64 product of the dequantized NVFP4 operands, within the float64
    dot-product bound K 2^-52 sum |terms| (each dequantized value is exact, but
    a product of two carries up to 60 significant bits)."""
    rng = np.random.default_rng(3)
    M, N, K = 5, 4, 64
    qa = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x08, 0x7E, (M, K // 16), dtype=np.uint8)      # positive finite E4M3
    sb = rng.integers(0x08, 0x7E, (N, K // 16), dtype=np.uint8)
    sta, stb = np.float32(3.0 / 2688.0), np.float32(5.0 / 2688.0)
    y = oracle.nv_gemm_ref(qa, sa, sta, qb, sb, stb)
    e2m1 = oracle.e2m1_values()
    e4m3 = oracle.e4m3_values()
    def val(q, s, st, r, k):
        code = (q[r, k // 2] >> (4 * (k % 2))) & 0xF
        return Fraction(float(e2m1[code])) * Fraction(float(e4m3[s[r, k // 16]])) * Fraction(float(st))
    for m in range(M):
        for n in range(N):
            terms = [val(qa, sa, sta, m, k) * val(qb, sb, stb, n, k) for k in range(K)]
            exact = sum(terms)
            assert abs(Fraction(float(y[m, n])) - exact) <= K * Fraction(1, 2 ** 52) * sum(abs(t) for t in terms)


def test_moe_up_gate_closed_form(oracle):
    """h = SiLU(X W_g^T) * (X W_u^T): with one-hot token rows the projections are
    columns of W, so h is SiLU(W_g[j, i]) * W_u[j, i] for token i, channel j."""
    rng = np.random.default_rng(4)
    T, H, I = 3, 5, 4
    x = np.eye(T, H)
    w1 = rng.standard_normal((2 * I, H))
    h = oracle.moe_up_gate(x, w1, I)
    g, u = w1[:I, :T].T, w1[I:, :T].T                  # [T, I]
    want = g / (1.0 + np.exp(-g)) * u
    assert h.shape == (T, I) and np.allclose(h, want, rtol=1e-15, atol=0)
