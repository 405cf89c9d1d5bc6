"""GPU parity of the column path, the 2D weight scaling and the deterministic
H16 against the oracle (bit-exact), through the C ABI.

Column-wise quantize (block axis 0) and FP4RowToFP8Col: "Practical FP4
Training for Large-Scale MoE Models on Hopper GPUs", French summary 2.C and
Spanish summary 2.  16x16 NVFP4 weight scaling and the RHT on the Wgrad inputs:
"Pretraining Large Language Models with NVFP4", 2.B.  Deterministic H16:
"Pretraining large language models with MXFP4 on Native FP4 Hardware", Wgrad
section.
"""
import numpy as np
import pytest

from _helpers import dev, dev_bf16, from_mma_layout, host, rel_frobenius

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import micro_scaled_fp4_gb300.fp4q as fq
    fq.load()
    return fq


def _scales(fq, r, rows, scols, layout, key="scales"):
    sg = host(r[key] if isinstance(r, dict) else r)
    return from_mma_layout(sg.reshape(-1), rows, scols) if layout else sg


# ---------------------------------------------------------------------------
# deterministic H16 (rht = 2), row-wise
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rounding", [0, 1])
def test_nv_quantize_deterministic_h16(fq, oracle, rounding):
    from micro_scaled_fp4_gb300 import workloads as W
    x = W.gradient_bf16(129, 2048, seed=5)
    r = fq.nv_quantize(dev_bf16(x), rht=2, rht_seed=99, rounding=rounding, sr_seed=1234)
    ref = oracle.nv_quantize(x, rht=2, rounding="sr" if rounding else "rne", sr_seed=1234)
    assert host(r["amax"])[0] == ref["amax"] and host(r["s_t"])[0] == ref["s_t"]
    assert np.array_equal(host(r["q"]), ref["q"]) and np.array_equal(host(r["scales"]), ref["s"])


# ---------------------------------------------------------------------------
# column-wise NVFP4 and MXFP4 (block axis 0: quantization of X^T)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(128, 64), (384, 192), (256, 1024)])
@pytest.mark.parametrize("rht", [0, 1, 2])
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("layout", [0, 1])
def test_nv_quantize_column_wise(fq, oracle, shape, rht, rounding, layout):
    from micro_scaled_fp4_gb300 import workloads as W
    R, C = shape
    x = W.gradient_bf16(R, C, seed=R + 3 * C)
    r = fq.nv_quantize(dev_bf16(x), rht=rht, rht_seed=7, rounding=rounding, sr_seed=1234, layout=layout,
                       block_axis=0)
    ref = oracle.nv_quantize_col(x, rht=rht, rht_seed=7, rounding="sr" if rounding else "rne", sr_seed=1234)
    assert host(r["amax"])[0] == ref["amax"] and host(r["s_t"])[0] == ref["s_t"]
    assert np.array_equal(host(r["q"]), ref["q"])
    assert np.array_equal(_scales(fq, r, C, R // 16, layout), ref["s"])


@pytest.mark.parametrize("shape", [(128, 128), (384, 256), (256, 1152)])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("pad", [0, 64])
def test_mx_quantize_column_wise(fq, oracle, shape, layout, pad):
    R, C = shape
    rng = np.random.default_rng(R + C + pad)
    xf = (rng.standard_normal((R, C)) * np.exp2(rng.integers(-6, 6, (R, 1)))).astype(np.float32)
    xf[:, 7] *= 40.0
    xb = ((xf.view(np.uint32) + 0x7FFF + ((xf.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    big = np.zeros((R, C + pad), dtype=np.uint16)
    big[:, :C] = xb
    q, s = fq.mx_quantize(dev_bf16(big)[:, :C], layout=layout, block_axis=0)
    qr, sr = oracle.mx_quantize_col(xb)
    assert np.array_equal(host(q), qr)
    assert np.array_equal(_scales(fq, s, C, R // 32, layout), sr)


def test_nv_quantize_column_wise_full_size(fq, oracle):
    """The whole 8192x14336 gradient quantized column-wise (the Wgrad operand
    along the token axis) with the deterministic H16 and SR, then RNE: tensor
    amax, tensor scale, every code and every scale against the oracle's
    quantization of the transpose."""
    from micro_scaled_fp4_gb300 import workloads as W
    x = W.gradient_bf16()
    xd = dev_bf16(x)
    for rounding in ("sr", "rne"):
        r = fq.nv_quantize(xd, rht=2, rounding=1 if rounding == "sr" else 0, sr_seed=1234, block_axis=0)
        ref = oracle.nv_quantize_col(x, rht=2, rounding=rounding, sr_seed=1234)
        assert host(r["amax"])[0] == ref["amax"] and host(r["s_t"])[0] == ref["s_t"]
        assert np.count_nonzero(host(r["q"]) != ref["q"]) == 0, rounding
        assert np.count_nonzero(host(r["scales"]) != ref["s"]) == 0, rounding
        del r, ref


# ---------------------------------------------------------------------------
# 16x16 NVFP4 weights
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(16, 16), (64, 96), (4096, 7168)])
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("layout", [0, 1])
def test_nv_quantize_2d(fq, oracle, shape, rounding, layout):
    R, C = shape
    rng = np.random.default_rng(R + C)
    w = (rng.standard_normal((R, C)) * 0.02).astype(np.float32)
    w[:, 3] *= 25.0
    wb = ((w.view(np.uint32) + 0x7FFF + ((w.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    r = fq.nv_quantize(dev_bf16(wb), rounding=rounding, sr_seed=77, layout=layout, two_d=True)
    ref = oracle.nv_quantize_2d(wb, rounding="sr" if rounding else "rne", sr_seed=77)
    assert host(r["amax"])[0] == ref["amax"] and host(r["s_t"])[0] == ref["s_t"]
    assert np.array_equal(host(r["q"]), ref["q"])
    assert np.array_equal(_scales(fq, r, R, C // 16, layout), ref["s"])


def test_nv_2d_forward_and_transposed_weights_agree(fq, oracle):
    """The property 2D scaling exists for, on the GPU path: quantizing W and W^T
    gives transposed copies of the same values."""
    from micro_scaled_fp4_gb300 import workloads as W
    rng = np.random.default_rng(21)
    w = W.to_bf16_bits((rng.standard_normal((256, 512)) * 0.02).astype(np.float32))
    wt = np.ascontiguousarray(w.T)
    a = fq.nv_quantize(dev_bf16(w), two_d=True)
    b = fq.nv_quantize(dev_bf16(wt), two_d=True)
    # both kernel results are the oracle's 2D quantizations of W and W^T ...
    ra, rb = oracle.nv_quantize_2d(w), oracle.nv_quantize_2d(wt)
    for got, ref in ((a, ra), (b, rb)):
        assert np.array_equal(host(got["q"]), ref["q"]) and np.array_equal(host(got["scales"]), ref["s"])
        assert host(got["s_t"])[0] == ref["s_t"]
    # ... which hold transposed copies of the same values
    da = oracle.nv_dequantize_f64(ra["q"], ra["s"], ra["s_t"])
    db = oracle.nv_dequantize_f64(rb["q"], rb["s"], rb["s_t"])
    assert np.array_equal(da, db.T)


# ---------------------------------------------------------------------------
# FP4RowToFP8Col
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (640, 256), (128, 512), (256, 2560), (640, 1024)])
def test_fp4_row_to_fp8_col(fq, oracle, shape):
    R, C = shape
    rng = np.random.default_rng(R * 7 + C)
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    s = rng.integers(100, 160, (R, C // 32), dtype=np.uint8)
    s[::7] = rng.integers(0, 255, (len(s[::7]), C // 32), dtype=np.uint8)   # wide spreads: deep shifts, flushes
    y, ts = fq.fp4_row_to_fp8_col(dev(q), dev(s))
    yr, tsr = oracle.mx_to_fp8_col(q, s)
    assert np.array_equal(host(y), yr)
    assert np.array_equal(host(ts).view(np.uint32), tsr.view(np.uint32))


def test_fp4_row_to_fp8_col_full_size(fq, oracle):
    """The 8192x7168 FP8 activation after direct FP8 -> MXFP4, converted to the
    column (Wgrad) FP8 layout: bit-exact over the whole tensor."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    e4, ts = W.fp8_activation()
    qr, sr = oracle.fp8_to_mx(e4, ts)
    y, yts = fq.fp4_row_to_fp8_col(dev(qr), dev(sr))
    yr, ytsr = oracle.mx_to_fp8_col(qr, sr)
    assert np.array_equal(host(y), yr)
    assert np.array_equal(host(yts).view(np.uint32), ytsr.view(np.uint32))


def _grouped_col_run(fq, q, s, offs, G, canary=True):
    """Raw call of fp4q_fp4_row_to_fp8_col_grouped into canary-filled outputs of
    the documented size; returns host (y [C, ld], tile scales [C, ld/128])."""
    import torch
    R, C = q.shape[0], 2 * q.shape[1]
    ld = fq.fp4q_fp4_row_to_fp8_col_grouped_ld(R, G)
    y = torch.full((C, ld), 0xAB, dtype=torch.uint8, device="cuda")
    ts = torch.full((C, ld // 128), 7.0, dtype=torch.float32, device="cuda")
    fq.fp4q_fp4_row_to_fp8_col_grouped(dev(q), dev(s), R, C, dev(np.asarray(offs, dtype=np.int64)), G, y, ts)
    torch.cuda.synchronize()
    return host(y), host(ts)


def _check_grouped_col(oracle, y, ts, q, s, offs):
    yr, tsr = oracle.mx_to_fp8_col_grouped(q, s, offs)
    T = tsr.shape[1]
    assert np.array_equal(y[:, : 128 * T], yr)
    assert np.array_equal(ts[:, :T].view(np.uint32), tsr.view(np.uint32))
    assert np.all(y[:, 128 * T:] == 0xAB) and np.all(ts[:, T:] == 7.0)      # nothing written past the groups


@pytest.mark.parametrize("C", [128, 256, 2048])
def test_fp4_row_to_fp8_col_grouped(fq, oracle, C):
    """Ragged expert groups (empty, 1, 127-129, 255, 300 and 2 rows) and rows
    past the last offset: every group's tiles restart at its first row, its last
    tile is partial and padded with zeros, bit-exact against the oracle."""
    sizes = [0, 1, 127, 128, 129, 0, 255, 300, 2]
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = int(offs[-1]) + 9
    rng = np.random.default_rng(C + 5)
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    s = rng.integers(100, 160, (R, C // 32), dtype=np.uint8)
    s[::7] = rng.integers(0, 255, (len(s[::7]), C // 32), dtype=np.uint8)   # wide spreads: deep shifts, flushes
    y, ts = _grouped_col_run(fq, q, s, offs, len(sizes))
    _check_grouped_col(oracle, y, ts, q[: offs[-1]], s[: offs[-1]], offs)


def test_fp4_row_to_fp8_col_grouped_moe_size(fq, oracle):
    """8192 tokens routed top-8 over 64 experts (Zipf 1.1): the 65536
    dispatched rows of the 2048-wide expert activation h, converted to the
    column FP8 layout of the down-projection's weight gradient; every byte and
    tile scale checked."""
    from micro_scaled_fp4_gb300 import workloads as W
    topk = W.moe_routing(tokens=8192, experts=64, top_k=8, seed=33)
    _, offs = oracle.moe_dispatch(topk, 64)
    R, C = int(offs[-1]), 2048
    rng = np.random.default_rng(34)
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    s = rng.integers(110, 140, (R, C // 32), dtype=np.uint8)
    y, ts = _grouped_col_run(fq, q, s, offs, 64)
    _check_grouped_col(oracle, y, ts, q, s, offs)


def test_fp4_row_to_fp8_col_grouped_clamps_malformed_offsets(fq, oracle):
    """Offsets that decrease or run past `rows` are clamped (each into
    [previous offset, rows]) and give the result of the clamped offsets;
    nothing is written past the groups."""
    rng = np.random.default_rng(35)
    R, C = 350, 256
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    s = rng.integers(110, 140, (R, C // 32), dtype=np.uint8)
    y, ts = _grouped_col_run(fq, q, s, [0, 300, 100, 400, 50], 4)
    _check_grouped_col(oracle, y, ts, q, s, [0, 300, 300, 350, 350])


def test_widen_argument_errors(fq):
    import torch
    x = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((16, 32), dtype=torch.uint8, device="cuda")
    s = torch.zeros((16, 4), dtype=torch.uint8, device="cuda")
    f = torch.zeros(4, dtype=torch.float32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    cases = [
        (lambda: fq.fp4q_nv_quantize_2d(x, 8, 64, 64, 0, 0, None, f, f, q, s, 0, ws, 256), 2),       # rows % 16
        (lambda: fq.fp4q_nv_quantize(x, 16, 64, 64, 0, 0, 0, 0, 0, None, f, f, q, s, 0, ws, 256), 2),  # rows % 128
        (lambda: fq.fp4q_nv_quantize(x, 16, 64, 64, 1, 3, 0, 0, 0, None, f, f, q, s, 0, ws, 256), 1),  # rht 3
        (lambda: fq.fp4q_fp4_row_to_fp8_col(q, s, 16, 64, q, f), 2),                                   # rows % 128
        (lambda: fq.fp4q_mx_quantize(x, 1, None, 128, 128, 128, 0, q, s, 0), 2),                       # FP32 axis 0
    ]
    for fn, status in cases:
        with pytest.raises(fq.Fp4qError) as e:
            fn()
        assert e.value.status == status


# ---------------------------------------------------------------------------
# Wgrad with the deterministic H16: dW = dY^T X, both operands quantized along
# the token axis (column-wise) with the same rotation, NVFP4 GEMM
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rounding", [0, 1])
def test_wgrad_deterministic_h16(fq, oracle, rounding):
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    T, H, I = 512, 256, 384                       # tokens (K), output rows, output cols
    dy = W.gradient_bf16(T, H, seed=31)
    x = W.gradient_bf16(T, I, seed=32, scale=1.0)
    ra = fq.nv_quantize(dev_bf16(dy), rht=2, rounding=rounding, sr_seed=5, layout=fq.FP4Q_SCALES_MMA, block_axis=0)
    rb = fq.nv_quantize(dev_bf16(x), rht=2, rounding=rounding, sr_seed=6, layout=fq.FP4Q_SCALES_MMA, block_axis=0)
    d32 = fq.gemm(ra["q"], ra["scales"], rb["q"], rb["scales"], fq.FP4Q_NVFP4, ra["s_t"], rb["s_t"],
                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    oa = oracle.nv_quantize_col(dy, rht=2, rounding="sr" if rounding else "rne", sr_seed=5)
    ob = oracle.nv_quantize_col(x, rht=2, rounding="sr" if rounding else "rne", sr_seed=6)
    assert np.array_equal(host(ra["q"]), oa["q"]) and np.array_equal(host(rb["q"]), ob["q"])
    ref = oracle.nv_gemm_ref(oa["q"], oa["s"], oa["s_t"], ob["q"], ob["s"], ob["s_t"])
    assert rel_frobenius(host(d32).astype(np.float64), ref) <= 1e-3
    # the rotation cancels along the token axis: the product tracks dY^T X up to FP4 error
    exact = oracle.bf16_bits_to_f32(dy).astype(np.float64).T @ oracle.bf16_bits_to_f32(x).astype(np.float64)
    assert rel_frobenius(host(d32).astype(np.float64), exact) < 0.2


# ---------------------------------------------------------------------------
# the FP8 consumer: MXFP8 GEMM on the outputs of FP4 -> FP8 (row and column)
# ---------------------------------------------------------------------------
def _bf16_round(y):
    u = np.ascontiguousarray(y, dtype=np.float32).view(np.uint32)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def test_fp8_tile_scales_to_e8m0(fq):
    import torch
    ts = np.exp2(np.arange(-127, 128, dtype=np.float64)).astype(np.float32).reshape(5, 51)
    ts = np.concatenate([ts, np.full((5, 1), 2.0 ** 5, dtype=np.float32)], axis=1)      # [5, 52]
    s = torch.empty((5, 52 * 4), dtype=torch.uint8, device="cuda")
    fq.fp4q_device_status(reset=True)
    fq.fp4q_fp8_tile_scales_to_e8m0(dev(ts), 5, 52 * 128, s, 0)
    want = np.repeat(np.log2(ts.astype(np.float64)).astype(np.int64) + 127, 4, axis=1)
    assert np.array_equal(host(s).astype(np.int64), want)
    assert fq.fp4q_device_status() == 0
    bad = ts.copy()
    bad[2, 3] = 3.0                                            # not a power of two
    fq.fp4q_fp8_tile_scales_to_e8m0(dev(bad), 5, 52 * 128, s, 0)
    assert fq.fp4q_device_status(reset=True) & 8          # bit 3: a scale it could not convert
    assert np.all(host(s)[2, 12:16] == 0xFF)
    assert fq.fp4q_device_status() == 0


@pytest.mark.parametrize("shape", [(200, 300, 256), (128, 256, 1024), (1000, 512, 384)])
def test_mxfp8_gemm_on_fp4_to_fp8_outputs(fq, oracle, shape):
    """Forward-style FP8 GEMM: both operands stored MXFP4, expanded by the
    bit-remap FP4 -> FP8 conversion, multiplied as MXFP8 on the tensor cores."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    M, N, K = shape
    rng = np.random.default_rng(M + N + K)
    a = W.to_bf16_bits((rng.standard_normal((M, K)) * np.exp2(rng.integers(-4, 4, (M, 1)))).astype(np.float32))
    b = W.to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    qa, sa = fq.mx_quantize(dev_bf16(a))
    qb, sb = fq.mx_quantize(dev_bf16(b))
    ya, tsa = fq.fp4_to_fp8(qa, sa)
    yb, tsb = fq.fp4_to_fp8(qb, sb)
    d32 = fq.gemm(ya, fq.fp8_mma_scales(tsa), yb, fq.fp8_mma_scales(tsb), fq.FP4Q_MXFP8, out_dtype=torch.float32)
    d16 = fq.gemm(ya, fq.fp8_mma_scales(tsa), yb, fq.fp8_mma_scales(tsb), fq.FP4Q_MXFP8, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    # the oracle's own operands (the kernels' equal them bit for bit)
    qra, sra = oracle.mx_quantize(a)
    qrb, srb = oracle.mx_quantize(b)
    yra, tsra = oracle.mx_to_fp8(qra, sra)
    yrb, tsrb = oracle.mx_to_fp8(qrb, srb)
    assert np.array_equal(host(ya), yra) and np.array_equal(host(yb), yrb)
    assert np.array_equal(host(tsa).view(np.uint32), tsra.view(np.uint32))
    assert np.array_equal(host(tsb).view(np.uint32), tsrb.view(np.uint32))
    ref = oracle.fp8_gemm_ref(yra, tsra, yrb, tsrb)
    assert rel_frobenius(host(d32).astype(np.float64), ref) <= 1e-3
    assert rel_frobenius(host(d16.float()).astype(np.float64), _bf16_round(ref)) <= 1e-3
    # the BF16 epilogue writes the nearest-even BF16 of the FP32 result, every element in place
    assert torch.equal(d16, d32.to(torch.bfloat16))
    # lossless chain: the FP8 operands are the MXFP4 values, so this is also the MXFP4 product
    mx = oracle.mx_gemm_ref(qra, sra, qrb, srb)
    assert oracle.rel_frobenius(ref, mx) < 1e-12


def test_mxfp8_gemm_banded_tile_order(fq, oracle):
    """An A operand too large for L2 (4224 x 12288 E4M3, 52 MB) runs the dense
    GEMM's banded tile order: a full band of 32 m-tiles, a band of one, and a
    ragged last n-tile.  Sampled rows from both bands, every column."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    M, N, K = 4224, 640, 12288
    rng = np.random.default_rng(51)
    a = W.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    b = W.to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    ya, tsa = fq.fp4_to_fp8(*fq.mx_quantize(dev_bf16(a)))
    yb, tsb = fq.fp4_to_fp8(*fq.mx_quantize(dev_bf16(b)))
    d = fq.gemm(ya, fq.fp8_mma_scales(tsa), yb, fq.fp8_mma_scales(tsb), fq.FP4Q_MXFP8, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    rows = np.sort(np.concatenate([rng.choice(4096, 40, replace=False), 4096 + np.arange(0, 128, 16)]))
    yra, tsra = oracle.mx_to_fp8(*oracle.mx_quantize(a[rows]))      # row-local: only the sampled rows
    yrb, tsrb = oracle.mx_to_fp8(*oracle.mx_quantize(b))
    assert np.array_equal(host(ya)[rows], yra) and np.array_equal(host(yb), yrb)
    ref = oracle.fp8_gemm_ref(yra, tsra, yrb, tsrb)
    assert rel_frobenius(host(d)[rows].astype(np.float64), ref) <= 1e-3


def test_mxfp8_wgrad_on_fp4_row_to_fp8_col(fq, oracle):
    """Backward-style FP8 GEMM: dW = dY^T X with both operands converted by
    FP4RowToFP8Col from their row-wise MXFP4 storage (tokens become K)."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    T, H, I = 512, 256, 384
    rng = np.random.default_rng(41)
    dy = W.to_bf16_bits((rng.standard_t(3, (T, H)) * 1e-3).astype(np.float32))
    x = W.to_bf16_bits(rng.standard_normal((T, I)).astype(np.float32))
    qd, sd = fq.mx_quantize(dev_bf16(dy))
    qx, sx = fq.mx_quantize(dev_bf16(x))
    yd, tsd = fq.fp4_row_to_fp8_col(qd, sd)            # [H, T]
    yx, tsx = fq.fp4_row_to_fp8_col(qx, sx)            # [I, T]
    d32 = fq.gemm(yd, fq.fp8_mma_scales(tsd), yx, fq.fp8_mma_scales(tsx), fq.FP4Q_MXFP8, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    # the oracle's own operands (the kernels' equal them bit for bit)
    qrd, srd = oracle.mx_quantize(dy)
    qrx, srx = oracle.mx_quantize(x)
    yrd, tsrd = oracle.mx_to_fp8_col(qrd, srd)
    yrx, tsrx = oracle.mx_to_fp8_col(qrx, srx)
    assert np.array_equal(host(yd), yrd) and np.array_equal(host(yx), yrx)
    assert np.array_equal(host(tsd).view(np.uint32), tsrd.view(np.uint32))
    assert np.array_equal(host(tsx).view(np.uint32), tsrx.view(np.uint32))
    ref = oracle.fp8_gemm_ref(yrd, tsrd, yrx, tsrx)
    assert rel_frobenius(host(d32).astype(np.float64), ref) <= 1e-3
    # and it is dY_mx^T X_mx of the stored MXFP4 values (no flush at these spreads)
    exact = oracle.mx_dequantize_f64(qrd, srd).T @ oracle.mx_dequantize_f64(qrx, srx)
    assert oracle.rel_frobenius(ref, exact) < 1e-9
