"""Seeded random-shape sweep of the streaming entry points against the oracle.

The fixed-shape tests pin each path's corner cases; this sweep draws further
shapes inside each call's documented constraints (one seed per case, printed
in the test id), so that row tails, column counts that leave partial warps or
CTAs, and odd block counts are exercised beyond the hand-picked ones.  Every
comparison is bit-exact: codes, scales, tensor scales, FP8 bytes.
"""
import numpy as np
import pytest

from _helpers import dev, dev_bf16, from_mma_layout, host

pytestmark = pytest.mark.gpu

CASES = range(8)


@pytest.fixture(scope="module")
def fq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import micro_scaled_fp4_gb300.fp4q as fq
    fq.load()
    return fq


def _bf16(rng, rows, cols):
    from micro_scaled_fp4_gb300 import workloads as W
    x = (rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-30, 30, (rows, 1)))).astype(np.float32)
    x[:, rng.integers(0, cols)] *= np.float32(40.0)            # an outlier column
    return W.to_bf16_bits(x)


@pytest.mark.parametrize("case", CASES)
def test_sweep_mx_quantize_and_dequantize(fq, oracle, case):
    """BF16 -> MXFP4 in both scale layouts, then MXFP4 -> BF16 and FP32."""
    import torch
    rng = np.random.default_rng(1000 + case)
    R, C = int(rng.integers(1, 700)), 32 * int(rng.integers(1, 300))
    x = _bf16(rng, R, C)
    qr, sr = oracle.mx_quantize(x)
    for layout in (0, 1):
        q, s = fq.mx_quantize(dev_bf16(x), layout=layout)
        assert np.array_equal(host(q), qr), (R, C, layout)
        sg = host(s)
        assert np.array_equal(from_mma_layout(sg, R, C // 32) if layout else sg, sr), (R, C, layout)
    q, s = fq.mx_quantize(dev_bf16(x))
    yr32, yr16 = oracle.mx_dequantize(qr, sr)
    y32 = fq.mx_dequantize(q, s, dtype=torch.float32)
    assert np.array_equal(host(y32).view(np.uint32), yr32.view(np.uint32)), (R, C)
    y16 = fq.mx_dequantize(q, s, dtype=torch.bfloat16)
    assert np.array_equal(host(y16.view(torch.int16)).view(np.uint16), yr16), (R, C)


@pytest.mark.parametrize("case", CASES)
def test_sweep_fp8_to_mx_and_back(fq, oracle, case):
    """E4M3 + 1x128 tile scales -> MXFP4 (direct) -> FP8 with tile scales."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    rng = np.random.default_rng(2000 + case)
    R, C = int(rng.integers(1, 900)), 128 * int(rng.integers(1, 70))
    e4, ts = W.fp8_activation(R, C, seed=3000 + case, outlier_seed=case)
    q, s = fq.mx_quantize(dev(e4).view(torch.float8_e4m3fn), tile_scale=dev(ts))
    qr, sr = oracle.fp8_to_mx(e4, ts)
    assert np.array_equal(host(q), qr) and np.array_equal(host(s), sr), (R, C)
    y, yts = fq.fp4_to_fp8(q, s)
    yr, ytsr = oracle.mx_to_fp8(qr, sr)
    assert np.array_equal(host(y), yr), (R, C)
    assert np.array_equal(host(yts).view(np.uint32), ytsr.view(np.uint32)), (R, C)


@pytest.mark.parametrize("case", CASES)
def test_sweep_nv_quantize(fq, oracle, case):
    """BF16 -> NVFP4 with a drawn rotation mode (none, random signs, H16) and
    rounding (RNE, SR), in a drawn scale layout."""
    from micro_scaled_fp4_gb300 import workloads as W
    rng = np.random.default_rng(4000 + case)
    R, C = int(rng.integers(1, 500)), 16 * int(rng.integers(1, 500))
    rht, rounding, layout = int(rng.integers(0, 3)), int(rng.integers(0, 2)), int(rng.integers(0, 2))
    x = W.gradient_bf16(R, C, seed=5000 + case)
    r = fq.nv_quantize(dev_bf16(x), rht=rht, rht_seed=11 + case, rounding=rounding, sr_seed=77 + case,
                       layout=layout)
    ref = oracle.nv_quantize(x, rht=rht, rht_seed=11 + case, rounding="sr" if rounding else "rne",
                             sr_seed=77 + case)
    what = (R, C, rht, rounding, layout)
    assert host(r["amax"])[0] == ref["amax"] and host(r["s_t"])[0] == ref["s_t"], what
    assert np.array_equal(host(r["q"]), ref["q"]), what
    sg = host(r["scales"])
    assert np.array_equal(from_mma_layout(sg, R, C // 16) if layout else sg, ref["s"]), what


@pytest.mark.parametrize("case", CASES)
def test_sweep_column_paths(fq, oracle, case):
    """FP4RowToFP8Col (rows, cols multiples of 128) and column-wise MXFP4 of
    BF16 (block axis 0) on drawn shapes."""
    rng = np.random.default_rng(6000 + case)
    R, C = 128 * int(rng.integers(1, 7)), 128 * int(rng.integers(1, 24))
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    s = rng.integers(100, 160, (R, C // 32), dtype=np.uint8)
    y, ts = fq.fp4_row_to_fp8_col(dev(q), dev(s))
    yr, tsr = oracle.mx_to_fp8_col(q, s)
    assert np.array_equal(host(y), yr), (R, C)
    assert np.array_equal(host(ts).view(np.uint32), tsr.view(np.uint32)), (R, C)
    x = _bf16(rng, R, C)
    qc, sc = fq.mx_quantize(dev_bf16(x), block_axis=0)
    qcr, scr = oracle.mx_quantize_col(x)
    assert np.array_equal(host(qc), qcr) and np.array_equal(host(sc), scr), (R, C)
