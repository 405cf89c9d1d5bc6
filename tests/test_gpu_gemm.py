"""GPU parity of the tcgen05 block-scaled FP4 GEMM against the float64 oracle.

D = A . B^T with both operands FP4 along K ("Pretraining large language
models with MXFP4 on Native FP4 Hardware", investigation section: Fprop
Y = X W^T).  Gate: relative Frobenius error <= 1e-3 against float64 matmul of
the dequantized operands, for FP32 output directly and for BF16 output
against the BF16 rounding of the float64 result (BF16 rounding alone is
~1.5e-3 relative, so the unrounded comparison is reported, not gated).
"""
import numpy as np
import pytest

from _helpers import dev_bf16, from_mma_layout, host, rel_frobenius

pytestmark = pytest.mark.gpu

TOL = 1e-3


@pytest.fixture(scope="module")
def fq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import micro_scaled_fp4_gb300.fp4q as fq
    fq.load()
    return fq


def _bf16_round(y: np.ndarray) -> np.ndarray:
    import torch
    return torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _operands(M, N, K, seed):
    from micro_scaled_fp4_gb300 import workloads as W
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K)).astype(np.float32)
    a[rng.choice(M, max(1, M // 200), replace=False)] *= 40.0
    b = rng.standard_normal((N, K)).astype(np.float32)
    return W.to_bf16_bits(a), W.to_bf16_bits(b)


def _same_operand(q_dev, s_dev, q_ref, s_ref, rows, scale_cols):
    """The kernel's quantized operand (MMA-layout scales) equals the oracle's."""
    assert np.array_equal(host(q_dev), q_ref)
    assert np.array_equal(from_mma_layout(host(s_dev), rows, scale_cols), s_ref)


def _check(oracle, d_bf16, d_f32, ref):
    e32 = rel_frobenius(host(d_f32).astype(np.float64), ref)
    import torch
    eb = rel_frobenius(host(d_bf16.float()).astype(np.float64), _bf16_round(ref))
    assert e32 <= TOL, e32
    assert eb <= TOL, eb
    # the BF16 epilogue writes the nearest-even BF16 of the FP32 result, every element in place
    assert torch.equal(d_bf16, d_f32.to(torch.bfloat16))
    return e32, eb


# M <= 128 runs on single CTAs, larger M on CTA pairs (256-row tiles over two
# SMs): one whole pair tile; three m-tiles (the last pair's second CTA past
# the end) with an N tail and a half last K stage; a single row; N = 4 x 256
# + 8; a lone 128-element K stage.
SHAPES = [(256, 256, 256), (128, 256, 256), (128, 256, 128), (200, 300, 384), (384, 136, 640), (1000, 520, 1024),
          (64, 64, 512), (512, 2048, 2048), (1, 1032, 256), (3, 136, 128)]


@pytest.mark.parametrize("shape", SHAPES)
def test_mxfp4_gemm(fq, oracle, shape):
    import torch
    M, N, K = shape
    a, b = _operands(M, N, K, M + N + K)
    qa, sa = fq.mx_quantize(dev_bf16(a), layout=fq.FP4Q_SCALES_MMA)
    qb, sb = fq.mx_quantize(dev_bf16(b), layout=fq.FP4Q_SCALES_MMA)
    d32 = fq.gemm(qa, sa, qb, sb, fq.FP4Q_MXFP4, out_dtype=torch.float32)
    d16 = fq.gemm(qa, sa, qb, sb, fq.FP4Q_MXFP4, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    # the reference multiplies the oracle's own operands (equal to the kernel's)
    qra, sra = oracle.mx_quantize(a)
    qrb, srb = oracle.mx_quantize(b)
    _same_operand(qa, sa, qra, sra, M, K // 32)
    _same_operand(qb, sb, qrb, srb, N, K // 32)
    _check(oracle, d16, d32, oracle.mx_gemm_ref(qra, sra, qrb, srb))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("rht", [False, True])
def test_nvfp4_gemm(fq, oracle, shape, rht):
    import torch
    M, N, K = shape
    a, b = _operands(M, N, K, 3 * M + N + K)
    ra = fq.nv_quantize(dev_bf16(a), rht=rht, rht_seed=7, layout=fq.FP4Q_SCALES_MMA)
    rb = fq.nv_quantize(dev_bf16(b), rht=rht, rht_seed=7, layout=fq.FP4Q_SCALES_MMA)
    args = (ra["q"], ra["scales"], rb["q"], rb["scales"], fq.FP4Q_NVFP4, ra["s_t"], rb["s_t"])
    d32 = fq.gemm(*args, out_dtype=torch.float32)
    d16 = fq.gemm(*args, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    oa = oracle.nv_quantize(a, rht=rht, rht_seed=7)
    ob = oracle.nv_quantize(b, rht=rht, rht_seed=7)
    _same_operand(ra["q"], ra["scales"], oa["q"], oa["s"], M, K // 16)
    _same_operand(rb["q"], rb["scales"], ob["q"], ob["s"], N, K // 16)
    assert host(ra["s_t"])[0] == oa["s_t"] and host(rb["s_t"])[0] == ob["s_t"]
    ref = oracle.nv_gemm_ref(oa["q"], oa["s"], oa["s_t"], ob["q"], ob["s"], ob["s_t"])
    _check(oracle, d16, d32, ref)
    if rht and M * N <= 2 ** 20:
        # the rotation cancels along K: the product tracks the unrotated A . B^T
        # up to the FP4 quantization error (reported bound, not the kernel's)
        exact = oracle.bf16_bits_to_f32(a).astype(np.float64) @ oracle.bf16_bits_to_f32(b).astype(np.float64).T
        assert rel_frobenius(host(d32), exact) < 0.2


@pytest.mark.parametrize("case", range(9))
def test_gemm_random_shapes(fq, oracle, case):
    """Seeded random M, N in [1, 900) and K a multiple of 128 up to 1152, for
    MXFP4, NVFP4 and NVFP4 with RHT operands (case % 3): operands equal to the
    oracle's, FP32 and BF16 outputs within 1e-3 of the float64 product."""
    import torch
    rng = np.random.default_rng(7000 + case)
    M, N, K = int(rng.integers(1, 900)), int(rng.integers(1, 900)), 128 * int(rng.integers(1, 10))
    a, b = _operands(M, N, K, 8000 + case)
    if case % 3 == 0:
        qa, sa = fq.mx_quantize(dev_bf16(a), layout=fq.FP4Q_SCALES_MMA)
        qb, sb = fq.mx_quantize(dev_bf16(b), layout=fq.FP4Q_SCALES_MMA)
        args = (qa, sa, qb, sb, fq.FP4Q_MXFP4)
        qra, sra = oracle.mx_quantize(a)
        qrb, srb = oracle.mx_quantize(b)
        _same_operand(qa, sa, qra, sra, M, K // 32)
        _same_operand(qb, sb, qrb, srb, N, K // 32)
        ref = oracle.mx_gemm_ref(qra, sra, qrb, srb)
    else:
        rht = case % 3 == 2
        ra = fq.nv_quantize(dev_bf16(a), rht=rht, rht_seed=9, layout=fq.FP4Q_SCALES_MMA)
        rb = fq.nv_quantize(dev_bf16(b), rht=rht, rht_seed=9, layout=fq.FP4Q_SCALES_MMA)
        args = (ra["q"], ra["scales"], rb["q"], rb["scales"], fq.FP4Q_NVFP4, ra["s_t"], rb["s_t"])
        oa = oracle.nv_quantize(a, rht=rht, rht_seed=9)
        ob = oracle.nv_quantize(b, rht=rht, rht_seed=9)
        _same_operand(ra["q"], ra["scales"], oa["q"], oa["s"], M, K // 16)
        _same_operand(rb["q"], rb["scales"], ob["q"], ob["s"], N, K // 16)
        ref = oracle.nv_gemm_ref(oa["q"], oa["s"], oa["s_t"], ob["q"], ob["s"], ob["s_t"])
    d32 = fq.gemm(*args, out_dtype=torch.float32)
    d16 = fq.gemm(*args, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    _check(oracle, d16, d32, ref)


def test_gemm_full_size(fq, oracle):
    """8192^3, MXFP4 (A with 0.5 % outlier rows x40) and NVFP4 with the RHT on
    both operands, BF16 output as the benchmark runs it.  Every code and scale
    of both operands equals the oracle's quantization of the whole tensors,
    and the whole output is within 1e-3 of the BF16 rounding of the float64
    product of the oracle's operands."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    a, b = W.gemm_operands()
    ad, bd = dev_bf16(a), dev_bf16(b)
    M = N = K = 8192
    qa, sa = fq.mx_quantize(ad, layout=fq.FP4Q_SCALES_MMA)
    qb, sb = fq.mx_quantize(bd, layout=fq.FP4Q_SCALES_MMA)
    d = fq.gemm(qa, sa, qb, sb, fq.FP4Q_MXFP4)
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    qra, sra = oracle.mx_quantize(a)
    qrb, srb = oracle.mx_quantize(b)
    assert np.array_equal(host(qa), qra) and np.array_equal(from_mma_layout(host(sa), M, K // 32), sra)
    assert np.array_equal(host(qb), qrb) and np.array_equal(from_mma_layout(host(sb), N, K // 32), srb)
    del qa, sa, qb, sb
    ref = oracle.mx_gemm_ref(qra, sra, qrb, srb)
    assert rel_frobenius(host(d.float()), _bf16_round(ref)) <= TOL
    del ref, qra, sra, qrb, srb
    ra = fq.nv_quantize(ad, rht=True, rht_seed=7, layout=fq.FP4Q_SCALES_MMA)
    rb = fq.nv_quantize(bd, rht=True, rht_seed=7, layout=fq.FP4Q_SCALES_MMA)
    d = fq.gemm(ra["q"], ra["scales"], rb["q"], rb["scales"], fq.FP4Q_NVFP4, ra["s_t"], rb["s_t"])
    torch.cuda.synchronize()
    assert fq.fp4q_device_status() == 0
    oa = oracle.nv_quantize(a, rht=True, rht_seed=7)
    ob = oracle.nv_quantize(b, rht=True, rht_seed=7)
    assert np.array_equal(host(ra["q"]), oa["q"]) and np.array_equal(from_mma_layout(host(ra["scales"]), M, K // 16), oa["s"])
    assert np.array_equal(host(rb["q"]), ob["q"]) and np.array_equal(from_mma_layout(host(rb["scales"]), N, K // 16), ob["s"])
    assert host(ra["s_t"])[0] == oa["s_t"] and host(rb["s_t"])[0] == ob["s_t"]
    ref = oracle.nv_gemm_ref(oa["q"], oa["s"], oa["s_t"], ob["q"], ob["s"], ob["s_t"])
    assert rel_frobenius(host(d.float()), _bf16_round(ref)) <= TOL


def test_gemm_argument_errors(fq):
    import torch
    q = torch.zeros((128, 64), dtype=torch.uint8, device="cuda")
    s = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    d = torch.zeros((128, 128), dtype=torch.float32, device="cuda")
    A = fq.make_operand(q, s, fq.FP4Q_MXFP4)
    B = fq.make_operand(q, s, fq.FP4Q_NVFP4)
    with pytest.raises(fq.Fp4qError) as e:
        fq.fp4q_block_scaled_gemm(A, B, 128, 128, 128, d, fq.FP4Q_FP32, 128)
    assert e.value.status == 1
    with pytest.raises(fq.Fp4qError) as e:
        fq.fp4q_block_scaled_gemm(A, A, 128, 128, 96, d, fq.FP4Q_FP32, 128)
    assert e.value.status == 2
    with pytest.raises(fq.Fp4qError) as e:
        fq.fp4q_block_scaled_gemm(A, A, 128, 128, 128, d.data_ptr() + 4, fq.FP4Q_FP32, 128)
    assert e.value.status == 3
