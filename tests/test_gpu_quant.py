"""GPU parity of the streaming kernels against the oracle (bit-exact).

MXFP4 quantize / dequantize, direct FP8 -> MXFP4, scaled MXFP4 -> FP8 and
NVFP4 quantize (RHT, RNE, SR), called through the C ABI on the same seeded
inputs as the oracle, at sizes that span several CTAs and ragged row tails,
and at the full workload sizes the benchmark times.
"""
import numpy as np
import pytest

from _helpers import dev, dev_bf16, from_mma_layout, host, unpack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import micro_scaled_fp4_gb300.fp4q as fq
    fq.load()
    return fq


# ---------------------------------------------------------------------------
# hardware rounding instructions against the oracle's rounding rules
# ---------------------------------------------------------------------------
def test_e2m1_rounding_every_fp32_in_range(fq, oracle):
    """Every FP32 pattern with |v| in [2^-6, 8), both signs, quantized in blocks
    whose first element is 4.0 (so E = 0 and the code is the rounding of v
    itself): GPU codes == oracle round-to-nearest-even codes."""
    import torch
    lo_bits, hi_bits = (127 - 6) << 23, (127 + 3) << 23
    chunk = 31 * (1 << 19)
    for sign in (0, 1):
        for start in range(lo_bits, hi_bits, chunk):
            bits = np.arange(start, min(start + chunk, hi_bits), dtype=np.uint32) | np.uint32(sign << 31)
            v = bits.view(np.float32)
            nblk = (v.size + 30) // 31
            x = np.zeros((nblk, 32), dtype=np.float32)
            x[:, 0] = 4.0
            flat = x[:, 1:].reshape(-1)
            flat[: v.size] = v
            x[:, 1:] = flat.reshape(nblk, 31)
            xd = dev(x.reshape(-1, 256) if nblk % 8 == 0 else x)
            q, s = fq.mx_quantize(xd)
            torch.cuda.synchronize()
            codes = unpack(host(q)).reshape(nblk, 32)
            assert np.all(host(s).reshape(-1) == 127)
            got = codes[:, 1:].reshape(-1)[: v.size]
            assert np.array_equal(got, oracle.e2m1_rne(v)), hex(start)


def test_e4m3_scale_rounding_all_bf16_block_amax(fq, oracle):
    """NVFP4 block scale = E4M3 RNE-satfinite of blockamax / (6 s_t): every
    finite BF16 value as the block's only non-zero element, several tensor
    amax values supplied by the caller."""
    import torch
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_bits_to_f32(b)
    b = b[np.isfinite(f)]
    x = np.zeros((b.size, 16), dtype=np.uint16)
    x[:, 5] = b
    xd = dev_bf16(x)
    for amax in (1.0, 3.0e-3, 2.5e4, 1e-30):
        r = fq.nv_quantize(xd, amax=torch.tensor([amax], dtype=torch.float32, device="cuda"))
        ref = oracle.nv_quantize(x, amax=np.float32(amax))
        assert np.array_equal(host(r["scales"]), ref["s"]), amax
        assert np.array_equal(host(r["q"]), ref["q"]), amax
        assert host(r["s_t"])[0] == ref["s_t"]


# ---------------------------------------------------------------------------
# MXFP4 quantize / dequantize
# ---------------------------------------------------------------------------
SHAPES = [(1, 32), (3, 96), (256, 4096), (129, 7168), (70, 2048 + 32), (5, 14336)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_mx_quantize_bf16(fq, oracle, shape, layout):
    from micro_scaled_fp4_gb300 import workloads as W
    R, C = shape
    rng = np.random.default_rng(R * 7 + C)
    x32 = (rng.standard_normal((R, C)) * np.exp2(rng.integers(-40, 40, (R, 1)))).astype(np.float32)
    x32[0, :32] = 0.0                      # an all-zero block
    if R > 2:
        x32[2, :] *= np.float32(1e-38)     # subnormal values
    x = W.to_bf16_bits(x32)
    q, s = fq.mx_quantize(dev_bf16(x), layout=layout)
    qr, sr = oracle.mx_quantize(x)
    assert np.array_equal(host(q), qr)
    sg = host(s)
    assert np.array_equal(from_mma_layout(sg, R, C // 32) if layout else sg, sr)


def test_mx_quantize_bf16_strided(fq, oracle):
    from micro_scaled_fp4_gb300 import workloads as W
    x = W.activation_bf16(64, 1024 + 256, seed=3)
    xd = dev_bf16(x)[:, 128:128 + 1024]          # ld_x = 1280 elements
    q, s = fq.mx_quantize(xd)
    qr, sr = oracle.mx_quantize(np.ascontiguousarray(x[:, 128:128 + 1024]))
    assert np.array_equal(host(q), qr) and np.array_equal(host(s), sr)


@pytest.mark.parametrize("shape", [(3, 96), (256, 4096), (129, 2048)])
def test_mx_quantize_fp32(fq, oracle, shape):
    R, C = shape
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((R, C)) * np.exp2(rng.integers(-60, 60, (R, C // 32)).repeat(32, 1))).astype(np.float32)
    q, s = fq.mx_quantize(dev(x))
    qr, sr = oracle.mx_quantize(x)
    assert np.array_equal(host(q), qr) and np.array_equal(host(s), sr)


def test_mx_roundtrip_c1(fq, oracle):
    """256x4096 BF16 N(0,1), seed 0: quantize then dequantize (BF16 and FP32)."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    x = W.activation_bf16()
    q, s = fq.mx_quantize(dev_bf16(x))
    yb = fq.mx_dequantize(q, s, torch.bfloat16)
    yf = fq.mx_dequantize(q, s, torch.float32)
    rf, rb = oracle.mx_dequantize(*oracle.mx_quantize(x))
    assert np.array_equal(host(yb.view(torch.int16)).view(np.uint16), rb)
    assert np.array_equal(host(yf), rf)
    # quantize(dequantize(q)) == q
    q2, s2 = fq.mx_quantize(yb)
    assert torch.equal(q2, q) and torch.equal(s2, s)


def test_mx_dequantize_edge_scales(fq, oracle):
    import torch
    rng = np.random.default_rng(2)
    q = rng.integers(0, 256, (8, 64), dtype=np.uint8)
    s = np.array([[0, 1, 2, 127], [126, 125, 200, 250], [254, 253, 130, 3], [10, 20, 30, 40]] * 2, dtype=np.uint8)
    yf = fq.mx_dequantize(dev(q), dev(s), torch.float32)
    yb = fq.mx_dequantize(dev(q), dev(s), torch.bfloat16)
    rf, rb = oracle.mx_dequantize(q, s)
    assert np.array_equal(host(yf).view(np.uint32), rf.view(np.uint32))
    assert np.array_equal(host(yb.view(torch.int16)).view(np.uint16), rb)


# ---------------------------------------------------------------------------
# Direct FP8 -> MXFP4 and scaled MXFP4 -> FP8
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(1, 128), (37, 1024), (300, 7168)])
def test_fp8_to_mx_and_back(fq, oracle, shape):
    from micro_scaled_fp4_gb300 import workloads as W
    R, C = shape
    e4, ts = W.fp8_activation(R, C, seed=R, outlier_seed=C)
    q, s = fq.mx_quantize(dev(e4).view(__import__("torch").float8_e4m3fn), tile_scale=dev(ts))
    qr, sr = oracle.fp8_to_mx(e4, ts)
    assert np.array_equal(host(q), qr) and np.array_equal(host(s), sr)
    y, yts = fq.fp4_to_fp8(q, s)
    yr, ytsr = oracle.mx_to_fp8(qr, sr)
    assert np.array_equal(host(y), yr)
    assert np.array_equal(host(yts).view(np.uint32), ytsr.view(np.uint32))


@pytest.mark.parametrize("shape", [(37, 1024), (300, 7168), (3, 640), (3, 16384), (130, 2560)])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("pad", [0, 512])
def test_fp8_to_mx_layouts_strides_paths(fq, oracle, shape, layout, pad):
    """E4M3 -> MXFP4 and back on every launch form: shapes whose rows go through
    the shared-memory ring (cols % 512 == 0, a row that fits a stage) and shapes
    that take the register path (cols 640; 16384-wide E4M3 rows), row-major and
    MMA scale layouts, dense and padded rows (ld_x = cols + pad)."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    R, C = shape
    e4, ts = W.fp8_activation(R, C, seed=R + pad, outlier_seed=C + layout)
    big = np.zeros((R, C + pad), dtype=np.uint8)
    big[:, :C] = e4
    xd = dev(big)[:, :C].view(torch.float8_e4m3fn)
    q, s = fq.mx_quantize(xd, tile_scale=dev(ts), layout=layout)
    qr, sr = oracle.fp8_to_mx(e4, ts)
    assert np.array_equal(host(q), qr)
    got = host(s).reshape(-1)
    if layout:
        got = from_mma_layout(got, R, C // 32)
    assert np.array_equal(got.reshape(R, C // 32), sr)
    y, yts = fq.fp4_to_fp8(dev(qr), dev(sr))
    yr, ytsr = oracle.mx_to_fp8(qr, sr)
    assert np.array_equal(host(y), yr)
    assert np.array_equal(host(yts).view(np.uint32), ytsr.view(np.uint32))


def test_fp4_to_fp8_every_shift(fq, oracle):
    """Random codes under block exponents spread over the whole E8M0 range, so
    every shift d in [-254, 0] and every code meets the kernel's remap."""
    rng = np.random.default_rng(3)
    R, C = 512, 1024
    q = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    s = rng.integers(0, 255, (R, C // 32), dtype=np.uint8)
    s[:, ::8] = 254
    s[::3, 1::8] = 0
    s[1::5] = (s[1::5] % 14) + 120          # small spreads: the exact/subnormal region
    y, ts = fq.fp4_to_fp8(dev(q), dev(s))
    yr, tsr = oracle.mx_to_fp8(q, s)
    assert np.array_equal(host(y), yr)
    assert np.array_equal(host(ts).view(np.uint32), tsr.view(np.uint32))


def test_fp8_pipeline_full_size(fq, oracle):
    """8192x7168 E4M3 activation (0.5 % outlier columns x40, 1x128 tile scales):
    direct FP8 -> MXFP4, then MXFP4 -> FP8, both bit-exact over the whole tensor."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    e4, ts = W.fp8_activation()
    q, s = fq.mx_quantize(dev(e4).view(torch.float8_e4m3fn), tile_scale=dev(ts))
    y, yts = fq.fp4_to_fp8(q, s)
    qr, sr = oracle.fp8_to_mx(e4, ts)
    assert np.array_equal(host(q), qr) and np.array_equal(host(s), sr)
    yr, ytsr = oracle.mx_to_fp8(qr, sr)
    assert np.array_equal(host(y), yr)
    assert np.array_equal(host(yts).view(np.uint32), ytsr.view(np.uint32))
    # lossless: the FP8 copy represents the MXFP4 values exactly (no flush here)
    e8 = oracle.e4m3_values()[yr[:64]] * np.repeat(ytsr[:64].astype(np.float64), 128, axis=1)
    assert np.array_equal(e8, oracle.mx_dequantize_f64(qr[:64], sr[:64]))


# ---------------------------------------------------------------------------
# the FP8 path on host buffers (chunked, copies overlapped on streams)
# ---------------------------------------------------------------------------
def _check_host_outputs(out, qr, sr, yr, ytr):
    assert np.array_equal(out["q"].numpy(), qr)
    assert np.array_equal(out["scales"].numpy(), sr)
    assert np.array_equal(out["y"].numpy(), yr)
    assert np.array_equal(out["y_tile_scale"].numpy().view(np.uint32), ytr.view(np.uint32))


@pytest.mark.parametrize("rows,cols,chunk", [(1000, 1024, 256), (5, 512, 0), (300, 7168, 1000), (777, 256, 64)])
@pytest.mark.parametrize("pinned", [True, False])
def test_fp8_pipeline_host(fq, oracle, rows, cols, chunk, pinned):
    """Host E4M3 + tile scales -> host MXFP4 and FP8, in chunks (ragged last
    chunk, chunk larger than the tensor, default chunk), pinned or pageable
    host memory: bit-identical to the oracle."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    e4, ts = W.fp8_activation(rows, cols, seed=rows + cols)
    hx, ht = torch.from_numpy(e4), torch.from_numpy(ts)
    if pinned:
        hx, ht = hx.pin_memory(), ht.pin_memory()
    out = fq.fp8_pipeline_host(hx, ht, chunk_rows=chunk, pinned=pinned)
    qr, sr = oracle.fp8_to_mx(e4, ts)
    yr, ytr = oracle.mx_to_fp8(qr, sr)
    _check_host_outputs(out, qr, sr, yr, ytr)


def test_fp8_pipeline_host_back_to_back_calls(fq, oracle):
    """Two calls queued on one stream before any synchronisation reuse the
    workspace slots: each call's results are its own."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    R, C, chunk = 700, 2048, 128
    wsb = fq.fp4q_fp8_pipeline_host_workspace_bytes(C, chunk)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    runs = []
    for seed in (3, 4):
        e4, ts = W.fp8_activation(R, C, seed=seed)
        hx, ht = torch.from_numpy(e4).pin_memory(), torch.from_numpy(ts).pin_memory()
        out = {"q": torch.empty((R, C // 2), dtype=torch.uint8).pin_memory(),
               "scales": torch.empty((R, C // 32), dtype=torch.uint8).pin_memory(),
               "y": torch.empty((R, C), dtype=torch.uint8).pin_memory(),
               "y_tile_scale": torch.empty((R, C // 128), dtype=torch.float32).pin_memory()}
        fq.fp4q_fp8_pipeline_host(hx, ht, R, C, out["q"], out["scales"], out["y"], out["y_tile_scale"], chunk, ws,
                                  wsb, stream)
        runs.append((e4, ts, hx, ht, out))
    stream.synchronize()
    for e4, ts, _, _, out in runs:
        qr, sr = oracle.fp8_to_mx(e4, ts)
        yr, ytr = oracle.mx_to_fp8(qr, sr)
        _check_host_outputs(out, qr, sr, yr, ytr)


def test_fp8_pipeline_host_release_and_reuse(fq, oracle):
    """Releasing the call's copy streams and events between two calls on this
    thread (twice in a row, the second a no-op): the next call recreates them
    and its results are still the oracle's."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    e4, ts = W.fp8_activation(300, 1024, seed=5)
    qr, sr = oracle.fp8_to_mx(e4, ts)
    yr, ytr = oracle.mx_to_fp8(qr, sr)
    for _ in range(2):
        out = fq.fp8_pipeline_host(torch.from_numpy(e4).pin_memory(), torch.from_numpy(ts).pin_memory(),
                                   chunk_rows=64)
        _check_host_outputs(out, qr, sr, yr, ytr)
        fq.fp4q_fp8_pipeline_host_release()
        fq.fp4q_fp8_pipeline_host_release()


def test_fp8_pipeline_host_full_size(fq, oracle):
    """The benchmark's 8192 x 7168 activation through the host-buffer call
    with the default chunk: bit-identical to the oracle."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    e4, ts = W.fp8_activation()
    out = fq.fp8_pipeline_host(torch.from_numpy(e4).pin_memory(), torch.from_numpy(ts).pin_memory())
    qr, sr = oracle.fp8_to_mx(e4, ts)
    yr, ytr = oracle.mx_to_fp8(qr, sr)
    _check_host_outputs(out, qr, sr, yr, ytr)


# ---------------------------------------------------------------------------
# NVFP4
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(1, 16), (5, 48), (129, 2048), (64, 14336)])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("layout", [0, 1])
def test_nv_quantize(fq, oracle, shape, rht, rounding, layout):
    from micro_scaled_fp4_gb300 import workloads as W
    R, C = shape
    x = W.gradient_bf16(R, C, seed=R + C)
    r = fq.nv_quantize(dev_bf16(x), rht=rht, rht_seed=7, rounding=rounding, sr_seed=1234, layout=layout)
    ref = oracle.nv_quantize(x, rht=rht, rht_seed=7, rounding="sr" if rounding else "rne", sr_seed=1234)
    assert host(r["amax"])[0] == ref["amax"]
    assert host(r["s_t"])[0] == ref["s_t"]
    assert np.array_equal(host(r["q"]), ref["q"])
    sg = host(r["scales"])
    assert np.array_equal(from_mma_layout(sg, R, C // 16) if layout else sg, ref["s"])


@pytest.mark.parametrize("pad,offset", [(0, 0), (16, 0), (48, 16), (256, 256)])
@pytest.mark.parametrize("rounding", [0, 1])
def test_nv_quantize_strided_sources(fq, oracle, pad, offset, rounding):
    """Row-strided BF16 views (row stride and base a multiple of 32 bytes, an
    odd row count): the same result as the contiguous tensor."""
    import torch
    from micro_scaled_fp4_gb300 import workloads as W
    R, C = 37, 768
    x = W.gradient_bf16(R, C, seed=11)
    big = torch.zeros((R, C + pad + offset), dtype=torch.bfloat16, device="cuda")
    big[:, offset:offset + C] = dev_bf16(x)
    xv = big[:, offset:offset + C]
    r = fq.nv_quantize(xv, rht=True, rht_seed=7, rounding=rounding, sr_seed=99)
    ref = oracle.nv_quantize(x, rht=True, rht_seed=7, rounding="sr" if rounding else "rne", sr_seed=99)
    assert host(r["amax"])[0] == ref["amax"]
    assert np.array_equal(host(r["q"]), ref["q"])
    assert np.array_equal(host(r["scales"]), ref["s"])


def test_nv_quantize_zero_and_tiny(fq, oracle):
    x = np.zeros((4, 64), dtype=np.uint16)
    r = fq.nv_quantize(dev_bf16(x))
    ref = oracle.nv_quantize(x)
    assert host(r["s_t"])[0] == 0.0
    assert np.array_equal(host(r["q"]), ref["q"]) and np.array_equal(host(r["scales"]), ref["s"])
    x[1, 3] = 0x8000                      # -0.0
    x[2, :] = 0x0001                      # smallest BF16 subnormal
    x[3, 0] = 0x4000                      # 2.0: makes the subnormal blocks' scales underflow
    r = fq.nv_quantize(dev_bf16(x))
    ref = oracle.nv_quantize(x)
    assert np.array_equal(host(r["q"]), ref["q"]) and np.array_equal(host(r["scales"]), ref["s"])


@pytest.mark.parametrize("shape", [(1, 16), (5, 48), (64, 256), (129, 1040), (300, 7168)])
@pytest.mark.parametrize("rht", [0, 1, 2])
@pytest.mark.parametrize("layout", [0, 1])
def test_nv_quantize_sr_rne(fq, oracle, shape, rht, layout):
    """Both roundings from one pass equal the oracle's SR and RNE quantizations
    of the same tensor (same scales), across tiles, ragged rows and all three
    rotation modes."""
    from micro_scaled_fp4_gb300 import workloads as W
    R, C = shape
    x = W.gradient_bf16(R, C, seed=R * 7 + C)
    r = fq.nv_quantize_sr_rne(dev_bf16(x), rht=rht, rht_seed=7, sr_seed=1234, layout=layout)
    sr = oracle.nv_quantize(x, rht=rht, rht_seed=7, rounding="sr", sr_seed=1234)
    rne = oracle.nv_quantize(x, rht=rht, rht_seed=7)
    assert np.array_equal(host(r["q_sr"]), sr["q"])
    assert np.array_equal(host(r["q_rne"]), rne["q"])
    sg = host(r["scales"]) if layout == 0 else from_mma_layout(host(r["scales"]), R, C // 16)
    assert np.array_equal(sg, sr["s"]) and np.array_equal(sg, rne["s"])
    assert host(r["s_t"])[0] == sr["s_t"] and host(r["amax"])[0] == sr["amax"]


def test_nv_quantize_sr_rne_zero_and_given_amax(fq, oracle):
    """An all-zero tensor (s_t = 0: signed-zero codes in both outputs) and a
    caller-supplied amax (one pass)."""
    import torch
    x = np.zeros((8, 64), dtype=np.uint16)
    x[3, 5] = 0x8000                                  # -0
    r = fq.nv_quantize_sr_rne(dev_bf16(x), rht=0, sr_seed=1)
    ref = oracle.nv_quantize(x)
    assert np.array_equal(host(r["q_sr"]), ref["q"]) and np.array_equal(host(r["q_rne"]), ref["q"])
    from micro_scaled_fp4_gb300 import workloads as W
    xg = W.gradient_bf16(32, 512, seed=9)
    am = oracle.nv_amax(xg, 1, 7) * 2.0
    r = fq.nv_quantize_sr_rne(dev_bf16(xg), rht=1, rht_seed=7, sr_seed=5,
                              amax=torch.tensor([am], dtype=torch.float32, device="cuda"))
    sr = oracle.nv_quantize(xg, rht=1, rht_seed=7, rounding="sr", sr_seed=5, amax=am)
    rne = oracle.nv_quantize(xg, rht=1, rht_seed=7, amax=am)
    assert np.array_equal(host(r["q_sr"]), sr["q"]) and np.array_equal(host(r["q_rne"]), rne["q"])
    assert np.array_equal(host(r["scales"]), sr["s"])


def test_nv_quantize_full_size(fq, oracle):
    """The whole 8192x14336 Student-t(3)*1e-3 gradient with the RHT (seed 7):
    SR pass (seed 1234) then RNE pass, and both from the one-pass call.  Tensor
    amax, tensor scale, every code and every scale equal the oracle's
    quantization of the whole tensor."""
    from micro_scaled_fp4_gb300 import workloads as W
    x = W.gradient_bf16()
    xd = dev_bf16(x)
    both = fq.nv_quantize_sr_rne(xd, rht=True, rht_seed=7, sr_seed=1234)
    for rounding in ("sr", "rne"):
        r = fq.nv_quantize(xd, rht=True, rht_seed=7, rounding=1 if rounding == "sr" else 0, sr_seed=1234)
        ref = oracle.nv_quantize(x, rht=True, rht_seed=7, rounding=rounding, sr_seed=1234)
        assert host(r["amax"])[0] == ref["amax"] and host(r["s_t"])[0] == ref["s_t"]
        qg, sg = host(r["q"]), host(r["scales"])
        assert np.count_nonzero(qg != ref["q"]) == 0, rounding
        assert np.count_nonzero(sg != ref["s"]) == 0, rounding
        # the one-pass form of both roundings, as the benchmark times it
        assert np.count_nonzero(host(both["q_" + rounding]) != ref["q"]) == 0, rounding
        assert np.count_nonzero(host(both["scales"]) != ref["s"]) == 0, rounding
        del r, qg, sg, ref


# ---------------------------------------------------------------------------
# argument validation through the C ABI (no launch happens)
# ---------------------------------------------------------------------------
def test_argument_errors(fq):
    import torch
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((4, 32), dtype=torch.uint8, device="cuda")
    s = torch.zeros((4, 2), dtype=torch.uint8, device="cuda")
    with pytest.raises(fq.Fp4qError) as e:
        fq.fp4q_mx_quantize(x, 0, None, 4, 48, 64, 1, q, s, 0)
    assert e.value.status == 2
    with pytest.raises(fq.Fp4qError) as e:
        fq.fp4q_mx_quantize(x, 0, None, 4, 64, 64, 0, q, s, 0)
    assert e.value.status == 2
    with pytest.raises(fq.Fp4qError) as e:
        fq.fp4q_mx_quantize(None, 0, None, 4, 64, 64, 1, q, s, 0)
    assert e.value.status == 1
    with pytest.raises(fq.Fp4qError) as e:
        fq.fp4q_mx_quantize(x.data_ptr() + 2, 0, None, 4, 64, 64, 1, q, s, 0)
    assert e.value.status == 3
    # empty tensors are fine and launch nothing
    fq.fp4q_mx_quantize(None, 0, None, 0, 64, 64, 1, None, None, 0)
