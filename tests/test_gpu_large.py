"""Parity past the 32-bit element counts: 131080 x 32768 tensors (4.3 G
elements), so that rows beyond element 2^31 and 2^32 -- and Philox counters
past 2^32 -- go through every index computation of the streaming kernels.

The inputs come from an integer hash of (row, column) that the GPU evaluates
chunk by chunk (the full tensors never exist on the host) and the host
evaluates for the sampled rows, bit for bit the same.  The oracle quantizes
only the sampled rows: MX blocks are row-local, NVFP4 rows depend on the rest
of the tensor only through the tensor amax, which both sides take as given.
"""
import numpy as np
import pytest

from _helpers import host

pytestmark = pytest.mark.gpu

R, C = 131080, 32768                    # rows 65536 and 131072 start at elements 2^31 and 2^32
ROWS = np.array([0, 1, 65535, 65536, 65537, 131071, 131072, 131073, R - 1])
CHUNK = 2048


@pytest.fixture(scope="module")
def fq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import micro_scaled_fp4_gb300.fp4q as fq
    fq.load()
    return fq


def _hash(r, c, seed):
    """32-bit hash of (row, column) in int64 arithmetic (numpy or torch)."""
    return (r * 2654435761 + c * 40503 + seed * 97) & 0xFFFFFFFF


def _bf16_bits(h):
    # sign, exponent 118..130 (2^-9 .. 2^3), 7 mantissa bits
    return ((h & 1) << 15) | ((118 + (h >> 1) % 13) << 7) | ((h >> 8) & 0x7F)


def _e4m3_byte(h):
    # sign and magnitude code 0 .. 0x7d (never the NaN code 0x7f)
    return ((h & 1) << 7) | ((h >> 3) % 0x7E)


def _tile_scale(h):
    # (1 + h % 7) / 8 * 2^(k - 4): exact in FP32 on both sides
    return (1 + h % 7) / 8.0 * 2.0 ** ((h >> 3) % 9 - 4)


def _host_rows(fn, seed, cols=C):
    r = ROWS.astype(np.int64)[:, None]
    c = np.arange(cols, dtype=np.int64)[None, :]
    return fn(_hash(r, c, seed))


def _device_tensor(fn, seed, dtype, cols=C, rows=R):
    import torch
    out = torch.empty((rows, cols), dtype=dtype, device="cuda")
    c = torch.arange(cols, dtype=torch.int64, device="cuda")[None, :]
    for r0 in range(0, rows, CHUNK):
        r = torch.arange(r0, min(rows, r0 + CHUNK), dtype=torch.int64, device="cuda")[:, None]
        v = fn(_hash(r, c, seed))
        if dtype == torch.int16:                       # 16-bit patterns 0 .. 65535 as two's complement
            v = torch.where(v >= 32768, v - 65536, v)
        out[r0:r0 + r.shape[0]] = v.to(dtype)
    return out


def test_mx_quantize_bf16_beyond_2e32_elements(fq, oracle):
    import torch
    x = _device_tensor(_bf16_bits, 1, torch.int16).view(torch.bfloat16)
    q, s = fq.mx_quantize(x)
    torch.cuda.synchronize()
    del x
    qr, sr = oracle.mx_quantize(_host_rows(_bf16_bits, 1).astype(np.uint16))
    idx = torch.from_numpy(ROWS).cuda()
    assert np.array_equal(host(q[idx]), qr)
    assert np.array_equal(host(s[idx]), sr)


def test_nv_quantize_rht_sr_beyond_2e32_elements(fq, oracle):
    import torch
    x = _device_tensor(_bf16_bits, 2, torch.int16).view(torch.bfloat16)
    amax = torch.tensor([64.0], dtype=torch.float32, device="cuda")     # >= 4 x max |x| bounds the rotated values
    r = fq.nv_quantize(x, rht=True, rht_seed=7, rounding=fq.FP4Q_SR, sr_seed=11, amax=amax)
    torch.cuda.synchronize()
    del x
    xr = _host_rows(_bf16_bits, 2).astype(np.uint16)
    idx = torch.from_numpy(ROWS).cuda()
    qg, sg = host(r["q"][idx]), host(r["scales"][idx])
    for i, row in enumerate(ROWS):
        ref = oracle.nv_quantize(xr[i:i + 1], rht=True, rht_seed=7, rounding="sr", sr_seed=11, amax=64.0,
                                 row_offset=int(row))
        assert np.array_equal(qg[i], ref["q"][0]), row
        assert np.array_equal(sg[i], ref["s"][0]), row


def test_fp8_to_mx_and_back_beyond_2e32_elements(fq, oracle):
    import torch
    x = _device_tensor(_e4m3_byte, 3, torch.uint8)
    ts = _device_tensor(_tile_scale, 4, torch.float32, cols=C // 128)
    q, s = fq.mx_quantize(x.view(torch.float8_e4m3fn), tile_scale=ts)
    del x, ts
    y, yts = fq.fp4_to_fp8(q, s)
    torch.cuda.synchronize()
    e4 = _host_rows(_e4m3_byte, 3).astype(np.uint8)
    tsr = _host_rows(_tile_scale, 4, cols=C // 128).astype(np.float32)
    qr, sr = oracle.fp8_to_mx(e4, tsr)
    yr, ytr = oracle.mx_to_fp8(qr, sr)
    idx = torch.from_numpy(ROWS).cuda()
    assert np.array_equal(host(q[idx]), qr) and np.array_equal(host(s[idx]), sr)
    assert np.array_equal(host(y[idx]), yr)
    assert np.array_equal(host(yts[idx]).view(np.uint32), ytr.view(np.uint32))
