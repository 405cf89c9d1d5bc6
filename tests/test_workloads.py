"""The seeded input recipe: every generator is reproducible from its seed and
has the shapes, formats and structure the workloads state (outlier columns,
1x128 tile scales, heavy-tailed gradients, Zipf-skewed top-k routing)."""
import numpy as np
import pytest

from micro_scaled_fp4_gb300 import workloads as W


def test_generators_are_seeded():
    a = W.activation_bf16(8, 64, seed=0)
    assert a.dtype == np.uint16 and a.shape == (8, 64)
    assert np.array_equal(a, W.activation_bf16(8, 64, seed=0))
    assert not np.array_equal(a, W.activation_bf16(8, 64, seed=1))
    e1, t1 = W.fp8_activation(4, 256)
    e2, t2 = W.fp8_activation(4, 256)
    assert np.array_equal(e1, e2) and np.array_equal(t1, t2)


@pytest.mark.parametrize("value,bits", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),                  # halfway, mantissa 0 is even
    (1.0 + 3 * 2.0 ** -8, 0x3F82),              # halfway, rounds to the even mantissa 2
    (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),     # above halfway
    (-1.0 - 2.0 ** -8, 0xBF80),
    (3.0e38, 0x7F62),                           # 0x7F61 and 0x7F62 bracket it; nearer is 0x7F62
])
def test_bf16_storage_rounds_to_nearest_even(value, bits):
    assert int(W.to_bf16_bits(np.array([value], dtype=np.float32))[0]) == bits


def test_fp8_activation_recipe():
    import torch
    rows, cols = 16, 7168
    e4, ts = W.fp8_activation(rows, cols)
    assert e4.dtype == np.uint8 and e4.shape == (rows, cols)
    assert ts.dtype == np.float32 and ts.shape == (rows, cols // 128)
    assert not np.any((e4 & 0x7F) == 0x7F)                  # no NaN code
    v = torch.from_numpy(e4).view(torch.float8_e4m3fn).float().numpy().reshape(rows, cols // 128, 128)
    # the tile scale maps each tile's amax onto 448, the largest E4M3 value
    assert np.all(np.abs(v).max(axis=2) == 448.0)
    x = v * ts[:, :, None]
    oc = W.outlier_columns(cols)
    assert oc.size == round(0.005 * cols) == 36
    others = np.setdiff1d(np.arange(cols), oc)
    ratio = np.abs(x.reshape(rows, cols)[:, oc]).mean() / np.abs(x.reshape(rows, cols)[:, others]).mean()
    assert 30.0 < ratio < 50.0                              # the outlier columns are scaled x40


def test_gradient_is_heavy_tailed_and_scaled():
    import torch
    g = W.gradient_bf16(64, 1024)
    x = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).float().numpy()
    med = np.median(np.abs(x))
    assert 0.7e-3 < med < 0.83e-3                           # median |t_3| = 0.765
    # Student-t(3): P(|T| > 10) ~ 2e-3, far above a normal's
    assert 5e-4 < np.mean(np.abs(x) > 10e-3) < 6e-3


def test_gemm_operands_outlier_rows():
    import torch
    a, b = W.gemm_operands(400, 8, 64)
    assert a.shape == (400, 64) and b.shape == (8, 64)
    af = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).float().numpy()
    big = np.abs(af).mean(axis=1) > 10.0
    assert big.sum() == round(0.005 * 400)


def test_moe_routing_recipe():
    T, E, k = 4096, 64, 8
    r = W.moe_routing(tokens=T, experts=E, top_k=k)
    assert r.dtype == np.int32 and r.shape == (T, k)
    assert r.min() >= 0 and r.max() < E
    assert all(len(set(row)) == k for row in r.tolist())    # k distinct experts per token
    counts = np.bincount(r.reshape(-1), minlength=E)
    assert counts[:8].sum() > 2 * counts[-8:].sum()         # Zipf(1.1): popular experts first
    assert counts[0] == counts.max()
