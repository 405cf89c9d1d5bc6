"""Seeded synthetic inputs for the FP4 hot path (shared by tests and bench.py).

Holds no quantization arithmetic: it draws random numbers and stores them in
the source formats the kernels take (BF16 by round-to-nearest-even, E4M3 by
torch's round-to-nearest cast after clipping to +-448).  Every generator uses
NumPy's PCG64 with the stated seed, so the oracle and the GPU see the same
bytes.  Shapes and distributions:

  activation_bf16   N(0, 1), BF16 [256, 4096], seed 0 (MXFP4 round trip)
  fp8_activation    N(0, 1) with 0.5 % of the columns (seeded permutation)
                    scaled x40, stored as E4M3 with one FP32 scale per 1x128
                    tile = tile amax / 448, [8192, 7168], seeds 1 / 2
  gradient_bf16     Student-t(3) * 1e-3, BF16 [8192, 14336], seed 3
  gemm_operands     A, B N(0, 1) BF16 [8192, 8192], seeds 4 / 5, 0.5 % of the
                    rows of A (seed 6) scaled x40
  moe_*             65536 tokens x 7168, top-8 of 64 experts with Zipf(1.1)
                    popularity (Gumbel top-k, seed 9), expert weights
                    N(0, 0.02^2) (seed 10), activations N(0, 1) (seed 8)
"""
from __future__ import annotations

import numpy as np


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns (uint16), round to nearest even (torch cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def activation_bf16(rows: int = 256, cols: int = 4096, seed: int = 0) -> np.ndarray:
    return to_bf16_bits(_rng(seed).standard_normal((rows, cols), dtype=np.float32))


def outlier_columns(cols: int, frac: float = 0.005, seed: int = 2) -> np.ndarray:
    n = int(round(frac * cols))
    return np.sort(_rng(seed).permutation(cols)[:n])


def fp8_activation(rows: int = 8192, cols: int = 7168, seed: int = 1, outlier_seed: int = 2,
                   outlier_scale: float = 40.0):
    """Returns (e4m3 bytes uint8 [rows, cols], tile_scale float32 [rows, cols/128])."""
    import torch
    x = _rng(seed).standard_normal((rows, cols), dtype=np.float32)
    x[:, outlier_columns(cols, seed=outlier_seed)] *= np.float32(outlier_scale)
    tiles = x.reshape(rows, cols // 128, 128)
    amax = np.abs(tiles).max(axis=2)
    s = (amax / np.float32(448.0)).astype(np.float32)
    s = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    v = np.clip(tiles / s[:, :, None], -448.0, 448.0).astype(np.float32).reshape(rows, cols)
    e4m3 = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return e4m3, s


def gradient_bf16(rows: int = 8192, cols: int = 14336, seed: int = 3, scale: float = 1e-3) -> np.ndarray:
    x = (_rng(seed).standard_t(3, (rows, cols)) * scale).astype(np.float32)
    return to_bf16_bits(x)


def gemm_operands(m: int = 8192, n: int = 8192, k: int = 8192, seed_a: int = 4, seed_b: int = 5,
                  outlier_seed: int = 6, outlier_scale: float = 40.0):
    """Returns (A bf16 bits [m, k], B bf16 bits [n, k])."""
    a = _rng(seed_a).standard_normal((m, k), dtype=np.float32)
    rows = np.sort(_rng(outlier_seed).permutation(m)[: int(round(0.005 * m))])
    a[rows] *= np.float32(outlier_scale)
    b = _rng(seed_b).standard_normal((n, k), dtype=np.float32)
    return to_bf16_bits(a), to_bf16_bits(b)


def moe_routing(tokens: int = 65536, experts: int = 64, top_k: int = 8, zipf_s: float = 1.1,
                seed: int = 9) -> np.ndarray:
    """Top-k experts per token, drawn without replacement with probability
    proportional to (e + 1)^-s (Gumbel top-k on the log-popularity).
    Returns int32 [tokens, top_k] (slot order = decreasing perturbed score)."""
    logp = -zipf_s * np.log(np.arange(1, experts + 1, dtype=np.float64))
    g = _rng(seed).gumbel(size=(tokens, experts))
    score = logp[None, :] + g
    top = np.argsort(-score, axis=1, kind="stable")[:, :top_k]
    return top.astype(np.int32)


def moe_activations(tokens: int = 65536, hidden: int = 7168, seed: int = 8) -> np.ndarray:
    return to_bf16_bits(_rng(seed).standard_normal((tokens, hidden), dtype=np.float32))


def moe_weights_torch(experts: int, rows: int, cols: int, seed: int, device, std: float = 0.02):
    """Expert weights N(0, std^2) as BF16 [experts, rows, cols], drawn on `device`
    with a seeded torch generator (the full-size tensors are several GB)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w = torch.empty((experts, rows, cols), dtype=torch.bfloat16, device=device)
    for e in range(experts):
        w[e].normal_(0.0, std, generator=g)
    return w
