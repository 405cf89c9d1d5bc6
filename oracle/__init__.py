"""fp4q oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow CPU implementation of the micro-scaled FP4 hot path that the
CUDA library is checked against.  The elementwise and block rules live in
scalar C (``fp4q_oracle.c``, compiled with ``-ffp-contract=off`` so that every
float operation is one IEEE round-to-nearest operation); the contractions
(GEMMs, the MoE expert FFN) are float64 NumPy on the dequantized operands.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline /
reference arm may import this package.  It shares no code with
``micro_scaled_fp4_gb300`` and imports nothing from it.

Sources (web pages):
  * "Pretraining large language models with MXFP4 on Native FP4 Hardware"
    (news article), section "Qu'est-ce que le MXFP4 ?" -- MX blocks of 32, E8M0
    shared exponent, reconstruction 2^E * Q_FP4(X / 2^E); section
    "Expérience d'investigation" -- the three GEMMs of a linear layer.
  * "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs"
    (technical summaries) section 2 -- direct FP8->FP4, FP4->FP8 bit remap
    with hierarchical scale alignment, ragged MoE tensors.
  * "Pretraining Large Language Models with NVFP4" (technical summary)
    section 2 -- NVFP4 two-level scaling, random Hadamard transform,
    stochastic rounding.

Parity status of each function is stated in its docstring ("pinned by ...").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4q_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc) into oracle/_build/liboracle.so."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, u64, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
            lib.or_e2m1_value.restype = ctypes.c_double
            lib.or_e2m1_value.argtypes = [ctypes.c_int]
            lib.or_e2m1_rne.restype = ctypes.c_int
            lib.or_e2m1_rne.argtypes = [ctypes.c_float]
            lib.or_e4m3_value.restype = ctypes.c_double
            lib.or_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.or_mx_shared_exponent.restype = ctypes.c_int
            lib.or_mx_shared_exponent.argtypes = [ctypes.c_double]
            lib.or_fp8_from_e2m1_shifted.restype = ctypes.c_uint8
            lib.or_fp8_from_e2m1_shifted.argtypes = [ctypes.c_int, ctypes.c_int]
            lib.or_sr_word.restype = ctypes.c_uint32
            lib.or_sr_word.argtypes = [u64, u64]
            lib.or_nv_amax.restype = ctypes.c_float
            lib.or_nv_amax.argtypes = [vp, i64, i64, i64, ctypes.c_int, u64]
            for name, args in {
                "or_mx_quantize_f32": [vp, i64, i64, i64, vp, vp],
                "or_mx_quantize_bf16": [vp, i64, i64, i64, vp, vp],
                "or_mx_dequantize": [vp, vp, i64, i64, vp, vp],
                "or_mx_dequantize_f64": [vp, vp, i64, i64, vp],
                "or_fp8_to_mx": [vp, vp, i64, i64, i64, vp, vp],
                "or_mx_to_fp8": [vp, vp, i64, i64, vp, vp],
                "or_mx_to_fp8_col": [vp, vp, i64, i64, vp, vp],
                "or_nv_quantize_2d": [vp, i64, i64, i64, ctypes.c_int, u64, vp, vp, vp, vp, vp],
                "or_philox4x32_10": [vp, vp, vp],
                "or_rht16_signs": [u64, vp],
                "or_rht16": [vp, vp, vp],
                "or_nv_quantize": [vp, i64, i64, i64, ctypes.c_int, u64, ctypes.c_int, u64,
                                   vp, vp, vp, vp, vp, i64],
                "or_nv_dequantize": [vp, vp, ctypes.c_float, i64, i64, vp],
                "or_e2m1_rne_array": [vp, i64, vp],
                "or_e4m3_rn_satfinite_array": [vp, i64, vp],
                "or_e2m1_sr_array": [vp, vp, i64, vp],
                "or_sr_words": [u64, u64, i64, vp],
                "or_rht16_rows": [vp, i64, u64, vp],
            }.items():
                getattr(lib, name).restype = None
                getattr(lib, name).argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------
# Scalar formats
# ---------------------------------------------------------------------------
def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code (OCP MX element format)."""
    return _L().or_e2m1_value(int(code))


def e2m1_values() -> np.ndarray:
    """float64 values of the 16 E2M1 codes, indexed by code."""
    return np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def e4m3_value(b: int) -> float:
    """Value of an E4M3 (FN) byte; NaN for S.1111.111."""
    return _L().or_e4m3_value(int(b))


def e4m3_values() -> np.ndarray:
    return np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def e2m1_rne(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even, saturating, onto E2M1; one code per element."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _L().or_e2m1_rne_array(_p(v), v.size, _p(out))
    return out


def e4m3_rn_satfinite(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _L().or_e4m3_rn_satfinite_array(_p(v), v.size, _p(out))
    return out


def e2m1_sr(v: np.ndarray, r: np.ndarray) -> np.ndarray:
    """Stochastic rounding onto E2M1 with the given 32-bit words."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    r = np.ascontiguousarray(r, dtype=np.uint32)
    assert v.shape == r.shape
    out = np.empty(v.shape, dtype=np.uint8)
    _L().or_e2m1_sr_array(_p(v), _p(r), v.size, _p(out))
    return out


def mx_shared_exponent(amax: float) -> int:
    """E = floor(log2 amax) - 2, -127 for amax 0, clamped to [-127, 127].
    Pinned by tests/test_oracle_mx.py (edges and clamps)."""
    return _L().or_mx_shared_exponent(float(amax))


def fp8_from_e2m1_shifted(code: int, d: int) -> int:
    """E4M3 byte of value(code) * 2^d (the scaled FP4 -> FP8 element rule)."""
    return _L().or_fp8_from_e2m1_shifted(int(code), int(d))


# ---------------------------------------------------------------------------
# Philox
# ---------------------------------------------------------------------------
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    _L().or_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sr_words(seed: int, first: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    _L().or_sr_words(int(seed), int(first), int(n), _p(out))
    return out


# ---------------------------------------------------------------------------
# Hadamard
# ---------------------------------------------------------------------------
def rht16_signs(seed: int) -> np.ndarray:
    d = np.zeros(16, dtype=np.float32)
    _L().or_rht16_signs(int(seed), _p(d))
    return d


def rht16(x: np.ndarray, seed: int) -> np.ndarray:
    """(1/4) H16 D x on every 16-element tile of the last axis (FP32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape[-1] % 16 == 0
    y = np.empty_like(x)
    _L().or_rht16_rows(_p(x), x.size // 16, int(seed), _p(y))
    return y


# ---------------------------------------------------------------------------
# MXFP4
# ---------------------------------------------------------------------------
def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def mx_quantize(x: np.ndarray):
    """MXFP4 quantize along the last axis.

    x: uint16 array (BF16 bit patterns) or float32 array, shape [R, C], C % 32 == 0.
    Returns (q [R, C/2] uint8 packed codes, s [R, C/32] uint8 E8M0).
    Pinned by: reconstruction identity, code set, |deq| <= 6 * 2^E, qmax in
    {4, 6}, idempotence, brute force over all BF16 values (tests/test_oracle_mx.py)
    and the hand-derived golden blocks in tests/golden/mx_blocks.txt.
    """
    R, C = x.shape
    assert C % 32 == 0
    q = np.empty((R, C // 2), dtype=np.uint8)
    s = np.empty((R, C // 32), dtype=np.uint8)
    if x.dtype == np.uint16:
        x = np.ascontiguousarray(x)
        _L().or_mx_quantize_bf16(_p(x), R, C, C, _p(q), _p(s))
    else:
        x = np.ascontiguousarray(x, dtype=np.float32)
        _L().or_mx_quantize_f32(_p(x), R, C, C, _p(q), _p(s))
    return q, s


def mx_dequantize(q: np.ndarray, s: np.ndarray):
    """Returns (y_f32, y_bf16_bits) with y = 2^E * value(q), exact then rounded."""
    q = np.ascontiguousarray(q)
    s = np.ascontiguousarray(s)
    R, C2 = q.shape
    C = 2 * C2
    yf = np.empty((R, C), dtype=np.float32)
    yb = np.empty((R, C), dtype=np.uint16)
    _L().or_mx_dequantize(_p(q), _p(s), R, C, _p(yf), _p(yb))
    return yf, yb


def mx_dequantize_f64(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q)
    s = np.ascontiguousarray(s)
    R, C2 = q.shape
    y = np.empty((R, 2 * C2), dtype=np.float64)
    _L().or_mx_dequantize_f64(_p(q), _p(s), R, 2 * C2, _p(y))
    return y


def fp8_to_mx(x_e4m3: np.ndarray, tile_scale: np.ndarray):
    """Direct E4M3 (+ FP32 scale per 1x128 tile) -> MXFP4 (no BF16 step)."""
    x = np.ascontiguousarray(x_e4m3, dtype=np.uint8)
    ts = np.ascontiguousarray(tile_scale, dtype=np.float32)
    R, C = x.shape
    assert C % 128 == 0 and ts.shape == (R, C // 128)
    q = np.empty((R, C // 2), dtype=np.uint8)
    s = np.empty((R, C // 32), dtype=np.uint8)
    _L().or_fp8_to_mx(_p(x), _p(ts), R, C, C, _p(q), _p(s))
    return q, s


def mx_to_fp8(q: np.ndarray, s: np.ndarray):
    """Scaled MXFP4 -> (E4M3 [R, C], FP32 tile scale [R, C/128])."""
    q = np.ascontiguousarray(q)
    s = np.ascontiguousarray(s)
    R, C2 = q.shape
    C = 2 * C2
    assert C % 128 == 0
    y = np.empty((R, C), dtype=np.uint8)
    ts = np.empty((R, C // 128), dtype=np.float32)
    _L().or_mx_to_fp8(_p(q), _p(s), R, C, _p(y), _p(ts))
    return y, ts


def mx_to_fp8_col(q: np.ndarray, s: np.ndarray):
    """FP4RowToFP8Col: row-wise MXFP4 [R, C] -> (E4M3 of the transpose [C, R],
    FP32 scale per 1x128 tile along R [C, R/128])."""
    q = np.ascontiguousarray(q)
    s = np.ascontiguousarray(s)
    R, C2 = q.shape
    C = 2 * C2
    assert R % 128 == 0 and C % 32 == 0
    y = np.empty((C, R), dtype=np.uint8)
    ts = np.empty((C, R // 128), dtype=np.float32)
    _L().or_mx_to_fp8_col(_p(q), _p(s), R, C, _p(y), _p(ts))
    return y, ts


def mx_to_fp8_col_grouped(q: np.ndarray, s: np.ndarray, offsets):
    """FP4RowToFP8Col on ragged expert groups ("Practical FP4 Training for
    Large-Scale MoE Models on Hopper GPUs", Spanish summary section 2 for the
    kernel, French summary 2.C for ragged per-expert tensors with precomputed
    offsets).  The 1x128 tiles of the transposed output run along each group's
    rows and restart at its first row; the pages leave the group's last,
    partial tile open, and the reading taken here is the plainest one: its
    scale is 2^Emax over its real rows only, and the output pads every group
    to whole tiles with zeros.  Written as the dense rule (mx_to_fp8_col) on
    each group's rows padded to a multiple of 128 with zero codes and zero
    E8M0 bytes: a zero byte (2^-127) never raises a tile's maximum, and zero
    codes give zero bytes.  Returns (E4M3 [C, 128 T], FP32 tile scales
    [C, T]), T = sum over groups of ceil(n_g / 128), group g's rows at columns
    128 T_g .. 128 T_g + n_g - 1 (T_g its tiles' start).  Pinned by
    tests/test_oracle_widen.py (tile-aligned groups equal the dense rule on
    their rows; a hand-derived partial tile; an element-wise brute force)."""
    q = np.ascontiguousarray(q)
    s = np.ascontiguousarray(s)
    offsets = [int(v) for v in offsets]
    C = 2 * q.shape[1]
    tiles = [(offsets[g + 1] - offsets[g] + 127) // 128 for g in range(len(offsets) - 1)]
    T = sum(tiles)
    y = np.zeros((C, 128 * T), dtype=np.uint8)
    ts = np.zeros((C, T), dtype=np.float32)
    t0 = 0
    for g, tg in enumerate(tiles):
        lo, hi = offsets[g], offsets[g + 1]
        if tg == 0:
            continue
        qg = np.zeros((128 * tg, C // 2), dtype=np.uint8)
        sg = np.zeros((128 * tg, C // 32), dtype=np.uint8)
        qg[: hi - lo] = q[lo:hi]
        sg[: hi - lo] = s[lo:hi]
        yg, tsg = mx_to_fp8_col(qg, sg)
        y[:, 128 * t0: 128 * (t0 + tg)] = yg
        ts[:, t0: t0 + tg] = tsg
        t0 += tg
    return y, ts


def mx_quantize_col(x: np.ndarray):
    """Column-wise MXFP4 (blocks of 32 along axis 0): by definition the
    row-wise quantization of the transpose, returned in the transposed layout
    (q [C, R/2], s [C, R/32]).  Pinned by a hand-derived case
    (tests/test_oracle_mx.py)."""
    return mx_quantize(np.ascontiguousarray(np.asarray(x).T))


# ---------------------------------------------------------------------------
# NVFP4
# ---------------------------------------------------------------------------
def _rht_mode(rht) -> int:
    """False/0: no rotation; True/1: random-sign RHT from the seed; 2: the
    deterministic H16 (no sign flips)."""
    m = int(rht)
    assert m in (0, 1, 2)
    return m


def nv_amax(x_bf16: np.ndarray, rht, rht_seed: int) -> float:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, C = x.shape
    return float(_L().or_nv_amax(_p(x), R, C, C, _rht_mode(rht), int(rht_seed)))


def nv_quantize(x_bf16: np.ndarray, rht=False, rht_seed: int = 0, rounding: str = "rne",
                sr_seed: int = 0, amax: float | None = None, row_offset: int = 0):
    """NVFP4 quantize of a BF16 tensor along the last axis.

    x_bf16 may be a slice of rows of a larger tensor: row_offset is its first
    row's index there (the stochastic-rounding words follow the full tensor's
    linear element index); pass that tensor's amax too.
    Returns dict(q [R, C/2], s [R, C/16] E4M3 bytes, s_t float32, amax float32).
    """
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, C = x.shape
    assert C % 16 == 0
    q = np.empty((R, C // 2), dtype=np.uint8)
    s = np.empty((R, C // 16), dtype=np.uint8)
    amax_out = np.zeros(1, dtype=np.float32)
    st_out = np.zeros(1, dtype=np.float32)
    amax_in = None if amax is None else np.array([amax], dtype=np.float32)
    _L().or_nv_quantize(_p(x), R, C, C, _rht_mode(rht), int(rht_seed), 1 if rounding == "sr" else 0,
                        int(sr_seed), None if amax_in is None else _p(amax_in), _p(amax_out),
                        _p(st_out), _p(q), _p(s), int(row_offset))
    return {"q": q, "s": s, "s_t": np.float32(st_out[0]), "amax": np.float32(amax_out[0])}


def nv_quantize_col(x_bf16: np.ndarray, **kw):
    """Column-wise NVFP4 (16-blocks and RHT tiles along axis 0): by definition
    the row-wise quantization of the transpose, in the transposed layout; the
    stochastic-rounding words follow the transpose's linear element index.
    Pinned by its structure on constant columns (tests/test_oracle_nv.py) and
    the Wgrad contraction tests (tests/test_oracle_widen.py)."""
    return nv_quantize(np.ascontiguousarray(np.asarray(x_bf16).T), **kw)


def nv_quantize_2d(x_bf16: np.ndarray, rounding: str = "rne", sr_seed: int = 0, amax: float | None = None):
    """NVFP4 with one E4M3 scale per 16x16 tile (weights), scales stored per
    row ([R, C/16], 16 equal rows per tile).  Returns the dict of nv_quantize."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, C = x.shape
    assert R % 16 == 0 and C % 16 == 0
    q = np.empty((R, C // 2), dtype=np.uint8)
    s = np.empty((R, C // 16), dtype=np.uint8)
    amax_out = np.zeros(1, dtype=np.float32)
    st_out = np.zeros(1, dtype=np.float32)
    amax_in = None if amax is None else np.array([amax], dtype=np.float32)
    _L().or_nv_quantize_2d(_p(x), R, C, C, 1 if rounding == "sr" else 0, int(sr_seed),
                           None if amax_in is None else _p(amax_in), _p(amax_out), _p(st_out), _p(q), _p(s))
    return {"q": q, "s": s, "s_t": np.float32(st_out[0]), "amax": np.float32(amax_out[0])}


def nv_dequantize_f64(q: np.ndarray, s: np.ndarray, s_t: float) -> np.ndarray:
    q = np.ascontiguousarray(q)
    s = np.ascontiguousarray(s)
    R, C2 = q.shape
    y = np.empty((R, 2 * C2), dtype=np.float64)
    _L().or_nv_dequantize(_p(q), _p(s), float(s_t), R, 2 * C2, _p(y))
    return y


# ---------------------------------------------------------------------------
# GEMM (float64 on the dequantized operands)
# ---------------------------------------------------------------------------
def gemm_ref(a_deq: np.ndarray, b_deq: np.ndarray) -> np.ndarray:
    """Y = A . B^T in float64 (the Fprop GEMM Y = X W^T of a linear layer,
    "Pretraining ... MXFP4 on Native FP4 Hardware", section "Expérience
    d'investigation").  Pinned by an explicit triple loop on small shapes."""
    return np.asarray(a_deq, dtype=np.float64) @ np.asarray(b_deq, dtype=np.float64).T


def mx_gemm_ref(qa, sa, qb, sb) -> np.ndarray:
    return gemm_ref(mx_dequantize_f64(qa, sa), mx_dequantize_f64(qb, sb))


def nv_gemm_ref(qa, sa, sta, qb, sb, stb) -> np.ndarray:
    """float64 Y = A . B^T of dequantized NVFP4 operands.  Pinned by an exact
    rational triple loop (tests/test_oracle_gemm.py)."""
    return gemm_ref(nv_dequantize_f64(qa, sa, sta), nv_dequantize_f64(qb, sb, stb))


def fp8_gemm_ref(ya: np.ndarray, tsa: np.ndarray, yb: np.ndarray, tsb: np.ndarray) -> np.ndarray:
    """float64 D = A . B^T of FP8 operands with FP32 scales per 1x128 tile:
    A = value(E4M3 ya) * tsa (tile of the element), exact in float64."""
    lut = e4m3_values()
    a = lut[np.asarray(ya)] * np.repeat(np.asarray(tsa, dtype=np.float64), 128, axis=1)
    b = lut[np.asarray(yb)] * np.repeat(np.asarray(tsb, dtype=np.float64), 128, axis=1)
    return a @ b.T


def rel_frobenius(y: np.ndarray, ref: np.ndarray) -> float:
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(y - ref) / (den if den > 0 else 1.0))


# ---------------------------------------------------------------------------
# MoE expert FFN (routing, dispatch, grouped up/down projection)
# ---------------------------------------------------------------------------
def moe_dispatch(topk_experts: np.ndarray, n_experts: int):
    """Group (token, slot) pairs by expert, ascending token id inside an
    expert; returns (token_of_row [T*k] int64, offsets [E+1] int64).
    Ragged groups with precomputed offsets and no padding ("Practical FP4
    Training ... on Hopper GPUs", section 2.C: ragged tensors)."""
    T, k = topk_experts.shape
    tokens = np.repeat(np.arange(T, dtype=np.int64), k)
    experts = topk_experts.reshape(-1).astype(np.int64)
    order = np.lexsort((tokens, experts))        # primary: expert, secondary: token
    counts = np.bincount(experts, minlength=n_experts)
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    return tokens[order], offsets


def mx_rebase_scales(e8m0: np.ndarray):
    """MXFP4 block scales -> UE4M3 scales per 16 elements and a per-row
    factor, so MXFP4 rows can enter a block-scaled product whose other operand
    is NVFP4 (one scale type per product).  The pages quantize activations to
    MXFP4 before the expert dispatch ("Practical FP4 Training for Large-Scale
    MoE Models on Hopper GPUs", section 2.A) while NVFP4 ("Pretraining Large
    Language Models with NVFP4", section 2.B) scales blocks of 16 by E4M3; they
    do not say how the two meet, so this is the build's own reading, written
    out plainly.  Per row with block exponents E_j = byte_j - 127:
      B = max_j E_j - 8;  block j's scale 2^E_j = 2^(E_j - B) * 2^B;
      2^(E_j - B) is a UE4M3 value for E_j - B in [-9, 8] (normal from -6,
      subnormal 2^-7, 2^-8, 2^-9), and both 16-element halves of block j take
      that byte; E_j - B < -9 is not representable: the byte is 0 and the
      block is counted as a violation.
    Returns (ue4m3 [R, 2 S32] uint8, row factor 2^B [R] float32, violations).
    Pinned by hand-derived rows and by the reconstruction
    e4m3_value(byte) * 2^B == 2^E_j on every representable block
    (tests/test_oracle_gemm.py)."""
    e = np.asarray(e8m0, dtype=np.int64) - 127
    R = e.shape[0]
    B = (e.max(axis=1) if e.shape[1] else np.zeros(R, np.int64)) - 8
    k = e - B[:, None]                                   # in [-254 - 8, 8]
    ue = np.zeros(e.shape, dtype=np.uint8)
    normal = k >= -6
    ue[normal] = ((k[normal] + 7) << 3).astype(np.uint8)
    sub = (k >= -9) & ~normal
    ue[sub] = (1 << (k[sub] + 9)).astype(np.uint8)
    violations = int(np.count_nonzero(k < -9))
    factor = np.array([np.ldexp(np.float32(1.0), int(b)) for b in B], dtype=np.float32)
    return np.repeat(ue, 2, axis=1), factor, violations


def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g / (1 + exp(-g)) in float64."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def moe_up_gate(x_rows_deq: np.ndarray, w1_deq: np.ndarray, inter: int) -> np.ndarray:
    """U = X_e W1_e^T; h = SiLU(U[:, :inter]) * U[:, inter:] (float64).
    Pinned by a closed form on one-hot token rows (tests/test_oracle_gemm.py)."""
    u = gemm_ref(x_rows_deq, w1_deq)
    return silu(u[:, :inter]) * u[:, inter:]
