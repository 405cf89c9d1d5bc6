"""ctypes binding of the fp4q C ABI (include/fp4q.h).

Argument marshalling only: every function here has the name of the C entry
point it calls and forwards plain pointers (``tensor.data_ptr()`` or ints),
sizes and the CUDA stream (``torch.cuda.current_stream().cuda_stream`` unless
given).  All compute happens in the CUDA library; if libfp4q.so is missing the
first call raises.  The helpers at the bottom (``mx_quantize`` ...) allocate
their outputs with torch and call the same entry points.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

# enums of include/fp4q.h
FP4Q_OK = 0
STATUS_NAMES = {0: "FP4Q_OK", 1: "FP4Q_ERR_INVALID_ARGUMENT", 2: "FP4Q_ERR_UNSUPPORTED_SHAPE",
                3: "FP4Q_ERR_MISALIGNED", 4: "FP4Q_ERR_UNSUPPORTED_DEVICE", 5: "FP4Q_ERR_CUDA",
                6: "FP4Q_ERR_TIMEOUT"}
FP4Q_BF16, FP4Q_FP32, FP4Q_E4M3 = 0, 1, 2
FP4Q_SCALES_ROWMAJOR, FP4Q_SCALES_MMA = 0, 1
FP4Q_RNE, FP4Q_SR = 0, 1
FP4Q_MXFP4, FP4Q_NVFP4, FP4Q_MXFP8 = 0, 1, 2

FP4Q_EPI_STORE_BF16, FP4Q_EPI_SILU_GATE_MXFP4 = 0, 1

EXPORTED = [
    "fp4q_status_string", "fp4q_last_error", "fp4q_scales_bytes", "fp4q_mx_quantize",
    "fp4q_mx_dequantize", "fp4q_fp4_to_fp8", "fp4q_nv_quantize_workspace_bytes", "fp4q_nv_quantize",
    "fp4q_block_scaled_gemm", "fp4q_device_status", "fp4q_moe_dispatch_workspace_bytes",
    "fp4q_moe_dispatch", "fp4q_rebased_scales_bytes", "fp4q_mx_rebase_scales", "fp4q_grouped_gemm",
    "fp4q_moe_dispatch_static", "fp4q_check_wait_timeout", "fp4q_nv_quantize_2d", "fp4q_fp4_row_to_fp8_col",
    "fp4q_fp8_tile_scales_to_e8m0", "fp4q_fp8_pipeline_host_workspace_bytes", "fp4q_fp8_pipeline_host",
    "fp4q_stream_status", "fp4q_fp8_pipeline_host_release", "fp4q_nv_quantize_sr_rne",
    "fp4q_fp4_row_to_fp8_col_grouped_ld", "fp4q_fp4_row_to_fp8_col_grouped",
]
MOE_DISPATCH_STATIC_SCRATCH_BYTES = 4 * 1024 * 1024


class Fp4qError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(status, status)}: {detail}")
        self.status = status


class fp4q_operand(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("format", ctypes.c_int),
                ("tensor_scale", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libfp4q.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB_PATH):
                raise RuntimeError(f"fp4q CUDA library not built ({_build.LIB_PATH}); run __graft_entry__.build()")
            L = ctypes.CDLL(_build.LIB_PATH)
            i64, u64, vp, ci = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int
            L.fp4q_status_string.restype = ctypes.c_char_p
            L.fp4q_status_string.argtypes = [ci]
            L.fp4q_last_error.restype = ctypes.c_char_p
            L.fp4q_last_error.argtypes = []
            L.fp4q_scales_bytes.restype = ctypes.c_size_t
            L.fp4q_scales_bytes.argtypes = [i64, i64, ci]
            L.fp4q_nv_quantize_workspace_bytes.restype = ctypes.c_size_t
            L.fp4q_nv_quantize_workspace_bytes.argtypes = [i64, i64]
            for name, args in {"fp4q_moe_dispatch_workspace_bytes": [i64, ci, ci],
                               "fp4q_rebased_scales_bytes": [i64, i64, i64],
                               "fp4q_fp8_pipeline_host_workspace_bytes": [i64, i64]}.items():
                fn = getattr(L, name, None)
                if fn is not None:
                    fn.restype = ctypes.c_size_t
                    fn.argtypes = args
            fn = getattr(L, "fp4q_fp4_row_to_fp8_col_grouped_ld", None)
            if fn is not None:
                fn.restype = i64
                fn.argtypes = [i64, i64]
            sigs = {
                "fp4q_mx_quantize": [vp, ci, vp, i64, i64, i64, ci, vp, vp, ci, vp],
                "fp4q_mx_dequantize": [vp, vp, i64, i64, ci, vp, ci, vp],
                "fp4q_fp4_to_fp8": [vp, vp, i64, i64, ci, vp, vp, vp],
                "fp4q_nv_quantize": [vp, i64, i64, i64, ci, ci, u64, ci, u64, vp, vp, vp, vp, vp, ci, vp,
                                     ctypes.c_size_t, vp],
                "fp4q_block_scaled_gemm": [ctypes.POINTER(fp4q_operand), ctypes.POINTER(fp4q_operand), i64, i64,
                                           i64, vp, ci, i64, vp],
                "fp4q_device_status": [ctypes.POINTER(ctypes.c_uint32), ci],
                "fp4q_stream_status": [ctypes.POINTER(ctypes.c_uint32), ci, vp],
                "fp4q_moe_dispatch": [vp, i64, ci, ci, vp, vp, i64, vp, vp, vp, vp, vp, ctypes.c_size_t, vp],
                "fp4q_mx_rebase_scales": [vp, i64, i64, vp, i64, vp, vp, vp, vp],
                "fp4q_moe_dispatch_static": [vp, i64, ci, ci, vp, vp, i64, vp, vp, vp, vp, vp],
                "fp4q_check_wait_timeout": [u64, vp],
                "fp4q_nv_quantize_2d": [vp, i64, i64, i64, ci, u64, vp, vp, vp, vp, vp, ci, vp, ctypes.c_size_t, vp],
                "fp4q_nv_quantize_sr_rne": [vp, i64, i64, i64, ci, u64, u64, vp, vp, vp, vp, vp, vp, ci, vp,
                                            ctypes.c_size_t, vp],
                "fp4q_fp4_row_to_fp8_col": [vp, vp, i64, i64, vp, vp, vp],
                "fp4q_fp4_row_to_fp8_col_grouped": [vp, vp, i64, i64, vp, i64, vp, vp, vp],
                "fp4q_fp8_tile_scales_to_e8m0": [vp, i64, i64, vp, ci, vp],
                "fp4q_fp8_pipeline_host": [vp, vp, i64, i64, vp, vp, vp, vp, i64, vp, ctypes.c_size_t, vp],
                "fp4q_fp8_pipeline_host_release": [],
                "fp4q_grouped_gemm": [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, ci, vp, vp, vp, vp],
            }
            for name, args in sigs.items():
                fn = getattr(L, name, None)     # resolved here; a missing symbol fails at its call
                if fn is not None:
                    fn.restype = ci
                    fn.argtypes = args
            _lib = L
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int) -> int:
    if status != FP4Q_OK:
        raise Fp4qError(fn, status, load().fp4q_last_error().decode())
    return status


# ---------------------------------------------------------------------------
# 1:1 wrappers of the C entry points
# ---------------------------------------------------------------------------
def fp4q_status_string(status: int) -> str:
    return load().fp4q_status_string(status).decode()


def fp4q_scales_bytes(rows: int, scale_cols: int, layout: int) -> int:
    return load().fp4q_scales_bytes(rows, scale_cols, layout)


def fp4q_nv_quantize_workspace_bytes(rows: int, cols: int) -> int:
    return load().fp4q_nv_quantize_workspace_bytes(rows, cols)


def fp4q_mx_quantize(x, x_type, tile_scale, rows, cols, ld_x, block_axis, q, scales, layout, stream=None):
    return _check("fp4q_mx_quantize", load().fp4q_mx_quantize(
        _ptr(x), x_type, _ptr(tile_scale), rows, cols, ld_x, block_axis, _ptr(q), _ptr(scales), layout,
        _stream(stream)))


def fp4q_mx_dequantize(q, scales, rows, cols, block_axis, y, y_type, stream=None):
    return _check("fp4q_mx_dequantize", load().fp4q_mx_dequantize(
        _ptr(q), _ptr(scales), rows, cols, block_axis, _ptr(y), y_type, _stream(stream)))


def fp4q_fp4_to_fp8(q, scales, rows, cols, block_axis, y, tile_scale, stream=None):
    return _check("fp4q_fp4_to_fp8", load().fp4q_fp4_to_fp8(
        _ptr(q), _ptr(scales), rows, cols, block_axis, _ptr(y), _ptr(tile_scale), _stream(stream)))


def fp4q_fp8_pipeline_host_workspace_bytes(cols, chunk_rows=0):
    return int(load().fp4q_fp8_pipeline_host_workspace_bytes(cols, chunk_rows))


def fp4q_fp8_pipeline_host(x, tile_scale, rows, cols, q, scales, y, y_tile_scale, chunk_rows, workspace,
                           workspace_bytes, stream=None):
    """Host-buffer FP8 -> MXFP4 -> FP8 path (x, tile_scale, q, scales, y,
    y_tile_scale are host tensors or addresses; workspace is device memory)."""
    return _check("fp4q_fp8_pipeline_host", load().fp4q_fp8_pipeline_host(
        _ptr(x), _ptr(tile_scale), rows, cols, _ptr(q), _ptr(scales), _ptr(y), _ptr(y_tile_scale), chunk_rows,
        _ptr(workspace), workspace_bytes, _stream(stream)))


def fp4q_fp8_pipeline_host_release():
    return _check("fp4q_fp8_pipeline_host_release", load().fp4q_fp8_pipeline_host_release())


def fp8_pipeline_host(x, tile_scale, chunk_rows=0, pinned=True, stream=None):
    """E4M3 host tensor [R, C] (uint8 or float8_e4m3fn) + FP32 tile scales
    [R, C/128] -> host dict(q, scales, y, y_tile_scale); synchronizes the stream."""
    torch = _torch()
    for name, t in (("x", x), ("tile_scale", tile_scale)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    R, C = x.shape
    mk = (lambda shape, dt: torch.empty(shape, dtype=dt).pin_memory()) if pinned else \
        (lambda shape, dt: torch.empty(shape, dtype=dt))
    out = {"q": mk((R, C // 2), torch.uint8), "scales": mk((R, C // 32), torch.uint8),
           "y": mk((R, C), torch.uint8), "y_tile_scale": mk((R, C // 128), torch.float32)}
    wsb = fp4q_fp8_pipeline_host_workspace_bytes(C, min(chunk_rows or 2048, max(R, 1)))
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    fp4q_fp8_pipeline_host(x, tile_scale, R, C, out["q"], out["scales"], out["y"], out["y_tile_scale"], chunk_rows,
                           ws, wsb, stream)
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    return out


def fp4q_nv_quantize(x, rows, cols, ld_x, block_axis, rht, rht_seed, rounding, sr_seed, amax_in, amax_out,
                     tensor_scale_out, q, scales, layout, workspace, workspace_bytes, stream=None):
    return _check("fp4q_nv_quantize", load().fp4q_nv_quantize(
        _ptr(x), rows, cols, ld_x, block_axis, int(rht), rht_seed, rounding, sr_seed, _ptr(amax_in),
        _ptr(amax_out), _ptr(tensor_scale_out), _ptr(q), _ptr(scales), layout, _ptr(workspace),
        workspace_bytes, _stream(stream)))


def fp4q_nv_quantize_sr_rne(x, rows, cols, ld_x, rht, rht_seed, sr_seed, amax_in, amax_out, tensor_scale_out, q_sr,
                            q_rne, scales, layout, workspace, workspace_bytes, stream=None):
    return _check("fp4q_nv_quantize_sr_rne", load().fp4q_nv_quantize_sr_rne(
        _ptr(x), rows, cols, ld_x, int(rht), rht_seed, sr_seed, _ptr(amax_in), _ptr(amax_out),
        _ptr(tensor_scale_out), _ptr(q_sr), _ptr(q_rne), _ptr(scales), layout, _ptr(workspace), workspace_bytes,
        _stream(stream)))


def fp4q_nv_quantize_2d(x, rows, cols, ld_x, rounding, sr_seed, amax_in, amax_out, tensor_scale_out, q, scales,
                        layout, workspace, workspace_bytes, stream=None):
    return _check("fp4q_nv_quantize_2d", load().fp4q_nv_quantize_2d(
        _ptr(x), rows, cols, ld_x, rounding, sr_seed, _ptr(amax_in), _ptr(amax_out), _ptr(tensor_scale_out),
        _ptr(q), _ptr(scales), layout, _ptr(workspace), workspace_bytes, _stream(stream)))


def fp4q_fp4_row_to_fp8_col(q, scales, rows, cols, y, tile_scale, stream=None):
    return _check("fp4q_fp4_row_to_fp8_col", load().fp4q_fp4_row_to_fp8_col(
        _ptr(q), _ptr(scales), rows, cols, _ptr(y), _ptr(tile_scale), _stream(stream)))


def fp4q_fp4_row_to_fp8_col_grouped_ld(rows, groups):
    return load().fp4q_fp4_row_to_fp8_col_grouped_ld(rows, groups)


def fp4q_fp4_row_to_fp8_col_grouped(q, scales, rows, cols, offsets, groups, y, tile_scale, stream=None):
    return _check("fp4q_fp4_row_to_fp8_col_grouped", load().fp4q_fp4_row_to_fp8_col_grouped(
        _ptr(q), _ptr(scales), rows, cols, _ptr(offsets), groups, _ptr(y), _ptr(tile_scale), _stream(stream)))


def fp4q_fp8_tile_scales_to_e8m0(tile_scale, rows, cols, scales, layout, stream=None):
    return _check("fp4q_fp8_tile_scales_to_e8m0", load().fp4q_fp8_tile_scales_to_e8m0(
        _ptr(tile_scale), rows, cols, _ptr(scales), layout, _stream(stream)))


def make_operand(q, scales, fmt, tensor_scale=None) -> fp4q_operand:
    return fp4q_operand(_ptr(q), _ptr(scales), fmt, _ptr(tensor_scale))


def fp4q_block_scaled_gemm(A: fp4q_operand, B: fp4q_operand, M, N, K, D, d_type, ldd, stream=None):
    return _check("fp4q_block_scaled_gemm", load().fp4q_block_scaled_gemm(
        ctypes.byref(A), ctypes.byref(B), M, N, K, _ptr(D), d_type, ldd, _stream(stream)))


def fp4q_moe_dispatch_workspace_bytes(tokens: int, top_k: int, n_experts: int) -> int:
    return load().fp4q_moe_dispatch_workspace_bytes(tokens, top_k, n_experts)


def fp4q_rebased_scales_bytes(rows: int, cols: int, groups: int) -> int:
    return load().fp4q_rebased_scales_bytes(rows, cols, groups)


def fp4q_moe_dispatch(topk, tokens, top_k, n_experts, q, scales, cols, offsets, row_token, q_out, scales_out,
                      workspace, workspace_bytes, stream=None):
    return _check("fp4q_moe_dispatch", load().fp4q_moe_dispatch(
        _ptr(topk), tokens, top_k, n_experts, _ptr(q), _ptr(scales), cols, _ptr(offsets), _ptr(row_token),
        _ptr(q_out), _ptr(scales_out), _ptr(workspace), workspace_bytes, _stream(stream)))


def fp4q_moe_dispatch_static(topk, tokens, top_k, n_experts, q, scales, cols, offsets, row_token, q_out,
                             scales_out, stream=None):
    """fp4q_moe_dispatch with the library's static scratch instead of a workspace
    (for callers that must not allocate device memory on this path)."""
    return _check("fp4q_moe_dispatch_static", load().fp4q_moe_dispatch_static(
        _ptr(topk), tokens, top_k, n_experts, _ptr(q), _ptr(scales), cols, _ptr(offsets), _ptr(row_token),
        _ptr(q_out), _ptr(scales_out), _stream(stream)))


def fp4q_mx_rebase_scales(scales, rows, cols, offsets, groups, ue4m3_mma, row_scale, violations, stream=None):
    return _check("fp4q_mx_rebase_scales", load().fp4q_mx_rebase_scales(
        _ptr(scales), rows, cols, _ptr(offsets), groups, _ptr(ue4m3_mma), _ptr(row_scale), _ptr(violations),
        _stream(stream)))


def fp4q_grouped_gemm(a_q, a_scales, a_row_scale, b_q, b_scales, b_tensor_scale, offsets, rows, groups, N, K,
                      epilogue, D, d_scales, h_debug, stream=None):
    return _check("fp4q_grouped_gemm", load().fp4q_grouped_gemm(
        _ptr(a_q), _ptr(a_scales), _ptr(a_row_scale), _ptr(b_q), _ptr(b_scales), _ptr(b_tensor_scale),
        _ptr(offsets), rows, groups, N, K, epilogue, _ptr(D), _ptr(d_scales), _ptr(h_debug), _stream(stream)))


def fp4q_check_wait_timeout(limit_ns: int, stream=None):
    return _check("fp4q_check_wait_timeout", load().fp4q_check_wait_timeout(limit_ns, _stream(stream)))


def fp4q_stream_status(reset: bool = False, stream=None) -> int:
    """Waits for the stream, then returns the device status word (0 = no
    device-side wait timed out)."""
    v = ctypes.c_uint32(0)
    st = load().fp4q_stream_status(ctypes.byref(v), int(bool(reset)), _stream(stream))
    if st not in (FP4Q_OK, 6):
        _check("fp4q_stream_status", st)
    return int(v.value)


def fp4q_device_status(reset: bool = False) -> int:
    """Returns the device status word (0 = no device-side wait timed out)."""
    v = ctypes.c_uint32(0)
    st = load().fp4q_device_status(ctypes.byref(v), int(bool(reset)))
    if st not in (FP4Q_OK, 6):
        _check("fp4q_device_status", st)
    return int(v.value)


# ---------------------------------------------------------------------------
# Allocating helpers (torch for device memory; compute in the entry points)
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _on_device(name, t, rows_strided=False):
    """Checks a helper's tensor argument before its address reaches a kernel:
    a CUDA tensor on the current device, contiguous (``rows_strided``: unit
    stride along the last axis, any row stride).  None passes (optional)."""
    if t is None:
        return
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise ValueError(f"{name} is on {t.device}; the library works on the current device cuda:{cur}")
    ok = t.stride(-1) == 1 if (rows_strided and t.dim() == 2) else t.is_contiguous()
    if not ok:
        raise ValueError(f"{name} must be contiguous" + (" along its rows" if rows_strided else ""))


def mx_quantize(x, tile_scale=None, layout=FP4Q_SCALES_ROWMAJOR, block_axis=1, stream=None):
    """BF16 / FP32 / float8_e4m3fn [R, C] -> (q uint8, scales uint8).

    block_axis 1: q [R, C/2], scales of R x C/32.  block_axis 0 (BF16): the
    quantization of X^T, q [C, R/2], scales of C x R/32."""
    torch = _torch()
    _on_device("x", x, rows_strided=True)
    _on_device("tile_scale", tile_scale)
    R, C = x.shape
    xt = {torch.bfloat16: FP4Q_BF16, torch.float32: FP4Q_FP32, torch.float8_e4m3fn: FP4Q_E4M3,
          torch.uint8: FP4Q_E4M3}[x.dtype]
    OR, OC = (R, C) if block_axis == 1 else (C, R)
    q = torch.empty((OR, OC // 2), dtype=torch.uint8, device=x.device)
    s = torch.empty(fp4q_scales_bytes(OR, OC // 32, layout), dtype=torch.uint8, device=x.device)
    fp4q_mx_quantize(x, xt, tile_scale, R, C, x.stride(0), block_axis, q, s, layout, stream)
    return q, (s.view(OR, OC // 32) if layout == FP4Q_SCALES_ROWMAJOR else s)


def mx_dequantize(q, s, dtype=None, stream=None):
    torch = _torch()
    _on_device("q", q)
    _on_device("s", s)
    dtype = dtype or torch.bfloat16
    R, C = q.shape[0], q.shape[1] * 2
    y = torch.empty((R, C), dtype=dtype, device=q.device)
    fp4q_mx_dequantize(q, s, R, C, 1, y, FP4Q_BF16 if dtype == torch.bfloat16 else FP4Q_FP32, stream)
    return y


def fp8_mma_scales(tile_scale, stream=None):
    """FP32 power-of-two 1x128 tile scales [R, C/128] -> E8M0 per 32 in the MMA layout."""
    torch = _torch()
    _on_device("tile_scale", tile_scale)
    R, C = tile_scale.shape[0], tile_scale.shape[1] * 128
    s = torch.empty(fp4q_scales_bytes(R, C // 32, FP4Q_SCALES_MMA), dtype=torch.uint8, device=tile_scale.device)
    fp4q_fp8_tile_scales_to_e8m0(tile_scale, R, C, s, FP4Q_SCALES_MMA, stream)
    return s


def fp4_row_to_fp8_col(q, s, stream=None):
    """Row-wise MXFP4 [R, C] -> (E4M3 of the transpose [C, R], FP32 tile scales [C, R/128])."""
    torch = _torch()
    _on_device("q", q)
    _on_device("s", s)
    R, C = q.shape[0], q.shape[1] * 2
    y = torch.empty((C, R), dtype=torch.uint8, device=q.device)
    ts = torch.empty((C, R // 128), dtype=torch.float32, device=q.device)
    fp4q_fp4_row_to_fp8_col(q, s, R, C, y, ts, stream)
    return y, ts


def fp4_row_to_fp8_col_grouped(q, s, offsets, groups, stream=None):
    """Row-wise MXFP4 [R, C] in ragged groups (offsets [groups + 1], device) ->
    (E4M3 [C, ld], FP32 tile scales [C, ld/128]), each group padded to whole
    128-row tiles (ld = 128 * (ceil(R / 128) + groups))."""
    torch = _torch()
    for name, t in (("q", q), ("s", s), ("offsets", offsets)):
        _on_device(name, t)
    R, C = q.shape[0], q.shape[1] * 2
    ld = fp4q_fp4_row_to_fp8_col_grouped_ld(R, groups)
    y = torch.empty((C, ld), dtype=torch.uint8, device=q.device)
    ts = torch.empty((C, ld // 128), dtype=torch.float32, device=q.device)
    fp4q_fp4_row_to_fp8_col_grouped(q, s, R, C, offsets, groups, y, ts, stream)
    return y, ts


def fp4_to_fp8(q, s, stream=None):
    torch = _torch()
    _on_device("q", q)
    _on_device("s", s)
    R, C = q.shape[0], q.shape[1] * 2
    y = torch.empty((R, C), dtype=torch.uint8, device=q.device)
    ts = torch.empty((R, C // 128), dtype=torch.float32, device=q.device)
    fp4q_fp4_to_fp8(q, s, R, C, 1, y, ts, stream)
    return y, ts


def nv_quantize(x, rht=False, rht_seed=0, rounding=FP4Q_RNE, sr_seed=0, amax=None,
                layout=FP4Q_SCALES_ROWMAJOR, block_axis=1, two_d=False, stream=None):
    """BF16 [R, C] -> dict(q, scales, s_t (device [1]), amax (device [1])).

    rht: 0/False none, 1/True random signs from rht_seed, 2 deterministic H16.
    block_axis 0: the quantization of X^T (q [C, R/2]).  two_d: 16x16 tile
    scales (fp4q_nv_quantize_2d; no rotation, block_axis 1)."""
    torch = _torch()
    _on_device("x", x, rows_strided=True)
    _on_device("amax", amax)
    R, C = x.shape
    OR, OC = (R, C) if block_axis == 1 else (C, R)
    q = torch.empty((OR, OC // 2), dtype=torch.uint8, device=x.device)
    s = torch.empty(fp4q_scales_bytes(OR, OC // 16, layout), dtype=torch.uint8, device=x.device)
    st = torch.empty(1, dtype=torch.float32, device=x.device)
    am = torch.empty(1, dtype=torch.float32, device=x.device)
    wsb = fp4q_nv_quantize_workspace_bytes(R, C)
    ws = torch.empty(wsb, dtype=torch.uint8, device=x.device)
    if two_d:
        fp4q_nv_quantize_2d(x, R, C, x.stride(0), rounding, sr_seed, amax, am, st, q, s, layout, ws, wsb, stream)
    else:
        fp4q_nv_quantize(x, R, C, x.stride(0), block_axis, int(rht), rht_seed, rounding, sr_seed, amax, am, st, q,
                         s, layout, ws, wsb, stream)
    return {"q": q, "scales": s.view(OR, OC // 16) if layout == FP4Q_SCALES_ROWMAJOR else s, "s_t": st,
            "amax": am}


def nv_quantize_sr_rne(x, rht=False, rht_seed=0, sr_seed=0, amax=None, layout=FP4Q_SCALES_ROWMAJOR, stream=None):
    """BF16 [R, C] -> dict(q_sr, q_rne, scales, s_t, amax): both roundings over one
    set of scales (fp4q_nv_quantize_sr_rne)."""
    torch = _torch()
    _on_device("x", x, rows_strided=True)
    _on_device("amax", amax)
    R, C = x.shape
    q_sr = torch.empty((R, C // 2), dtype=torch.uint8, device=x.device)
    q_rne = torch.empty((R, C // 2), dtype=torch.uint8, device=x.device)
    s = torch.empty(fp4q_scales_bytes(R, C // 16, layout), dtype=torch.uint8, device=x.device)
    st = torch.empty(1, dtype=torch.float32, device=x.device)
    am = torch.empty(1, dtype=torch.float32, device=x.device)
    wsb = fp4q_nv_quantize_workspace_bytes(R, C)
    ws = torch.empty(wsb, dtype=torch.uint8, device=x.device)
    fp4q_nv_quantize_sr_rne(x, R, C, x.stride(0), int(rht), rht_seed, sr_seed, amax, am, st, q_sr, q_rne, s, layout,
                            ws, wsb, stream)
    return {"q_sr": q_sr, "q_rne": q_rne, "scales": s.view(R, C // 16) if layout == FP4Q_SCALES_ROWMAJOR else s,
            "s_t": st, "amax": am}


def gemm(qa, sa, qb, sb, fmt=FP4Q_MXFP4, ts_a=None, ts_b=None, out_dtype=None, stream=None):
    """D = A . B^T for packed FP4 (or MXFP8) operands with MMA-layout scales.

    qa [M, K/2], qb [N, K/2] uint8 ([M, K], [N, K] E4M3 for MXFP8); sa / sb scale buffers in FP4Q_SCALES_MMA
    layout; ts_a / ts_b device FP32 [1] tensor scales for NVFP4.  Returns a
    [M, N] view of a row-padded output (row stride a multiple of 16 bytes).
    """
    torch = _torch()
    for name, t in (("qa", qa), ("sa", sa), ("qb", qb), ("sb", sb), ("ts_a", ts_a), ("ts_b", ts_b)):
        _on_device(name, t)
    out_dtype = out_dtype or torch.bfloat16
    M, N, K = qa.shape[0], qb.shape[0], qa.shape[1] * (1 if fmt == FP4Q_MXFP8 else 2)
    esz = 2 if out_dtype == torch.bfloat16 else 4
    ldd = (N * esz + 15) // 16 * 16 // esz
    D = torch.empty((M, ldd), dtype=out_dtype, device=qa.device)
    A = make_operand(qa, sa, fmt, ts_a)
    B = make_operand(qb, sb, fmt, ts_b)
    fp4q_block_scaled_gemm(A, B, M, N, K, D, FP4Q_BF16 if out_dtype == torch.bfloat16 else FP4Q_FP32, ldd, stream)
    return D[:, :N]


def moe_dispatch(topk, q, s, n_experts, stream=None):
    """topk int32 [T, k] (device); q [T, C/2], s [T, C/32] ROWMAJOR.  Returns
    dict(offsets int64 [E+1], row_token int32 [T*k], q, s) of the dispatched rows."""
    torch = _torch()
    for name, t in (("topk", topk), ("q", q), ("s", s)):
        _on_device(name, t)
    T, k = topk.shape
    C = q.shape[1] * 2
    dev = q.device
    offsets = torch.empty(n_experts + 1, dtype=torch.int64, device=dev)
    row_token = torch.empty(T * k, dtype=torch.int32, device=dev)
    qo = torch.empty((T * k, C // 2), dtype=torch.uint8, device=dev)
    so = torch.empty((T * k, C // 32), dtype=torch.uint8, device=dev)
    wsb = fp4q_moe_dispatch_workspace_bytes(T, k, n_experts)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    fp4q_moe_dispatch(topk, T, k, n_experts, q, s, C, offsets, row_token, qo, so, ws, wsb, stream)
    return {"offsets": offsets, "row_token": row_token, "q": qo, "s": so}


def mx_rebase_scales(s, offsets, cols, groups, violations=None, stream=None):
    """ROWMAJOR E8M0 [R, cols/32] -> (UE4M3 MMA layout padded per group, FP32 row factor [R])."""
    torch = _torch()
    for name, t in (("s", s), ("offsets", offsets), ("violations", violations)):
        _on_device(name, t)
    R = s.shape[0]
    out = torch.zeros(fp4q_rebased_scales_bytes(R, cols, groups), dtype=torch.uint8, device=s.device)
    rs = torch.empty(R, dtype=torch.float32, device=s.device)
    fp4q_mx_rebase_scales(s, R, cols, offsets, groups, out, rs, violations, stream)
    return out, rs


def grouped_gemm(a_q, a_scales, a_row_scale, b_q, b_scales, b_ts, offsets, groups, N, epilogue=FP4Q_EPI_STORE_BF16,
                 h_debug=False, stream=None):
    """Returns D (BF16 [R, N]) or (h codes [R, N/4], h E8M0 [R, N/64], h FP32 or None) for the gated form."""
    torch = _torch()
    for name, t in (("a_q", a_q), ("a_scales", a_scales), ("a_row_scale", a_row_scale), ("b_q", b_q),
                    ("b_scales", b_scales), ("b_ts", b_ts), ("offsets", offsets)):
        _on_device(name, t)
    R, K = a_q.shape[0], a_q.shape[1] * 2
    dev = a_q.device
    if epilogue == FP4Q_EPI_STORE_BF16:
        D = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
        fp4q_grouped_gemm(a_q, a_scales, a_row_scale, b_q, b_scales, b_ts, offsets, R, groups, N, K, epilogue, D,
                          None, None, stream)
        return D
    hq = torch.empty((R, N // 4), dtype=torch.uint8, device=dev)
    hs = torch.empty((R, N // 64), dtype=torch.uint8, device=dev)
    hd = torch.empty((R, N // 2), dtype=torch.float32, device=dev) if h_debug else None
    fp4q_grouped_gemm(a_q, a_scales, a_row_scale, b_q, b_scales, b_ts, offsets, R, groups, N, K, epilogue, hq, hs,
                      hd, stream)
    return hq, hs, hd
