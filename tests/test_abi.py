"""The C-ABI library loads, exports every entry point include/fp4q.h declares,
and rejects bad arguments before it touches a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w ]*?[\s\*]+(fp4q_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from micro_scaled_fp4_gb300 import _build
    _build.build()
    import micro_scaled_fp4_gb300.fp4q as fq
    return fq


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["fp4q_mx_quantize", "fp4q_mx_dequantize", "fp4q_fp4_to_fp8", "fp4q_nv_quantize",
              "fp4q_block_scaled_gemm", "fp4q_status_string", "fp4q_device_status", "fp4q_stream_status",
              "fp4q_grouped_gemm", "fp4q_nv_quantize_workspace_bytes"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    L = lib.load()
    missing = [n for n in _declared() if getattr(L, n, None) is None]
    assert not missing, missing
    for n in lib.EXPORTED:
        assert getattr(L, n, None) is not None, n


def test_status_strings(lib):
    for code, name in lib.STATUS_NAMES.items():
        assert lib.fp4q_status_string(code) == name
    assert lib.fp4q_status_string(99) == "FP4Q_UNKNOWN_STATUS"


def test_scales_bytes(lib):
    assert lib.fp4q_scales_bytes(256, 128, lib.FP4Q_SCALES_ROWMAJOR) == 256 * 128
    assert lib.fp4q_scales_bytes(256, 128, lib.FP4Q_SCALES_MMA) == 2 * 32 * 512
    assert lib.fp4q_scales_bytes(129, 5, lib.FP4Q_SCALES_MMA) == 2 * 2 * 512
    assert lib.fp4q_scales_bytes(0, 5, lib.FP4Q_SCALES_MMA) == 0
    assert lib.fp4q_nv_quantize_workspace_bytes(8192, 14336) >= 4
    # byte counts that do not fit a size_t give 0 instead of a wrapped size
    huge = (1 << 63) - 1
    for layout in (lib.FP4Q_SCALES_ROWMAJOR, lib.FP4Q_SCALES_MMA):
        assert lib.fp4q_scales_bytes(huge, 4, layout) == 0
        assert lib.fp4q_scales_bytes(1 << 40, 1 << 40, layout) == 0
    assert lib.fp4q_rebased_scales_bytes(huge, 128, 1) == 0
    assert lib.fp4q_rebased_scales_bytes(1 << 40, 1 << 40, 8) == 0
    assert lib.fp4q_rebased_scales_bytes(300, 256, 4) == (3 + 4) * 4 * 512
    # row length of the grouped FP4RowToFP8Col output: 128 * (ceil(rows / 128) + groups)
    assert lib.fp4q_fp4_row_to_fp8_col_grouped_ld(300, 4) == 128 * (3 + 4)
    assert lib.fp4q_fp4_row_to_fp8_col_grouped_ld(0, 1) == 128
    assert lib.fp4q_fp4_row_to_fp8_col_grouped_ld(300, 0) == 0
    assert lib.fp4q_fp4_row_to_fp8_col_grouped_ld(300, 257) == 0
    assert lib.fp4q_fp4_row_to_fp8_col_grouped_ld(1 << 31, 4) == 0


def test_argument_errors_need_no_gpu(lib):
    E = lib.Fp4qError
    x = 1 << 20           # an aligned, never dereferenced address
    cases = [
        (lambda: lib.fp4q_mx_quantize(x, 7, None, 4, 64, 64, 1, x, x, 0, 0), 1),        # bad dtype
        (lambda: lib.fp4q_mx_quantize(x, 0, None, 4, 48, 64, 1, x, x, 0, 0), 2),        # cols % 32
        (lambda: lib.fp4q_mx_quantize(x, 0, None, 4, 64, 64, 0, x, x, 0, 0), 2),        # block axis
        (lambda: lib.fp4q_mx_quantize(x, 2, None, 4, 128, 128, 1, x, x, 0, 0), 1),     # E4M3 w/o scales
        (lambda: lib.fp4q_mx_quantize(x, 2, x, 4, 96, 96, 1, x, x, 0, 0), 2),          # E4M3 cols % 128
        (lambda: lib.fp4q_mx_quantize(x + 16, 0, None, 4, 64, 64, 1, x, x, 0, 0), 3),  # x not 32-B aligned
        (lambda: lib.fp4q_mx_quantize(x, 0, None, 4, 64, 72, 1, x, x, 0, 0), 3),       # ld_x*2 % 32
        (lambda: lib.fp4q_mx_dequantize(x, x, 4, 64, 1, x, 2, 0), 1),                  # y_type
        (lambda: lib.fp4q_fp4_to_fp8(x, x, 4, 96, 1, x, x, 0), 2),                     # cols % 128
        (lambda: lib.fp4q_fp4_to_fp8(None, x, 4, 128, 1, x, x, 0), 1),
        (lambda: lib.fp4q_nv_quantize(x, 4, 24, 24, 1, 0, 0, 0, 0, None, None, x, x, x, 0, x, 256, 0), 2),
        (lambda: lib.fp4q_nv_quantize(x, 4, 32, 32, 1, 0, 0, 5, 0, None, None, x, x, x, 0, x, 256, 0), 1),
        (lambda: lib.fp4q_nv_quantize(x, 4, 32, 32, 1, 0, 0, 0, 0, None, None, x, x, x, 0, None, 0, 0), 1),
        (lambda: lib.fp4q_nv_quantize(x, 4, 32, 32, 1, 0, 0, 0, 0, None, None, None, x, x, 0, x, 256, 0), 1),
    ]
    for fn, status in cases:
        with pytest.raises(E) as e:
            fn()
        assert e.value.status == status, (e.value, status)
    for fn, status in [
        (lambda: lib.fp4q_nv_quantize_2d(x, 8, 64, 64, 0, 0, None, x, x, x, x, 0, x, 256, stream=0), 2),
        (lambda: lib.fp4q_nv_quantize(x, 16, 64, 64, 0, 0, 0, 0, 0, None, x, x, x, x, 0, x, 256, 0), 2),
        (lambda: lib.fp4q_nv_quantize(x, 16, 64, 64, 1, 3, 0, 0, 0, None, x, x, x, x, 0, x, 256, 0), 1),
        (lambda: lib.fp4q_fp4_row_to_fp8_col(x, x, 16, 64, x, x, stream=0), 2),
        (lambda: lib.fp4q_fp4_row_to_fp8_col(x + 16, x, 128, 128, x, x, stream=0), 3),
        (lambda: lib.fp4q_mx_quantize(x, 1, None, 128, 128, 128, 0, x, x, 0, 0), 2),
    ]:
        with pytest.raises(E) as e:
            fn()
        assert e.value.status == status, (e.value, status)
    # host-buffer FP8 path: every argument error is returned before any CUDA call
    wsb = lib.fp4q_fp8_pipeline_host_workspace_bytes(256, 64)
    for fn, status in [
        (lambda: lib.fp4q_fp8_pipeline_host(x, x, -1, 256, x, x, x, x, 64, x, wsb, stream=0), 1),
        (lambda: lib.fp4q_fp8_pipeline_host(x, x, 64, 256, x, x, x, x, -5, x, wsb, stream=0), 1),
        (lambda: lib.fp4q_fp8_pipeline_host(x, x, 64, 192, x, x, x, x, 64, x, wsb, stream=0), 2),
        (lambda: lib.fp4q_fp8_pipeline_host(x, None, 64, 256, x, x, x, x, 64, x, wsb, stream=0), 1),
        (lambda: lib.fp4q_fp8_pipeline_host(x, x, 64, 256, x, x, None, x, 64, x, wsb, stream=0), 1),
        (lambda: lib.fp4q_fp8_pipeline_host(x, x, 64, 256, x, x, x, x, 64, x + 128, wsb, stream=0), 3),
        (lambda: lib.fp4q_fp8_pipeline_host(x, x, 64, 256, x, x, x, x, 64, x, wsb - 1, stream=0), 1),
        (lambda: lib.fp4q_fp8_pipeline_host(x, x, 200, 256, x, x, x, x, 128, x, wsb, stream=0), 1),
        (lambda: lib.fp4q_fp8_pipeline_host(x, x, 1 << 41, 7168, x, x, x, x, 1 << 41, x, wsb, stream=0), 2),
        (lambda: lib.fp4q_fp4_row_to_fp8_col_grouped(x, x, -1, 256, x, 4, x, x, stream=0), 1),
        (lambda: lib.fp4q_fp4_row_to_fp8_col_grouped(x, x, 300, 256, x, 0, x, x, stream=0), 1),
        (lambda: lib.fp4q_fp4_row_to_fp8_col_grouped(x, x, 300, 256, x, 257, x, x, stream=0), 1),
        (lambda: lib.fp4q_fp4_row_to_fp8_col_grouped(x, x, 300, 192, x, 4, x, x, stream=0), 2),
        (lambda: lib.fp4q_fp4_row_to_fp8_col_grouped(x, x, 1 << 31, 256, x, 4, x, x, stream=0), 2),
        (lambda: lib.fp4q_fp4_row_to_fp8_col_grouped(x, x, 300, 256, None, 4, x, x, stream=0), 1),
        (lambda: lib.fp4q_fp4_row_to_fp8_col_grouped(x + 16, x, 300, 256, x, 4, x, x, stream=0), 3),
        (lambda: lib.fp4q_fp4_row_to_fp8_col_grouped(x, x, 300, 256, x + 4, 4, x, x, stream=0), 3),
    ]:
        with pytest.raises(E) as e:
            fn()
        assert e.value.status == status, (e.value, status)
    for limit in (0, 3_000_000_000):
        with pytest.raises(E) as e:
            lib.fp4q_check_wait_timeout(limit, stream=0)
        assert e.value.status == 1
    with pytest.raises(E) as e:       # scratch of the static-array dispatch would not fit
        lib.fp4q_moe_dispatch_static(x, 1 << 22, 8, 64, x, x, 64, x, x, x, x, stream=0)
    assert e.value.status == 2
    # token counts whose dispatched rows (tokens x top_k) leave int32: rejected
    # before any size arithmetic can wrap, and the workspace size says 0
    for T, k in [(1 << 61, 8), ((2**31 - 1) // 8 + 1, 8), (1 << 31, 1)]:
        assert lib.fp4q_moe_dispatch_workspace_bytes(T, k, 64) == 0
        for fn in (lambda: lib.fp4q_moe_dispatch(x, T, k, 64, x, x, 64, x, x, x, x, x, 1 << 40, stream=0),
                   lambda: lib.fp4q_moe_dispatch_static(x, T, k, 64, x, x, 64, x, x, x, x, stream=0)):
            with pytest.raises(E) as e:
                fn()
            assert e.value.status == 2 and "2^31" in str(e.value), (T, k, e.value)
    assert lib.fp4q_moe_dispatch_workspace_bytes((2**31 - 1) // 8, 8, 64) > 0
    A = lib.make_operand(x, x, lib.FP4Q_MXFP4)
    B = lib.make_operand(x, x, lib.FP4Q_NVFP4, x)
    for args, status in [((A, B, 128, 128, 128, x, 0, 128), 1), ((A, A, 128, 128, 96, x, 0, 128), 2),
                         ((A, A, 128, 128, 128, x + 2, 0, 128), 3), ((A, A, 128, 128, 128, x, 0, 100), 1),
                         ((A, A, 128, 128, 128, x, 0, 132), 3),
                         ((A, A, 1 << 30, 1 << 30, 128, x, 0, 1 << 30), 2)]:     # 2^45 output tiles
        with pytest.raises(E) as e:
            lib.fp4q_block_scaled_gemm(*args, stream=0)
        assert e.value.status == status, (args, e.value)
    with pytest.raises(E) as e:       # E8M0 scales not 4-byte aligned
        lib.fp4q_mx_rebase_scales(x + 2, 4, 128, x, 1, x, x, None, stream=0)
    assert e.value.status == 3
    with pytest.raises(E) as e:       # 2^43 output tiles of the grouped form
        lib.fp4q_grouped_gemm(x, x, x, x, x, x, x, 1 << 30, 4, 1 << 28, 128, 0, x, None, None, stream=0)
    assert e.value.status == 2


def test_fp8_pipeline_host_workspace_bytes(lib):
    # three slots of one chunk: E4M3 in, tile scales, codes, E8M0, E4M3 out, tile scales (each 256-B aligned)
    def slot(n, c):
        a = lambda v: (v + 255) // 256 * 256
        return a(n * c) + a(n * c // 128 * 4) + a(n * c // 2) + a(n * c // 32) + a(n * c) + a(n * c // 128 * 4)
    assert lib.fp4q_fp8_pipeline_host_workspace_bytes(7168, 1024) == 3 * slot(1024, 7168)
    assert lib.fp4q_fp8_pipeline_host_workspace_bytes(7168, 0) == 3 * slot(2048, 7168)
    assert lib.fp4q_fp8_pipeline_host_workspace_bytes(128, 3) == 3 * slot(3, 128)
    assert lib.fp4q_fp8_pipeline_host_workspace_bytes(0, 64) == 0
    assert lib.fp4q_fp8_pipeline_host_workspace_bytes(1 << 32, 64) == 0          # cols > 2^31
    assert lib.fp4q_fp8_pipeline_host_workspace_bytes(7168, 1 << 62) == 0        # chunk past 2^40 elements


def test_empty_tensors_are_no_ops(lib):
    lib.fp4q_fp8_pipeline_host(None, None, 0, 256, None, None, None, None, 0, None, 0, stream=0)
    lib.fp4q_mx_quantize(None, 0, None, 0, 64, 64, 1, None, None, 0, 0)
    lib.fp4q_mx_dequantize(None, None, 0, 64, 1, None, 0, 0)
    lib.fp4q_fp4_to_fp8(None, None, 5, 0, 1, None, None, 0)


def test_no_cpu_fallback_when_library_missing(monkeypatch, tmp_path):
    # the binding refuses to run without the compiled library (no silent fallback)
    import micro_scaled_fp4_gb300.fp4q as fq
    from micro_scaled_fp4_gb300 import _build
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(fq, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        fq.load()


def test_helpers_reject_host_and_strided_tensors(lib):
    """The allocating helpers check their tensors before any address reaches
    the library: a host tensor, or a transposed one, is a ValueError."""
    import torch
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    for call in (lambda: lib.mx_quantize(x), lambda: lib.nv_quantize(x),
                 lambda: lib.fp4_to_fp8(torch.zeros((4, 64), dtype=torch.uint8), torch.zeros((4, 4), dtype=torch.uint8)),
                 lambda: lib.gemm(*(torch.zeros((128, 64), dtype=torch.uint8),) * 4)):
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
    with pytest.raises(ValueError, match="host tensor"):
        lib.fp8_pipeline_host(torch.zeros((128, 256), dtype=torch.uint8).t(), torch.zeros((128, 2)))
