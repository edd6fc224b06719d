"""CPU-side checks of the C ABI: the library builds, loads without a GPU and
exports every entry point declared in include/bsq.h; the size functions and
host-side argument checks behave as documented (no device work)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_scaled_precision_03_gb300 import _build
    import block_scaled_precision_03_gb300 as bsq
    _build.build()
    return bsq.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "bsq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bsq_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_boundary():
    names = declared_functions()
    for need in ["bsq_quantize", "bsq_dequantize", "bsq_gemm", "bsq_grouped_gemm", "bsq_mxfp4_to_mxfp8",
                 "bsq_codes_bytes", "bsq_scales_bytes", "bsq_sync_status", "bsq_status_string"]:
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_size_functions(lib):
    import block_scaled_precision_03_gb300 as bsq
    assert bsq.codes_bytes("mxfp8_e4m3", 8192, 4096) == 8192 * 4096
    assert bsq.codes_bytes("nvfp4", 8192, 4096) == 8192 * 2048
    assert bsq.scales_bytes("mxfp8_e4m3", 8192, 4096) == 8192 * 128
    assert bsq.scales_bytes("nvfp4", 8192, 4096) == 8192 * 256
    assert bsq.scales_bytes("mxfp4", 130, 96) == 256 * 4        # rows -> 256, 3 scales -> 4
    assert bsq.scales_bytes("mxfp8_e4m3", 10, 48) == 0           # cols not a block multiple
    assert bsq.codes_bytes(7, 1, 1) == 0


def test_grouped_scales_bytes_holds_every_offset_set(lib):
    # the per-expert padded layout needs sum_g ceil(count_g / 128) * 128 scale
    # rows (computed by the oracle); the size function's capacity must hold it
    # for any counts, and it rejects bad group counts and shapes
    import numpy as np
    import oracle
    import block_scaled_precision_03_gb300 as bsq
    rng = np.random.default_rng(70)
    for _ in range(200):
        G = int(rng.integers(1, 257))
        R = int(rng.integers(1, 5000))
        S = int(rng.integers(1, 12))
        cuts = np.sort(rng.integers(0, R + 1, G - 1))
        off = np.concatenate([[0], cuts, [R]]).astype(np.int64)
        _, total = oracle.grouped_scale_starts(off)
        cap = bsq.grouped_scales_bytes("mxfp8_e4m3", R, 32 * S, G)
        s_pad = (S + 3) // 4 * 4
        assert cap % (128 * s_pad) == 0 and cap >= total * s_pad, (G, R, S, cap, total)
    assert bsq.grouped_scales_bytes("mxfp8_e4m3", 1024, 256, 0) == 0
    assert bsq.grouped_scales_bytes("mxfp8_e4m3", 1024, 256, 257) == 0
    assert bsq.grouped_scales_bytes("mxfp8_e4m3", 1024, 48, 4) == 0


def test_host_argument_checks_launch_nothing(lib):
    import block_scaled_precision_03_gb300 as bsq
    T = bsq.BsqTensorC
    null = ctypes.c_void_p(None)
    # null source, bad axis, bad format: rejected before any CUDA call
    assert lib.bsq_quantize(None, 128, 128, 0, 1, None, None, null) == 1
    assert lib.bsq_quantize(ctypes.c_void_p(256), 128, 128, 0, 9, None, None, null) == 1
    assert lib.bsq_quantize(ctypes.c_void_p(256), 128, 128, 9, 1, None, None, null) == 1
    # misaligned source pointer
    t = T(0, 0, 128, 128, 256, 256, None)
    assert lib.bsq_quantize(ctypes.c_void_p(258), 128, 128, 0, 1, ctypes.byref(t), None, null) == 3
    # shape mismatch between request and output descriptor
    t2 = T(0, 0, 64, 128, 256, 256, None)
    assert lib.bsq_quantize(ctypes.c_void_p(256), 128, 128, 0, 1, ctypes.byref(t2), None, null) == 1
    # unsupported GEMM pairs
    a = T(0, 0, 128, 256, 256, 256, None)
    b = T(3, 0, 128, 256, 256, 256, 256)
    assert lib.bsq_gemm(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(256), 0, null) == 2
    b2 = T(0, 0, 128, 512, 256, 256, None)
    assert lib.bsq_gemm(ctypes.byref(a), ctypes.byref(b2), ctypes.c_void_p(256), 0, null) == 1
    # repack needs MXFP4 in, E4M3 out
    assert lib.bsq_mxfp4_to_mxfp8(ctypes.byref(a), ctypes.byref(a), null) == 2
    assert lib.bsq_status_string(5) == b"device wait timed out"
    # delayed NVFP4: history pointer and length are checked before anything else
    t4 = bsq.BsqTensorC(3, 0, 128, 128, 256, 512, 1024)
    assert lib.bsq_quantize_nvfp4_delayed(ctypes.c_void_p(256), 128, 128, 1, ctypes.byref(t4), None, None, 16, null) == 1
    assert lib.bsq_quantize_nvfp4_delayed(ctypes.c_void_p(256), 128, 128, 1, ctypes.byref(t4), None,
                                          ctypes.c_void_p(4096), 0, null) == 1
    assert lib.bsq_quantize_nvfp4_delayed(ctypes.c_void_p(256), 128, 128, 1, ctypes.byref(t4), None,
                                          ctypes.c_void_p(4098), 16, null) == 3
    assert lib.bsq_quantize_nvfp4_delayed(None, 128, 128, 1, ctypes.byref(t4), None, ctypes.c_void_p(4096), 16, null) == 1
    # grouped GEMM: offsets, group count, NVFP4, output type and alignment, and
    # expert weights that are not consecutive slices of one allocation
    ga = T(0, 0, 512, 256, 256, 256, None)
    gb = (T * 2)(T(0, 0, 128, 256, 4096, 8192, None), T(0, 0, 128, 256, 4096 + 128 * 256, 8448, None))
    C = ctypes.c_void_p(1 << 20)
    off = ctypes.c_void_p(1 << 16)
    assert lib.bsq_grouped_gemm(ctypes.byref(ga), None, 2, gb, C, 1, null) == 1
    assert lib.bsq_grouped_gemm(ctypes.byref(ga), off, 0, gb, C, 1, null) == 1
    assert lib.bsq_grouped_gemm(ctypes.byref(ga), off, 257, gb, C, 1, null) == 2
    assert lib.bsq_grouped_gemm(ctypes.byref(ga), off, 2, gb, C, 7, null) == 1
    assert lib.bsq_grouped_gemm(ctypes.byref(ga), off, 2, gb, ctypes.c_void_p((1 << 20) + 8), 1, null) == 3
    gbad = (T * 2)(T(0, 0, 128, 256, 4096, 8192, None), T(0, 0, 128, 256, 4096 + 128 * 256 + 16, 8448, None))
    assert lib.bsq_grouped_gemm(ctypes.byref(ga), off, 2, gbad, C, 1, null) == 2
    gshape = (T * 2)(T(0, 0, 128, 256, 4096, 8192, None), T(0, 0, 64, 256, 4096 + 128 * 256, 8448, None))
    assert lib.bsq_grouped_gemm_padded(ctypes.byref(ga), off, 2, gshape, C, 1, null) == 1
    gnv = T(3, 0, 512, 256, 256, 256, 512)
    gbnv = (T * 1)(T(3, 0, 128, 256, 4096, 8192, 512))
    assert lib.bsq_grouped_gemm(ctypes.byref(gnv), off, 1, gbnv, C, 1, null) == 2
    # empty tensors are rejected before any launch
    e0 = T(0, 0, 0, 256, 4096, 8192, None)
    e4 = T(2, 0, 0, 256, 4096, 8192, None)
    assert lib.bsq_quantize(ctypes.c_void_p(256), 0, 128, 0, 1, ctypes.byref(e0), None, null) == 1
    assert lib.bsq_quantize(ctypes.c_void_p(256), 128, 0, 0, 1, ctypes.byref(e0), None, null) == 1
    assert lib.bsq_dequantize(ctypes.byref(e0), ctypes.c_void_p(1 << 20), 0, null) == 1
    assert lib.bsq_gemm(ctypes.byref(e0), ctypes.byref(a), ctypes.c_void_p(1 << 20), 0, null) == 1
    assert lib.bsq_mxfp4_to_mxfp8(ctypes.byref(e4), ctypes.byref(e0), null) == 1
    assert lib.bsq_mxfp4_to_mxfp8_col(ctypes.byref(e4), ctypes.byref(e0), null) == 1
    assert lib.bsq_mxfp4_to_fp8_1x128(ctypes.byref(e4), ctypes.c_void_p(4096), ctypes.c_void_p(8192), null) == 1
    # row counts past the 32-bit row indexing of the GEMM and grouped kernels
    big = 0x7FFFFF00 + 32
    ab = T(0, 0, big, 256, 256, 256, None)
    assert lib.bsq_gemm(ctypes.byref(ab), ctypes.byref(a), ctypes.c_void_p(1 << 20), 0, null) == 2
    assert lib.bsq_gemm(ctypes.byref(a), ctypes.byref(ab), ctypes.c_void_p(1 << 20), 0, null) == 2
    assert lib.bsq_grouped_gemm(ctypes.byref(ab), off, 2, gb, C, 1, null) == 2
    gbig = (T * 2)(T(0, 0, big // 2, 256, 4096, 8192, None), T(0, 0, big // 2, 256, 4096 + (big // 2) * 256, 8448, None))
    assert lib.bsq_grouped_gemm(ctypes.byref(ga), off, 2, gbig, C, 1, null) == 2
    i4 = T(2, 0, big, 256, 256, 256, None)
    o8 = T(0, 0, big, 256, 4096, 8192, None)
    assert lib.bsq_mxfp4_to_mxfp8_grouped(ctypes.byref(i4), ctypes.byref(o8), off, 4, null) == 2
    # 1x128 re-encode: MXFP4 input, both output pointers, 16-byte aligned codes
    t5 = bsq.BsqTensorC(2, 0, 64, 256, 256, 512, None)
    assert lib.bsq_mxfp4_to_fp8_1x128(ctypes.byref(a), ctypes.c_void_p(4096), ctypes.c_void_p(8192), null) == 2
    assert lib.bsq_mxfp4_to_fp8_1x128(ctypes.byref(t5), None, ctypes.c_void_p(8192), null) == 1
    assert lib.bsq_mxfp4_to_fp8_1x128(ctypes.byref(t5), ctypes.c_void_p(4096), None, null) == 1
    assert lib.bsq_mxfp4_to_fp8_1x128(ctypes.byref(t5), ctypes.c_void_p(4104), ctypes.c_void_p(8192), null) == 3
    # GEMM wait-limit hook: the limit and the kernel selector are checked first
    C = ctypes.c_void_p(1 << 20)
    assert lib.bsq_debug_gemm_timeout(ctypes.byref(a), ctypes.byref(a), C, 0, 0, 0, null) == 1
    assert lib.bsq_debug_gemm_timeout(ctypes.byref(a), ctypes.byref(a), C, 0, 4_000_000_001, 0, null) == 1
    assert lib.bsq_debug_gemm_timeout(ctypes.byref(a), ctypes.byref(a), C, 0, 1000, 2, null) == 1
    assert lib.bsq_debug_gemm_timeout(ctypes.byref(a), ctypes.byref(b2), C, 0, 1000, 0, null) == 1
    m4 = T(2, 0, 128, 256, 256, 256, None)
    assert lib.bsq_debug_gemm_timeout(ctypes.byref(m4), ctypes.byref(m4), C, 0, 1000, 1, null) == 2


def test_binding_rejects_bad_group_offsets():
    """The grouped calls read int64 device offsets the C ABI cannot check:
    the binding rejects a wrong dtype, a host tensor, a strided view or a
    wrong length before any CUDA call."""
    import torch
    import block_scaled_precision_03_gb300 as bsq
    A = bsq.QTensor(0, 256, 256, None, None, None)
    groups = [bsq.QTensor(0, 128, 256, None, None, None)] * 2
    bad = [torch.zeros(3, dtype=torch.int32), torch.zeros(3, dtype=torch.int64), torch.zeros(6, dtype=torch.int64)[::2],
           torch.zeros(4, dtype=torch.int64)]
    for off in bad:
        with pytest.raises(bsq.BsqError):
            bsq.grouped_gemm_into(A, off, groups, None)
        with pytest.raises(bsq.BsqError):
            bsq.mxfp4_to_mxfp8_grouped_into(A, A, off, 2)
