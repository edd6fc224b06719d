"""Python binding of libbsq.so (block-scaled quantization and GEMM, sm_103a).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  PyTorch provides device memory and streams.  There is no
fallback: if libbsq.so is missing or fails to load, every call raises.

Names follow the C ABI in ``include/bsq.h``:

    quantize(x, fmt, axis)            -> (row QTensor | None, col QTensor | None)
    dequantize(q, dtype)              -> torch.Tensor
    gemm(A, B, dtype)                 -> torch.Tensor  C = A @ B^T
    grouped_gemm(A, offsets, B, dtype)-> torch.Tensor  per-group A_g @ B_g^T
    mxfp4_to_mxfp8(q)                 -> QTensor
    sync_status()                     -> raises BsqError on a recorded device fault
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbsq.so")

MXFP8_E4M3, MXFP8_E5M2, MXFP4_E2M1, NVFP4_E2M1 = 0, 1, 2, 3
FORMATS = {"mxfp8_e4m3": MXFP8_E4M3, "mxfp8_e5m2": MXFP8_E5M2, "mxfp4": MXFP4_E2M1, "nvfp4": NVFP4_E2M1}
ROWWISE, COLWISE, BOTH = 1, 2, 3
AXES = {"row": ROWWISE, "col": COLWISE, "both": BOTH}
OUT_F32, OUT_BF16 = 0, 1

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "alignment", 4: "cuda error", 5: "timeout"}


class BsqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)} (status {status})")
        self.status = status


class BsqTensorC(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p)]


_lib = None


def lib():
    """Load libbsq.so (raises if it is missing: there is no other path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libbsq.so not built ({LIB_PATH}); run block_scaled_precision_03_gb300._build.build()")
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    PT = ctypes.POINTER(BsqTensorC)
    sig = {
        "bsq_codes_bytes": (sz, [i32, i64, i64]),
        "bsq_scales_bytes": (sz, [i32, i64, i64]),
        "bsq_quantize": (i32, [vp, i64, i64, i32, i32, PT, PT, vp]),
        "bsq_quantize_nvfp4_delayed": (i32, [vp, i64, i64, i32, PT, PT, vp, i32, vp]),
        "bsq_dequantize": (i32, [PT, vp, i32, vp]),
        "bsq_gemm": (i32, [PT, PT, vp, i32, vp]),
        "bsq_grouped_gemm": (i32, [PT, vp, i32, PT, vp, i32, vp]),
        "bsq_grouped_gemm_padded": (i32, [PT, vp, i32, PT, vp, i32, vp]),
        "bsq_grouped_scales_bytes": (sz, [i32, i64, i64, i32]),
        "bsq_mxfp4_to_mxfp8_grouped": (i32, [PT, PT, vp, i32, vp]),
        "bsq_mxfp4_to_mxfp8": (i32, [PT, PT, vp]),
        "bsq_mxfp4_to_mxfp8_col": (i32, [PT, PT, vp]),
        "bsq_mxfp4_to_fp8_1x128": (i32, [PT, vp, vp, vp]),
        "bsq_sync_status": (i32, [vp]),
        "bsq_debug_timeout_probe": (i32, [ctypes.c_uint64, vp]),
        "bsq_debug_gemm_timeout": (i32, [PT, PT, vp, i32, ctypes.c_uint64, i32, vp]),
        "bsq_status_string": (ctypes.c_char_p, [i32]),
        "bsq_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(status: int, what: str):
    if status != 0:
        raise BsqError(status, what)


def _fmt(f) -> int:
    return FORMATS[f] if isinstance(f, str) else int(f)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def codes_bytes(fmt, rows: int, cols: int) -> int:
    return int(lib().bsq_codes_bytes(_fmt(fmt), rows, cols))


def scales_bytes(fmt, rows: int, cols: int) -> int:
    return int(lib().bsq_scales_bytes(_fmt(fmt), rows, cols))


@dataclass
class QTensor:
    """A quantized tensor: device buffers plus its C descriptor."""
    fmt: int
    rows: int
    cols: int
    codes: "object"           # torch.uint8 [codes_bytes]
    scales: "object"          # torch.uint8 [scales_bytes]
    tensor_scale: "object"    # torch.float32 [1] (NVFP4) or None

    def c(self) -> BsqTensorC:
        return BsqTensorC(self.fmt, 0, self.rows, self.cols, self.codes.data_ptr(), self.scales.data_ptr(),
                          self.tensor_scale.data_ptr() if self.tensor_scale is not None else None)


def empty(fmt, rows: int, cols: int, device="cuda") -> QTensor:
    import torch
    f = _fmt(fmt)
    nc, ns = codes_bytes(f, rows, cols), scales_bytes(f, rows, cols)
    if nc == 0 or ns == 0:
        raise BsqError(1, f"shape {rows}x{cols} not valid for format {f}")
    ts = torch.zeros(1, dtype=torch.float32, device=device) if f == NVFP4_E2M1 else None
    return QTensor(f, rows, cols, torch.empty(nc, dtype=torch.uint8, device=device),
                   torch.empty(ns, dtype=torch.uint8, device=device), ts)


def quantize_into(x, fmt, axis, out_row: QTensor | None, out_col: QTensor | None, stream=None):
    f, a = _fmt(fmt), AXES[axis] if isinstance(axis, str) else int(axis)
    R, C = x.shape
    cr = out_row.c() if out_row is not None else None
    cc = out_col.c() if out_col is not None else None
    st = lib().bsq_quantize(ctypes.c_void_p(x.data_ptr()), R, C, f, a,
                            ctypes.byref(cr) if cr is not None else None,
                            ctypes.byref(cc) if cc is not None else None, _stream(stream))
    _check(st, "bsq_quantize")


def quantize(x, fmt, axis="row", stream=None):
    """Quantize a contiguous BF16 CUDA matrix; returns (row, col) QTensors."""
    import torch
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous()
    a = AXES[axis] if isinstance(axis, str) else int(axis)
    R, C = x.shape
    row = empty(fmt, R, C, x.device) if a & ROWWISE else None
    col = empty(fmt, C, R, x.device) if a & COLWISE else None
    quantize_into(x, fmt, a, row, col, stream)
    return row, col


def quantize_nvfp4_delayed_into(x, axis, out_row: QTensor | None, out_col: QTensor | None, history, stream=None):
    """NVFP4 quantize with delayed scaling into given tensors; `history` is a
    float32 CUDA tensor of past amax values, updated in place."""
    import torch
    assert history.dtype == torch.float32 and history.is_cuda and history.is_contiguous()
    a = AXES[axis] if isinstance(axis, str) else int(axis)
    R, C = x.shape
    cr = out_row.c() if out_row is not None else None
    cc = out_col.c() if out_col is not None else None
    st = lib().bsq_quantize_nvfp4_delayed(ctypes.c_void_p(x.data_ptr()), R, C, a,
                                          ctypes.byref(cr) if cr is not None else None,
                                          ctypes.byref(cc) if cc is not None else None,
                                          ctypes.c_void_p(history.data_ptr()), history.numel(), _stream(stream))
    _check(st, "bsq_quantize_nvfp4_delayed")


def quantize_nvfp4_delayed(x, history, axis="row", stream=None):
    """NVFP4 quantize of a contiguous BF16 CUDA matrix with the tensor scale
    taken from `history` (see bsq_quantize_nvfp4_delayed); returns (row, col)."""
    import torch
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous()
    a = AXES[axis] if isinstance(axis, str) else int(axis)
    R, C = x.shape
    row = empty("nvfp4", R, C, x.device) if a & ROWWISE else None
    col = empty("nvfp4", C, R, x.device) if a & COLWISE else None
    quantize_nvfp4_delayed_into(x, a, row, col, history, stream)
    return row, col


def dequantize_into(q: QTensor, out, stream=None):
    """Exact dequantization into `out` ([rows, cols] float32 or bfloat16)."""
    import torch
    c = q.c()
    st = lib().bsq_dequantize(ctypes.byref(c), ctypes.c_void_p(out.data_ptr()),
                              OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32, _stream(stream))
    _check(st, "bsq_dequantize")
    return out


def dequantize(q: QTensor, dtype=None, stream=None):
    import torch
    dtype = dtype or torch.float32
    out = torch.empty((q.rows, q.cols), dtype=dtype, device=q.codes.device)
    return dequantize_into(q, out, stream)


def gemm_into(A: QTensor, B: QTensor, C, stream=None):
    import torch
    ca, cb = A.c(), B.c()
    st = lib().bsq_gemm(ctypes.byref(ca), ctypes.byref(cb), ctypes.c_void_p(C.data_ptr()),
                        OUT_BF16 if C.dtype == torch.bfloat16 else OUT_F32, _stream(stream))
    _check(st, "bsq_gemm")
    return C


def gemm(A: QTensor, B: QTensor, dtype=None, stream=None):
    import torch
    dtype = dtype or torch.float32
    C = torch.empty((A.rows, B.rows), dtype=dtype, device=A.codes.device)
    return gemm_into(A, B, C, stream)


def group_views(B: QTensor, groups: int) -> list[QTensor]:
    """Split a quantized [groups * N, K] matrix into per-group [N, K] views.

    Requires N to be a multiple of 128 so that each group's scales are whole
    128-row tiles of the combined scale buffer."""
    N = B.rows // groups
    assert N * groups == B.rows and N % 128 == 0
    cb, sb = codes_bytes(B.fmt, N, B.cols), scales_bytes(B.fmt, N, B.cols)
    return [QTensor(B.fmt, N, B.cols, B.codes[g * cb:(g + 1) * cb], B.scales[g * sb:(g + 1) * sb], B.tensor_scale)
            for g in range(groups)]


def _check_offsets(offsets_dev, groups: int):
    """The C ABI reads groups + 1 int64 row offsets from device memory and
    cannot check them; a wrong tensor is rejected here."""
    import torch
    if not (isinstance(offsets_dev, torch.Tensor) and offsets_dev.dtype == torch.int64 and offsets_dev.is_cuda
            and offsets_dev.is_contiguous() and offsets_dev.numel() == groups + 1):
        raise BsqError(1, f"group offsets must be a contiguous int64 CUDA tensor of {groups + 1} entries")


def grouped_gemm_into(A: QTensor, offsets_dev, B_groups: list[QTensor], C, stream=None, padded_scales=False):
    """Grouped GEMM into C; padded_scales: A's scales are in the per-expert
    padded layout (from mxfp4_to_mxfp8_grouped)."""
    import torch
    _check_offsets(offsets_dev, len(B_groups))
    ca = A.c()
    arr = (BsqTensorC * len(B_groups))(*[b.c() for b in B_groups])
    f = lib().bsq_grouped_gemm_padded if padded_scales else lib().bsq_grouped_gemm
    st = f(ctypes.byref(ca), ctypes.c_void_p(offsets_dev.data_ptr()), len(B_groups), arr, ctypes.c_void_p(C.data_ptr()),
           OUT_BF16 if C.dtype == torch.bfloat16 else OUT_F32, _stream(stream))
    _check(st, "bsq_grouped_gemm")
    return C


def grouped_gemm(A: QTensor, offsets_dev, B_groups: list[QTensor], dtype=None, stream=None, padded_scales=False):
    import torch
    dtype = dtype or torch.float32
    C = torch.empty((A.rows, B_groups[0].rows), dtype=dtype, device=A.codes.device)
    return grouped_gemm_into(A, offsets_dev, B_groups, C, stream, padded_scales)


def mxfp4_to_mxfp8_into(q: QTensor, out: QTensor, stream=None):
    ci, co = q.c(), out.c()
    _check(lib().bsq_mxfp4_to_mxfp8(ctypes.byref(ci), ctypes.byref(co), _stream(stream)), "bsq_mxfp4_to_mxfp8")
    return out


def mxfp4_to_mxfp8(q: QTensor, stream=None) -> QTensor:
    out = empty(MXFP8_E4M3, q.rows, q.cols, q.codes.device)
    return mxfp4_to_mxfp8_into(q, out, stream)


def grouped_scales_bytes(fmt, rows: int, cols: int, groups: int) -> int:
    return int(lib().bsq_grouped_scales_bytes(_fmt(fmt), rows, cols, groups))


def empty_grouped(fmt, rows: int, cols: int, groups: int, device="cuda") -> QTensor:
    """Uninitialized tensor whose scale buffer holds the per-expert padded layout."""
    import torch
    q = empty(fmt, rows, cols, device)
    q.scales = torch.empty(grouped_scales_bytes(fmt, rows, cols, groups), dtype=torch.uint8, device=device)
    return q


def mxfp4_to_mxfp8_grouped_into(q: QTensor, out: QTensor, offsets_dev, groups: int, stream=None):
    _check_offsets(offsets_dev, groups)
    ci, co = q.c(), out.c()
    _check(lib().bsq_mxfp4_to_mxfp8_grouped(ctypes.byref(ci), ctypes.byref(co), ctypes.c_void_p(offsets_dev.data_ptr()),
                                            groups, _stream(stream)), "bsq_mxfp4_to_mxfp8_grouped")


def mxfp4_to_mxfp8_grouped(q: QTensor, offsets_dev, groups: int, stream=None) -> QTensor:
    """MXFP4 -> MXFP8 E4M3 with the scales in the per-expert padded layout."""
    out = empty_grouped("mxfp8_e4m3", q.rows, q.cols, groups, q.codes.device)
    mxfp4_to_mxfp8_grouped_into(q, out, offsets_dev, groups, stream)
    return out


def mxfp4_to_mxfp8_col_into(q: QTensor, out: QTensor, stream=None):
    ci, co = q.c(), out.c()
    _check(lib().bsq_mxfp4_to_mxfp8_col(ctypes.byref(ci), ctypes.byref(co), _stream(stream)), "bsq_mxfp4_to_mxfp8_col")


def mxfp4_to_fp8_1x128_into(q: QTensor, codes, scales, stream=None):
    """codes: uint8 [rows, cols] E4M3; scales: uint8 [rows, ceil(cols/128)] E8M0."""
    ci = q.c()
    _check(lib().bsq_mxfp4_to_fp8_1x128(ctypes.byref(ci), ctypes.c_void_p(codes.data_ptr()),
                                        ctypes.c_void_p(scales.data_ptr()), _stream(stream)), "bsq_mxfp4_to_fp8_1x128")


def mxfp4_to_fp8_1x128(q: QTensor, stream=None):
    """MXFP4 -> FP8 E4M3 with 1x128 blocks; returns (codes [rows, cols],
    scales [rows, ceil(cols/128)]), both uint8 on the input's device."""
    import torch
    dev = q.codes.device
    codes = torch.empty((q.rows, q.cols), dtype=torch.uint8, device=dev)
    scales = torch.empty((q.rows, (q.cols + 127) // 128), dtype=torch.uint8, device=dev)
    mxfp4_to_fp8_1x128_into(q, codes, scales, stream)
    return codes, scales


def mxfp4_to_mxfp8_col(q: QTensor, stream=None) -> QTensor:
    """FP4RowToFP8Col: [R, C] MXFP4 (row-wise) -> [C, R] MXFP8 E4M3 of the transpose."""
    out = empty("mxfp8_e4m3", q.cols, q.rows, q.codes.device)
    mxfp4_to_mxfp8_col_into(q, out, stream)
    return out


def sync_status(stream=None):
    _check(lib().bsq_sync_status(_stream(stream)), "device status")


def debug_timeout_probe(limit_ns: int, stream=None):
    _check(lib().bsq_debug_timeout_probe(limit_ns, _stream(stream)), "bsq_debug_timeout_probe")


def debug_gemm_timeout_into(A: QTensor, B: QTensor, C, timeout_ns: int, kernel: int = 0, stream=None):
    """bsq_gemm into C with every wait of the kernel limited to timeout_ns
    (test hook for the failure path; see bsq_debug_gemm_timeout)."""
    import torch
    ca, cb = A.c(), B.c()
    st = lib().bsq_debug_gemm_timeout(ctypes.byref(ca), ctypes.byref(cb), ctypes.c_void_p(C.data_ptr()),
                                      OUT_BF16 if C.dtype == torch.bfloat16 else OUT_F32, timeout_ns, kernel,
                                      _stream(stream))
    _check(st, "bsq_debug_gemm_timeout")


def version() -> str:
    return lib().bsq_version().decode()
