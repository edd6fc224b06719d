"""CPU oracle for the block-scaled low-precision linear layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
CPU-baseline leg of the benchmark may import this package.  The library
(``block_scaled_precision_03_gb300``) never imports it, and this package
never imports the library: the two share no code, tables or constants.
Inputs reach both sides from the seeded generators in
``block_scaled_precision_03_gb300.inputs``, which hold none of the
method's arithmetic.

The per-element arithmetic lives in ``bsq_oracle.c`` (plain C, FP64 exact
values, FP32 only where the NVFP4 recipe fixes FP32 steps).  This module
adds the storage layout, written independently of the CUDA side:

* FP4 packing: two E2M1 codes per byte, the even-index element in the low
  nibble.
* Scale layout: scales of a [rows, S] matrix are stored in 512-byte tiles
  covering 128 rows x 4 scale columns; inside a tile the byte of (r, c) sits
  at (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4); tiles are ordered with
  the scale-column tile index fastest; rows are padded to a multiple of 128
  and scale columns to a multiple of 4, padding bytes are zero.  This is the
  tensor-core block-scale operand layout (PTX ISA, tcgen05 block scaling).

Sources for each rule are cited in ``bsq_oracle.c``: the FP8 page
("FP8 Training Infrastructure", sections "O panorama da precisao numerica"
and "Estrategias de escalonamento"), the MoE FP4 page ("Practical FP4
Training for Large-Scale MoE Models on Hopper GPUs", section 2
"Metodologia") and the OCP Microscaling v1.0 format definitions.

Parity pins for every function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

E4M3, E5M2, E2M1, UE4M3 = 0, 1, 2, 3
FMT_IDS = {"e4m3": E4M3, "e5m2": E5M2, "e2m1": E2M1}
BLOCK = {"mxfp8_e4m3": 32, "mxfp8_e5m2": 32, "mxfp4": 32, "nvfp4": 16}
ELEM = {"mxfp8_e4m3": E4M3, "mxfp8_e5m2": E5M2, "mxfp4": E2M1, "nvfp4": E2M1}

_lib = None


def build(force: bool = False) -> str:
    """Compile bsq_oracle.c into liboracle.so (gcc, plain C, no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    subprocess.check_call([
        "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
        "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    c_i64 = ctypes.c_int64
    p = ctypes.c_void_p
    lib.bsqo_decode.restype = ctypes.c_double
    lib.bsqo_decode.argtypes = [ctypes.c_int, ctypes.c_uint]
    lib.bsqo_decode_e8m0.restype = ctypes.c_double
    lib.bsqo_decode_e8m0.argtypes = [ctypes.c_uint]
    lib.bsqo_encode.restype = ctypes.c_uint
    lib.bsqo_encode.argtypes = [ctypes.c_int, ctypes.c_double]
    lib.bsqo_max_finite.restype = ctypes.c_double
    lib.bsqo_max_finite.argtypes = [ctypes.c_int]
    lib.bsqo_mx_block.restype = None
    lib.bsqo_mx_block.argtypes = [ctypes.c_int, p, ctypes.c_int, p, p]
    lib.bsqo_mx_quantize_rows.restype = None
    lib.bsqo_mx_quantize_rows.argtypes = [ctypes.c_int, ctypes.c_int, p, c_i64, c_i64, p, p]
    lib.bsqo_nvfp4_tensor_scale.restype = ctypes.c_float
    lib.bsqo_nvfp4_tensor_scale.argtypes = [p, c_i64]
    lib.bsqo_tensor_amax.restype = ctypes.c_float
    lib.bsqo_tensor_amax.argtypes = [p, c_i64]
    lib.bsqo_nvfp4_delayed_tensor_scale.restype = ctypes.c_float
    lib.bsqo_nvfp4_delayed_tensor_scale.argtypes = [p, c_i64]
    lib.bsqo_nvfp4_quantize_rows.restype = None
    lib.bsqo_nvfp4_quantize_rows.argtypes = [p, c_i64, c_i64, ctypes.c_float, p, p]
    lib.bsqo_mx_dequant_rows.restype = None
    lib.bsqo_mx_dequant_rows.argtypes = [ctypes.c_int, ctypes.c_int, p, p, c_i64, c_i64, p]
    lib.bsqo_nvfp4_dequant_rows.restype = None
    lib.bsqo_nvfp4_dequant_rows.argtypes = [p, p, ctypes.c_float, c_i64, c_i64, p]
    lib.bsqo_mxfp4_to_mxfp8_rows.restype = None
    lib.bsqo_mxfp4_to_mxfp8_rows.argtypes = [p, p, c_i64, c_i64, p, p]
    lib.bsqo_mxfp4_row_to_mxfp8_col.restype = None
    lib.bsqo_mxfp4_row_to_mxfp8_col.argtypes = [p, p, c_i64, c_i64, p, p]
    lib.bsqo_mxfp4_to_fp8_1x128.restype = None
    lib.bsqo_mxfp4_to_fp8_1x128.argtypes = [p, p, c_i64, c_i64, p, p]
    lib.bsqo_gemm_pairs.restype = None
    lib.bsqo_gemm_pairs.argtypes = [p, p, c_i64, p, p, c_i64, p, p]
    lib.bsqo_gemm_full.restype = None
    lib.bsqo_gemm_full.argtypes = [p, p, c_i64, c_i64, c_i64, p, p]
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- codecs
def decode(fmt: int, code: int) -> float:
    """Exact value of one element code (E4M3 / E5M2 / E2M1 / UE4M3)."""
    return _load().bsqo_decode(fmt, int(code))


def decode_e8m0(b: int) -> float:
    return _load().bsqo_decode_e8m0(int(b))


def encode(fmt: int, v: float) -> int:
    """Round-to-nearest-even code of v with saturation (sign kept)."""
    return int(_load().bsqo_encode(fmt, float(v)))


def max_finite(fmt: int) -> float:
    return _load().bsqo_max_finite(fmt)


def decode_table(fmt: int) -> np.ndarray:
    n = 16 if fmt == E2M1 else 256
    return np.array([decode(fmt, c) for c in range(n)], dtype=np.float64)


def mx_block(fmt: int, values) -> tuple[np.ndarray, int]:
    """Quantize one block of exact values; returns (codes, scale byte)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    codes = np.zeros(v.size, dtype=np.uint8)
    scale = np.zeros(1, dtype=np.uint8)
    _load().bsqo_mx_block(fmt, _ptr(v), v.size, _ptr(codes), _ptr(scale))
    return codes, int(scale[0])


# -------------------------------------------------------------- quantize
def mx_quantize_rows(x_bits: np.ndarray, fmt_name: str):
    """Row-wise MX quantize of a BF16 bit-pattern matrix [R, C].

    Returns (codes [R, C] one code per byte, scales [R, C/32] row-major)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, C = x.shape
    blk = BLOCK[fmt_name]
    assert C % blk == 0
    codes = np.empty((R, C), dtype=np.uint8)
    scales = np.empty((R, C // blk), dtype=np.uint8)
    _load().bsqo_mx_quantize_rows(ELEM[fmt_name], blk, _ptr(x), R, C, _ptr(codes), _ptr(scales))
    return codes, scales


def nvfp4_tensor_scale(x_bits: np.ndarray) -> float:
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    return float(np.float32(_load().bsqo_nvfp4_tensor_scale(_ptr(x), x.size)))


def nvfp4_quantize_rows(x_bits: np.ndarray, s_t: float | None = None):
    """Row-wise NVFP4 quantize; returns (codes [R, C], scales [R, C/16], s_t)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, C = x.shape
    assert C % 16 == 0
    if s_t is None:
        s_t = nvfp4_tensor_scale(x)
    codes = np.empty((R, C), dtype=np.uint8)
    scales = np.empty((R, C // 16), dtype=np.uint8)
    _load().bsqo_nvfp4_quantize_rows(_ptr(x), R, C, ctypes.c_float(s_t), _ptr(codes), _ptr(scales))
    return codes, scales, s_t


def tensor_amax(x_bits: np.ndarray) -> float:
    """Largest finite |x| of a BF16 tensor (bit patterns)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    return float(np.float32(_load().bsqo_tensor_amax(_ptr(x), x.size)))


def nvfp4_delayed_tensor_scale(history) -> float:
    """NVFP4 tensor scale under delayed scaling: max(history) / 2688 (FP32),
    1 when the history holds no positive finite value."""
    h = np.ascontiguousarray(history, dtype=np.float32)
    return float(np.float32(_load().bsqo_nvfp4_delayed_tensor_scale(_ptr(h), h.size)))


def nvfp4_delayed_quantize(x_bits: np.ndarray, history, axis: str = "row"):
    """NVFP4 quantize with a delayed tensor scale ("FP8 Training
    Infrastructure": delayed scaling from the amax history of previous
    iterations, length 16, algorithm max, margin 0).

    The tensor scale comes from the history as it stands before this step;
    the blocks are then encoded by the just-in-time NVFP4 steps with that
    scale (values beyond its range saturate); last, this tensor's amax is
    pushed to the front of the history and the oldest entry dropped.
    Returns {"row": (codes, scales), "col": (codes, scales), "s_t": s_t,
    "history": new_history}, with only the requested orientations."""
    h = np.asarray(history, dtype=np.float32)
    s_t = nvfp4_delayed_tensor_scale(h)
    out = {"s_t": s_t}
    if axis in ("row", "both"):
        c, s, _ = nvfp4_quantize_rows(x_bits, s_t)
        out["row"] = (c, s)
    if axis in ("col", "both"):
        c, s, _ = nvfp4_quantize_rows(np.ascontiguousarray(np.asarray(x_bits).T), s_t)
        out["col"] = (c, s)
    out["history"] = np.concatenate([np.float32([tensor_amax(x_bits)]), h[:-1]]).astype(np.float32)
    return out


def quantize_rows(x_bits: np.ndarray, fmt_name: str):
    """Row-wise quantize in any format; returns (codes, scales, s_t or None)."""
    if fmt_name == "nvfp4":
        return nvfp4_quantize_rows(x_bits)
    c, s = mx_quantize_rows(x_bits, fmt_name)
    return c, s, None


def quantize_cols(x_bits: np.ndarray, fmt_name: str):
    """Column-wise quantize = row-wise quantize of the transpose.

    The NVFP4 tensor scale is a whole-tensor amax, so it is the same for
    both orientations."""
    return quantize_rows(np.ascontiguousarray(np.asarray(x_bits).T), fmt_name)


# ---------------------------------------------------------------- layout
def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """[R, C] one E2M1 code per byte -> [R, C/2] bytes, even index low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    R, C = c.shape
    assert C % 2 == 0
    return ((c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)).astype(np.uint8)


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    R, H = p.shape
    out = np.empty((R, 2 * H), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def scale_tile_offset(r: int, c: int, S: int) -> int:
    """Byte offset of scale (r, c) of a [*, S] scale matrix in tiled storage."""
    s_pad = (S + 3) // 4 * 4
    tile = (r // 128) * (s_pad // 4) + (c // 4)
    return tile * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4)


def scales_nbytes(rows: int, S: int) -> int:
    return ((rows + 127) // 128 * 128) * ((S + 3) // 4 * 4)


def swizzle_scales(s: np.ndarray) -> np.ndarray:
    """Row-major [R, S] scales -> tiled byte stream (padding zero)."""
    s = np.asarray(s, dtype=np.uint8)
    R, S = s.shape
    out = np.zeros(scales_nbytes(R, S), dtype=np.uint8)
    r = np.arange(R)[:, None]
    c = np.arange(S)[None, :]
    s_pad = (S + 3) // 4 * 4
    off = ((r // 128) * (s_pad // 4) + (c // 4)) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4)
    out[off.ravel()] = s.ravel()
    return out


def unswizzle_scales(buf: np.ndarray, R: int, S: int) -> np.ndarray:
    buf = np.asarray(buf, dtype=np.uint8).ravel()
    r = np.arange(R)[:, None]
    c = np.arange(S)[None, :]
    s_pad = (S + 3) // 4 * 4
    off = ((r // 128) * (s_pad // 4) + (c // 4)) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4)
    return buf[off]


def grouped_scale_starts(offsets) -> tuple[np.ndarray, int]:
    """Per-expert padded scale layout: expert g's scale rows start at
    P_g = sum over earlier experts of their row counts rounded up to 128, so
    no 128-row scale tile holds two experts.  Returns (P [G], total rows)."""
    o = np.asarray(offsets, dtype=np.int64)
    padded = (np.diff(o) + 127) // 128 * 128
    P = np.concatenate([[0], np.cumsum(padded)[:-1]]).astype(np.int64)
    return P, int(padded.sum())


def swizzle_scales_grouped(s: np.ndarray, offsets, capacity_rows: int | None = None) -> np.ndarray:
    """Row-major [R, S] scales of rows grouped by `offsets` -> the tiled byte
    stream of the [P_total, S] matrix in which data row r of expert g sits at
    scale row P_g + (r - offsets[g]); every other byte is zero.  The buffer
    may be longer (capacity_rows, a multiple of 128)."""
    s = np.asarray(s, dtype=np.uint8)
    R, S = s.shape
    o = np.asarray(offsets, dtype=np.int64)
    P, total = grouped_scale_starts(o)
    rows = total if capacity_rows is None else capacity_rows
    assert rows >= total and rows % 128 == 0
    padded = np.zeros((rows, S), dtype=np.uint8)
    for g in range(len(o) - 1):
        n = o[g + 1] - o[g]
        padded[P[g]:P[g] + n] = s[o[g]:o[g + 1]]
    return swizzle_scales(padded)


def scale_pad_mask(R: int, S: int) -> np.ndarray:
    """Boolean mask over the tiled buffer: True where a byte is padding."""
    m = np.ones(scales_nbytes(R, S), dtype=bool)
    r = np.arange(R)[:, None]
    c = np.arange(S)[None, :]
    s_pad = (S + 3) // 4 * 4
    off = ((r // 128) * (s_pad // 4) + (c // 4)) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4)
    m[off.ravel()] = False
    return m


def storage_codes(codes: np.ndarray, fmt_name: str) -> np.ndarray:
    """Codes in the library's storage form (FP4 packed, FP8 one per byte)."""
    return pack_fp4(codes) if ELEM[fmt_name] == E2M1 else np.asarray(codes, dtype=np.uint8)


# ------------------------------------------------------------- dequantize
def dequant_rows(codes: np.ndarray, scales: np.ndarray, fmt_name: str, s_t: float | None = None):
    """Exact FP64 values of quantized rows (codes unpacked, scales row-major)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R, C = c.shape
    out = np.empty((R, C), dtype=np.float64)
    if fmt_name == "nvfp4":
        _load().bsqo_nvfp4_dequant_rows(_ptr(c), _ptr(s), ctypes.c_float(s_t), R, C, _ptr(out))
    else:
        _load().bsqo_mx_dequant_rows(ELEM[fmt_name], BLOCK[fmt_name], _ptr(c), _ptr(s), R, C, _ptr(out))
    return out


# ----------------------------------------------------------------- repack
def mxfp4_to_mxfp8_rows(codes4: np.ndarray, scales4: np.ndarray):
    """MXFP4 -> MXFP8 E4M3 re-encode (codes unpacked, scales row-major)."""
    c = np.ascontiguousarray(codes4, dtype=np.uint8)
    s = np.ascontiguousarray(scales4, dtype=np.uint8)
    R, C = c.shape
    oc = np.empty((R, C), dtype=np.uint8)
    os_ = np.empty((R, C // 32), dtype=np.uint8)
    _load().bsqo_mxfp4_to_mxfp8_rows(_ptr(c), _ptr(s), R, C, _ptr(oc), _ptr(os_))
    return oc, os_


# ------------------------------------------------------------------- GEMM
def mxfp4_row_to_mxfp8_col(codes4: np.ndarray, scales4: np.ndarray):
    """FP4RowToFP8Col: MXFP8 E4M3 column-wise quantization of the exactly
    dequantized MXFP4 matrix (codes [R, C] unpacked, scales [R, C/32]).
    Returns (codes [C, R], scales [C, R/32]) of the transpose."""
    c4 = np.ascontiguousarray(codes4, dtype=np.uint8)
    s4 = np.ascontiguousarray(scales4, dtype=np.uint8)
    R, C = c4.shape
    assert R % 32 == 0 and C % 32 == 0 and s4.shape == (R, C // 32)
    codes8 = np.empty((C, R), dtype=np.uint8)
    scales8 = np.empty((C, R // 32), dtype=np.uint8)
    _load().bsqo_mxfp4_row_to_mxfp8_col(_ptr(c4), _ptr(s4), R, C, _ptr(codes8), _ptr(scales8))
    return codes8, scales8


def mxfp4_to_fp8_1x128(codes4: np.ndarray, scales4: np.ndarray):
    """MXFP4 -> FP8 E4M3 with 1x128 blocks (the Hopper FP8 block): the block
    scale is the largest of the four 32-block E8M0 scales, each element the
    E4M3 code of its exact value over that scale (codes [R, C] unpacked,
    scales [R, C/32]).  Returns (codes [R, C], scales [R, ceil(C/128)])."""
    c4 = np.ascontiguousarray(codes4, dtype=np.uint8)
    s4 = np.ascontiguousarray(scales4, dtype=np.uint8)
    R, C = c4.shape
    assert C % 32 == 0 and s4.shape == (R, C // 32)
    codes8 = np.empty((R, C), dtype=np.uint8)
    scales8 = np.empty((R, (C + 127) // 128), dtype=np.uint8)
    _load().bsqo_mxfp4_to_fp8_1x128(_ptr(c4), _ptr(s4), R, C, _ptr(codes8), _ptr(scales8))
    return codes8, scales8


def gemm_pairs(A: np.ndarray, B: np.ndarray, ms, ns):
    """ref, mag for C[m, n] = sum_k A[m, k] B[n, k] at the given (m, n)."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    assert A.shape[1] == B.shape[1]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    ref = np.empty(ms.size, dtype=np.float64)
    mag = np.empty(ms.size, dtype=np.float64)
    _load().bsqo_gemm_pairs(_ptr(A), _ptr(B), A.shape[1], _ptr(ms), _ptr(ns), ms.size, _ptr(ref), _ptr(mag))
    return ref, mag


def gemm_full_matmul(A: np.ndarray, B: np.ndarray):
    """ref = A B^T and mag = |A| |B|^T in FP64 with numpy's matrix product
    (the library primitive as the summation step; the exactly dequantized
    products need at most 24 significant bits, so only the FP64 summation
    rounds, far below the 1e-5 bound).  For full-output checks."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    return A @ B.T, np.abs(A) @ np.abs(B).T


def gemm_full(A: np.ndarray, B: np.ndarray):
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    M, K = A.shape
    N = B.shape[0]
    ref = np.empty((M, N), dtype=np.float64)
    mag = np.empty((M, N), dtype=np.float64)
    _load().bsqo_gemm_full(_ptr(A), _ptr(B), M, N, K, _ptr(ref), _ptr(mag))
    return ref, mag
