"""Shared helpers for the parity tests: move seeded inputs to the device and
build the oracle's expected bytes in the library's storage layout."""
import numpy as np

import oracle

BLOCK = oracle.BLOCK


def dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_u8(t) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.uint8)


def dev_u8(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def expected(x_bits: np.ndarray, fmt: str, axis: str):
    """Oracle result in storage layout: {'row': (codes, scales, s_t), 'col': ...}."""
    out = {}
    if axis in ("row", "both"):
        c, s, t = oracle.quantize_rows(x_bits, fmt)
        out["row"] = (oracle.storage_codes(c, fmt), oracle.swizzle_scales(s), t, c, s)
    if axis in ("col", "both"):
        c, s, t = oracle.quantize_cols(x_bits, fmt)
        out["col"] = (oracle.storage_codes(c, fmt), oracle.swizzle_scales(s), t, c, s)
    return out


def assert_qtensor_equal(q, exp, what=""):
    codes, scales, s_t = exp[0], exp[1], exp[2]
    got_c = host_u8(q.codes).reshape(codes.shape)
    got_s = host_u8(q.scales)
    if not np.array_equal(got_c, codes):
        bad = np.argwhere(got_c != codes)
        r, k = bad[0]
        raise AssertionError(f"{what}: {len(bad)} code bytes differ; first at {tuple(bad[0])}: "
                             f"got {got_c[r, k]:#04x} want {codes[r, k]:#04x}")
    if not np.array_equal(got_s, scales):
        bad = np.flatnonzero(got_s != scales)
        raise AssertionError(f"{what}: {len(bad)} scale bytes differ; first at {bad[0]}: "
                             f"got {got_s[bad[0]]:#04x} want {scales[bad[0]]:#04x}")
    if s_t is not None:
        got_t = float(q.tensor_scale.cpu().numpy()[0])
        assert np.float32(got_t) == np.float32(s_t), (what, got_t, s_t)


def codes_at(out, align):
    """Give out a code buffer whose address is `align` (16 or 32) modulo 32;
    its code and scale bytes start as 0xAB."""
    import torch
    if align == 16:
        buf = torch.empty(out.codes.numel() + 16, dtype=torch.uint8, device=out.codes.device)
        out.codes = buf[16:]
        assert out.codes.data_ptr() % 32 == 16
    out.codes.fill_(0xAB)
    out.scales.fill_(0xAB)
    return out


def upload_q(bsq, fmt: str, codes_unpacked: np.ndarray, scales_rowmajor: np.ndarray, s_t=None):
    """Oracle-made quantized tensor -> device QTensor (storage layout)."""
    import torch
    R, C = codes_unpacked.shape
    q = bsq.empty(fmt, R, C)
    q.codes.copy_(dev_u8(oracle.storage_codes(codes_unpacked, fmt).ravel()))
    q.scales.copy_(dev_u8(oracle.swizzle_scales(scales_rowmajor)))
    if s_t is not None:
        q.tensor_scale.copy_(torch.tensor([s_t], dtype=torch.float32))
    return q


def round_to_bf16(d: np.ndarray) -> np.ndarray:
    """Exact doubles -> nearest-even BF16 bit patterns (normal range)."""
    d = np.asarray(d, dtype=np.float64)
    m, e = np.frexp(d)
    r = np.ldexp(np.rint(m * 256.0), e - 8)
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def gemm_tol_ok(C: np.ndarray, ref: np.ndarray, mag: np.ndarray, bf16: bool):
    """|C - ref| <= 1e-5 * sum|a*b| (+ BF16 output rounding, half an ulp)."""
    tol = 1e-5 * mag
    if bf16:
        tol = tol * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(ref)
    err = np.abs(C.astype(np.float64) - ref)
    return err <= tol, err, tol


POISON = 0xAB


def poisoned_qtensor(bsq, fmt: str, rows: int, cols: int):
    """An output QTensor whose code and scale bytes are all 0xAB (and whose
    NVFP4 tensor scale is NaN), so that any byte a kernel fails to write
    differs from the expected one."""
    import torch
    q = bsq.empty(fmt, rows, cols)
    q.codes.fill_(POISON)
    q.scales.fill_(POISON)
    if q.tensor_scale is not None:
        q.tensor_scale.fill_(float("nan"))
    return q


def guarded(shape, dtype, guard_bytes: int = 4096):
    """An output tensor of `shape` inside a larger 0xAB-filled allocation
    with guard bands of `guard_bytes` on both sides; returns (tensor, check)
    where check() asserts that the guard bands are untouched."""
    import torch
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((guard_bytes + n + guard_bytes,), POISON, dtype=torch.uint8, device="cuda")
    t = buf[guard_bytes:guard_bytes + n].view(dtype).view(*shape)

    def check():
        lo = buf[:guard_bytes].cpu().numpy()
        hi = buf[guard_bytes + n:].cpu().numpy()
        assert (lo == POISON).all() and (hi == POISON).all(), "a kernel wrote outside its output"
    return t, check


# ---- library calls with poisoned outputs (every output byte starts as 0xAB;
# dense and grouped GEMM outputs also sit between guard bands)
def qz(bsq, x_dev, fmt: str, axis: str = "row"):
    R, C = x_dev.shape
    row = poisoned_qtensor(bsq, fmt, R, C) if axis in ("row", "both") else None
    col = poisoned_qtensor(bsq, fmt, C, R) if axis in ("col", "both") else None
    bsq.quantize_into(x_dev, fmt, axis, row, col)
    return row, col


def qz_delayed(bsq, x_dev, history, axis: str = "row"):
    R, C = x_dev.shape
    row = poisoned_qtensor(bsq, "nvfp4", R, C) if axis in ("row", "both") else None
    col = poisoned_qtensor(bsq, "nvfp4", C, R) if axis in ("col", "both") else None
    bsq.quantize_nvfp4_delayed_into(x_dev, axis, row, col, history)
    return row, col


def deq(bsq, q, dtype):
    out, check = guarded((q.rows, q.cols), dtype)
    bsq.dequantize_into(q, out)
    check()
    return out


def gemm_g(bsq, A, B, dtype):
    C, check = guarded((A.rows, B.rows), dtype)
    bsq.gemm_into(A, B, C)
    check()
    return C


def grouped_g(bsq, A, offsets_dev, groups, dtype, padded_scales=False):
    C, check = guarded((A.rows, groups[0].rows), dtype)
    bsq.grouped_gemm_into(A, offsets_dev, groups, C, padded_scales=padded_scales)
    check()
    return C


def repack(bsq, q4):
    out = poisoned_qtensor(bsq, "mxfp8_e4m3", q4.rows, q4.cols)
    bsq.mxfp4_to_mxfp8_into(q4, out)
    return out


def repack_grouped(bsq, q4, offsets_dev, groups: int):
    out = poisoned_qtensor(bsq, "mxfp8_e4m3", q4.rows, q4.cols)
    out.scales = bsq.empty_grouped("mxfp8_e4m3", q4.rows, q4.cols, groups).scales.fill_(POISON)
    bsq.mxfp4_to_mxfp8_grouped_into(q4, out, offsets_dev, groups)
    return out


def repack_col(bsq, q4):
    out = poisoned_qtensor(bsq, "mxfp8_e4m3", q4.cols, q4.rows)
    bsq.mxfp4_to_mxfp8_col_into(q4, out)
    return out


def repack_1x128(bsq, q4):
    import torch
    codes = torch.full((q4.rows, q4.cols), POISON, dtype=torch.uint8, device="cuda")
    scales = torch.full((q4.rows, (q4.cols + 127) // 128), POISON, dtype=torch.uint8, device="cuda")
    bsq.mxfp4_to_fp8_1x128_into(q4, codes, scales)
    return codes, scales
