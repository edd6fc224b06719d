"""GPU-vs-oracle parity on small and ragged shapes, through the C ABI.

Codes, scales and repacked bytes must match the oracle bit for bit; GEMM
outputs must satisfy |C - ref| <= 1e-5 * sum_k |a_k b_k| against the
oracle's FP64 sum of exactly dequantized products (plus half a BF16 ulp for
BF16 output)."""
import numpy as np
import pytest

import oracle
from block_scaled_precision_03_gb300 import inputs
from _util import (expected, assert_qtensor_equal, dev_bf16, host_u8, dev_u8, upload_q, round_to_bf16, codes_at, gemm_tol_ok, qz, qz_delayed, gemm_g, deq, grouped_g, repack_grouped, repack_col, repack_1x128, repack, poisoned_qtensor, guarded)

pytestmark = pytest.mark.gpu

FMTS = ["mxfp8_e4m3", "mxfp8_e5m2", "mxfp4", "nvfp4"]


@pytest.fixture(scope="module")
def bsq():
    import block_scaled_precision_03_gb300 as b
    b.lib()
    return b


def _gen(shape, seed, kind):
    if kind == "outlier":
        return inputs.outlier_activations_bf16(shape, seed)
    if kind == "grad":
        return inputs.loguniform_grad_bf16(shape, seed)
    return inputs.normal_bf16(shape, seed, std=0.02 if kind == "weight" else 1.0)


# ------------------------------------------------------------------ quantize
ROW_SHAPES = [(256, 256), (130, 96), (7, 32), (1, 4096), (384, 1056), (129, 160)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", ROW_SHAPES)
@pytest.mark.parametrize("kind", ["outlier", "grad", "weight"])
def test_quantize_rows(bsq, fmt, shape, kind):
    x = _gen(shape, 11, kind)
    row, _ = qz(bsq, dev_bf16(x), fmt, "row")
    assert_qtensor_equal(row, expected(x, fmt, "row")["row"], f"{fmt} row {shape}")


COL_SHAPES = [(256, 256), (96, 200), (32, 8), (4096, 16), (1056, 384), (160, 136), (128, 96), (96, 1056)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", COL_SHAPES)
@pytest.mark.parametrize("axis", ["col", "both"])
def test_quantize_cols_and_both(bsq, fmt, shape, axis):
    R, C = shape
    if axis == "both" and C % oracle.BLOCK[fmt]:
        pytest.skip("row-wise blocks need cols % block == 0")
    x = _gen(shape, 5, "grad" if fmt == "mxfp8_e5m2" else "outlier")
    row, col = qz(bsq, dev_bf16(x), fmt, axis)
    exp = expected(x, fmt, axis)
    assert_qtensor_equal(col, exp["col"], f"{fmt} col {shape}")
    if axis == "both":
        assert_qtensor_equal(row, exp["row"], f"{fmt} both/row {shape}")


def _all_bf16_patterns(order_seed=None):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if order_seed is not None:
        bits = np.random.default_rng(order_seed).permutation(bits)
    return bits.reshape(2048, 32)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("order", [None, 1, 2])
def test_quantize_every_bf16_pattern(bsq, fmt, order):
    """All 65536 BF16 bit patterns (NaN, Inf, subnormals, zeros included) in
    natural and shuffled block groupings."""
    x = _all_bf16_patterns(order)
    if fmt == "nvfp4":
        # the tensor amax ignores non-finite values; keep them in blocks
        pass
    row, _ = qz(bsq, dev_bf16(x), fmt, "row")
    assert_qtensor_equal(row, expected(x, fmt, "row")["row"], f"{fmt} all-bf16 order={order}")


@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_every_bf16_pattern_scaled_blocks(bsq, fmt):
    """Each block = 31 patterns + an anchor 2^k above them: every finite BF16
    value is encoded at many block scales."""
    rng = np.random.default_rng(3)
    fin = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    fin = fin[(fin & 0x7F80) != 0x7F80]
    blocks = []
    for shift in (0, 1, 3, 7):
        v = rng.permutation(fin)
        n = len(v) // 31 * 31
        body = v[:n].reshape(-1, 31)
        mags = (body & 0x7FFF).max(axis=1)
        anchor = np.minimum(mags.astype(np.int64) + (shift << 7), 0x7F7F).astype(np.uint16)
        blocks.append(np.concatenate([body, anchor[:, None]], axis=1))
    x = np.ascontiguousarray(np.concatenate(blocks)[:, :32])
    if fmt == "nvfp4":
        x = np.ascontiguousarray(x.reshape(-1, 16))
    row, _ = qz(bsq, dev_bf16(x), fmt, "row")
    assert_qtensor_equal(row, expected(x, fmt, "row")["row"], f"{fmt} anchored")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("axis", ["col", "both"])
@pytest.mark.parametrize("order", [None, 1])
def test_quantize_every_bf16_pattern_columns(bsq, fmt, axis, order):
    """All 65536 BF16 bit patterns through the column-wise and both-ways
    kernel: the 32-row (NVFP4: 16-row) column blocks hold every NaN, Inf,
    subnormal and signed zero, and the row blocks of `both` every pattern
    again in another grouping."""
    x = _all_bf16_patterns(order)
    row, col = qz(bsq, dev_bf16(x), fmt, axis)
    exp = expected(x, fmt, axis)
    assert_qtensor_equal(col, exp["col"], f"{fmt} {axis} col all-bf16 order={order}")
    if axis == "both":
        assert_qtensor_equal(row, exp["row"], f"{fmt} both/row all-bf16 order={order}")


@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_every_bf16_pattern_scaled_columns(bsq, fmt):
    """The anchored blocks of the row test, transposed: each column block
    holds 31 (NVFP4: 15) patterns and an anchor 2^k above them."""
    rng = np.random.default_rng(4)
    fin = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    fin = fin[(fin & 0x7F80) != 0x7F80]
    blk = 16 if fmt == "nvfp4" else 32
    blocks = []
    for shift in (0, 1, 3, 7):
        v = rng.permutation(fin)
        n = len(v) // (blk - 1) * (blk - 1)
        body = v[:n].reshape(-1, blk - 1)
        mags = (body & 0x7FFF).max(axis=1)
        anchor = np.minimum(mags.astype(np.int64) + (shift << 7), 0x7F7F).astype(np.uint16)
        blocks.append(np.concatenate([body, anchor[:, None]], axis=1))
    b = np.concatenate(blocks)
    b = b[: len(b) // 8 * 8]                       # whole 8-column chunks
    x = np.ascontiguousarray(b.T)                  # [blk, n]: one block per column
    _, col = qz(bsq, dev_bf16(x), fmt, "col")
    assert_qtensor_equal(col, expected(x, fmt, "col")["col"], f"{fmt} anchored columns")


def test_quantize_zero_and_nonfinite_blocks(bsq):
    x = np.zeros((4, 64), dtype=np.uint16)
    x[1, 3] = 0x7FC0          # NaN
    x[2, 40] = 0xFF80         # -Inf
    x[3, :] = 0x8000          # -0
    x[3, 33] = 0x3F80
    for fmt in FMTS:
        row, col = qz(bsq, dev_bf16(x), fmt, "row")
        assert_qtensor_equal(row, expected(x, fmt, "row")["row"], f"{fmt} special")
    # the same blocks down the columns (32 rows: one block per column)
    xt = np.ascontiguousarray(np.tile(x.T, (1, 8)))          # [64, 32]
    for fmt in FMTS:
        row, col = qz(bsq, dev_bf16(xt), fmt, "both")
        exp = expected(xt, fmt, "both")
        assert_qtensor_equal(col, exp["col"], f"{fmt} special columns")
        assert_qtensor_equal(row, exp["row"], f"{fmt} special both/row")


def test_nvfp4_tensor_scale_shared(bsq):
    x = inputs.outlier_activations_bf16((128, 256), 9)
    row, col = qz(bsq, dev_bf16(x), "nvfp4", "both")
    st = oracle.nvfp4_tensor_scale(x)
    assert float(row.tensor_scale.cpu()[0]) == st == float(col.tensor_scale.cpu()[0])


# -------------------------------------------------------------------- repack
def _random_mxfp4(R, C, seed, scale_lo=0, scale_hi=256):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (R, C)).astype(np.uint8)
    # some all-zero and single-magnitude blocks
    codes[0, :32] = 0
    if R > 1:
        codes[1, :32] = rng.choice([0, 8, 1, 9], 32)
    scales = rng.integers(scale_lo, scale_hi, (R, C // 32)).astype(np.uint8)
    return codes, scales


@pytest.mark.parametrize("shape", [(64, 256), (130, 96), (1, 32), (300, 7168)])
@pytest.mark.parametrize("align", [32, 16])
def test_repack_bitexact(bsq, shape, align):
    """Both store paths: 32-byte stores (aligned output) and 16-byte halves."""
    R, C = shape
    codes, scales = _random_mxfp4(R, C, R + C)
    scales.ravel()[:12] = [0, 1, 2, 5, 6, 7, 8, 9, 250, 253, 254, 255][:scales.size]
    q = upload_q(bsq, "mxfp4", codes, scales)
    out = codes_at(bsq.empty("mxfp8_e4m3", R, C), align)
    bsq.mxfp4_to_mxfp8_into(q, out)
    c8, s8 = oracle.mxfp4_to_mxfp8_rows(codes, scales)
    assert_qtensor_equal(out, (c8, oracle.swizzle_scales(s8), None), f"repack {shape}")


def test_repack_every_nibble_pair_every_scale(bsq):
    rows = []
    for a in range(16):
        for b in range(16):
            blk = np.zeros(32, dtype=np.uint8)
            blk[0], blk[1] = a, b
            blk[2:] = (np.arange(30) * 5 + b) % 16
            rows.append(blk)
    base = np.array(rows, dtype=np.uint8)
    codes = np.tile(base, (1, 8))                         # 256 rows x 256
    scales = np.arange(256 * 8, dtype=np.uint32).reshape(256, 8).astype(np.uint8)
    q = upload_q(bsq, "mxfp4", codes, scales)
    out = repack(bsq, q)
    c8, s8 = oracle.mxfp4_to_mxfp8_rows(codes, scales)
    assert_qtensor_equal(out, (c8, oracle.swizzle_scales(s8), None), "repack exhaustive")


# ------------------------------------------------------------------- dequant
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_dequantize_exact(bsq, fmt, out):
    import torch
    x = inputs.outlier_activations_bf16((130, 256), 21)
    c, s, t = oracle.quantize_rows(x, fmt)
    q = upload_q(bsq, fmt, c, s, t)
    ref = oracle.dequant_rows(c, s, fmt, t)
    got = deq(bsq, q, torch.float32 if out == "f32" else torch.bfloat16)
    if out == "f32":
        np.testing.assert_array_equal(got.cpu().numpy(), ref.astype(np.float32))
    else:
        g = got.view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(g, round_to_bf16(ref))


# ---------------------------------------------------------------------- GEMM
def _q_oracle(x, fmt):
    c, s, t = oracle.quantize_rows(x, fmt)
    return c, s, t


def _check_gemm(bsq, xa, fa, xb, fb, dtype_name, full=True):
    import torch
    ca, sa, ta = _q_oracle(xa, fa)
    cb, sb, tb = _q_oracle(xb, fb)
    A = upload_q(bsq, fa, ca, sa, ta)
    B = upload_q(bsq, fb, cb, sb, tb)
    dt = torch.float32 if dtype_name == "f32" else torch.bfloat16
    C = gemm_g(bsq, A, B, dt).float().cpu().numpy()
    Ad = oracle.dequant_rows(ca, sa, fa, ta)
    Bd = oracle.dequant_rows(cb, sb, fb, tb)
    ref, mag = oracle.gemm_full(Ad, Bd)
    ok, err, tol = gemm_tol_ok(C, ref, mag, dtype_name == "bf16")
    if not ok.all():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{(~ok).sum()} of {ok.size} outside bound; worst {i}: got {C[i]} ref {ref[i]} "
                             f"mag {mag[i]} err {err[i]} tol {tol[i]}")
    return C, ref


def test_gemm_tiny_mxfp8_linear(bsq):
    """A 256x256 @ B 256x256^T, E4M3, FP32 out: every element."""
    d = inputs.tiny_linear()
    _check_gemm(bsq, d["A"], "mxfp8_e4m3", d["B"], "mxfp8_e4m3", "f32")


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (1, 1, 32), (200, 300, 96), (257, 513, 4160), (64, 640, 1024)])
@pytest.mark.parametrize("fa,fb", [("mxfp8_e4m3", "mxfp8_e4m3"), ("mxfp8_e5m2", "mxfp8_e4m3"),
                                   ("mxfp8_e4m3", "mxfp8_e5m2")])
def test_gemm_mxfp8_shapes(bsq, M, N, K, fa, fb):
    xa = inputs.loguniform_grad_bf16((M, K), 1) if fa == "mxfp8_e5m2" else inputs.outlier_activations_bf16((M, K), 1)
    xb = inputs.normal_bf16((N, K), 2, std=0.02)
    _check_gemm(bsq, xa, fa, xb, fb, "f32")


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 300, 96), (130, 260, 4128), (33, 512, 640)])
def test_gemm_nvfp4_shapes(bsq, M, N, K):
    xa = inputs.normal_bf16((M, K), 3)
    xb = inputs.normal_bf16((N, K), 4, std=0.02)
    _check_gemm(bsq, xa, "nvfp4", xb, "nvfp4", "f32")


@pytest.mark.parametrize("fmt", ["mxfp8_e4m3", "nvfp4"])
def test_gemm_bf16_output(bsq, fmt):
    xa = inputs.outlier_activations_bf16((300, 512), 5)
    xb = inputs.normal_bf16((520, 512), 6, std=0.02)
    _check_gemm(bsq, xa, fmt, xb, fmt, "bf16")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype_name", ["f32", "bf16"])
def test_gemm_nonfinite_blocks_propagate(bsq, fmt, dtype_name):
    """A block holding NaN or Inf quantizes to the NaN scale (E8M0 0xFF, or
    UE4M3 0x7F for NVFP4), whose value is NaN; every output of that row of A
    (or column of C for a row of B) must then be NaN, as in the oracle's FP64
    product, and no other output may be NaN or leave the bound.  Rows on
    both M tiles and a ragged N tail."""
    import torch
    M, N, K = 200, 300, 512
    xa = inputs.normal_bf16((M, K), 7)
    xb = inputs.normal_bf16((N, K), 8, std=0.02)
    xa[5, 40] = 0x7FC0      # NaN
    xa[9, 100] = 0x7F80     # +Inf
    xa[130, 511] = 0xFF80   # -Inf, last block of the row
    xb[17, 0] = 0xFFC1      # a NaN with a payload and the sign set
    xb[299, 256] = 0x7F80
    ca, sa, ta = _q_oracle(xa, fmt)
    cb, sb, tb = _q_oracle(xb, fmt)
    A = upload_q(bsq, fmt, ca, sa, ta)
    B = upload_q(bsq, fmt, cb, sb, tb)
    dt = torch.float32 if dtype_name == "f32" else torch.bfloat16
    C = gemm_g(bsq, A, B, dt).float().cpu().numpy()
    ref, mag = oracle.gemm_full(oracle.dequant_rows(ca, sa, fmt, ta), oracle.dequant_rows(cb, sb, fmt, tb))
    nan_ref = np.isnan(ref)
    rows, cols = np.array([5, 9, 130]), np.array([17, 299])
    assert nan_ref[rows].all() and nan_ref[:, cols].all()
    assert nan_ref.sum() == len(rows) * N + len(cols) * M - len(rows) * len(cols)
    np.testing.assert_array_equal(np.isnan(C), nan_ref)
    ok, _, _ = gemm_tol_ok(C[~nan_ref], ref[~nan_ref], mag[~nan_ref], dtype_name == "bf16")
    assert ok.all(), f"{(~ok).sum()} finite outputs outside the bound"


def test_gemm_single_scale_probe(bsq):
    """One non-unit scale per 128x4 tile position: checks that every scale
    byte reaches the MMA for the row / block it belongs to."""
    import torch
    M, N, K = 128, 256, 256
    ca = np.full((M, K), oracle.encode(oracle.E4M3, 1.0), np.uint8)
    cb = np.full((N, K), oracle.encode(oracle.E4M3, 1.0), np.uint8)
    rng = np.random.default_rng(0)
    sa = (127 + rng.integers(-3, 4, (M, K // 32))).astype(np.uint8)
    sb = (127 + rng.integers(-3, 4, (N, K // 32))).astype(np.uint8)
    A = upload_q(bsq, "mxfp8_e4m3", ca, sa)
    B = upload_q(bsq, "mxfp8_e4m3", cb, sb)
    C = gemm_g(bsq, A, B, torch.float32).cpu().numpy()
    ref = 32.0 * (np.exp2(sa.astype(np.float64) - 127) @ np.exp2(sb.astype(np.float64) - 127).T)
    np.testing.assert_array_equal(C, ref.astype(np.float32))


def test_grouped_gemm_small(bsq):
    import torch
    counts = np.array([100, 0, 300, 1, 129, 70], dtype=np.int64)
    G, N, K = len(counts), 256, 384
    off = inputs.group_offsets(counts)
    xa = inputs.normal_bf16((int(off[-1]), K), 7)
    xw = inputs.normal_bf16((G * N, K), 8, std=0.02)
    ca, sa, _ = _q_oracle(xa, "mxfp8_e4m3")
    cw, sw, _ = _q_oracle(xw, "mxfp8_e4m3")
    A = upload_q(bsq, "mxfp8_e4m3", ca, sa)
    W = upload_q(bsq, "mxfp8_e4m3", cw, sw)
    offd = torch.from_numpy(off).cuda()
    C = grouped_g(bsq, A, offd, bsq.group_views(W, G), torch.float32).cpu().numpy()
    Ad = oracle.dequant_rows(ca, sa, "mxfp8_e4m3")
    Wd = oracle.dequant_rows(cw, sw, "mxfp8_e4m3")
    for g in range(G):
        lo, hi = off[g], off[g + 1]
        if hi == lo:
            continue
        ref, mag = oracle.gemm_full(Ad[lo:hi], Wd[g * N:(g + 1) * N])
        ok, err, tol = gemm_tol_ok(C[lo:hi], ref, mag, False)
        assert ok.all(), (g, (~ok).sum())


GROUPED_CASES = {
    # expert sizes with odd band counts, an expert ending mid-band, empty experts
    "ragged": (np.array([700, 0, 129, 1, 383, 256, 1000, 0, 31], dtype=np.int64), 384, 4160),
    # every expert starts and ends on a 128-row boundary
    "aligned": (np.array([256, 128, 512, 0, 384], dtype=np.int64), 512, 256),
    # one expert holding every row
    "single": (np.array([1111], dtype=np.int64), 256, 96),
    # the most experts a call takes: tiny and empty experts (the first three
    # and the last two empty) and one large one; the device builds its expert
    # table in passes of 32 boundaries, carried from pass to pass
    "many": (np.concatenate([[0, 0, 0], np.random.default_rng(256).integers(0, 40, 250), [300], [0, 0]]).astype(np.int64),
             128, 96),
}


_GROUPED_CACHE = {}


def _grouped_case_oracle(case):
    """Oracle codes, scales and exactly dequantized operands of a case (cached
    across the kernel-path and output-type parametrizations)."""
    if case not in _GROUPED_CACHE:
        counts, N, K = GROUPED_CASES[case]
        off = inputs.group_offsets(counts)
        xa = inputs.normal_bf16((int(off[-1]), K), 21)
        xw = inputs.normal_bf16((len(counts) * N, K), 22, std=0.02)
        ca, sa, _ = _q_oracle(xa, "mxfp8_e4m3")
        cw, sw, _ = _q_oracle(xw, "mxfp8_e4m3")
        _GROUPED_CACHE[case] = (off, ca, sa, cw, sw, oracle.dequant_rows(ca, sa, "mxfp8_e4m3"),
                                oracle.dequant_rows(cw, sw, "mxfp8_e4m3"))
    return _GROUPED_CACHE[case]


@pytest.mark.parametrize("case", sorted(GROUPED_CASES))
@pytest.mark.parametrize("path", ["pair", "single_cta"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_grouped_gemm_cases(bsq, monkeypatch, case, path, out):
    """Grouped GEMM on both kernels against the oracle, inside a guarded
    output buffer: rows before and after C keep their sentinel."""
    import torch
    monkeypatch.setenv("BSQ_GEMM_1CTA" if path == "single_cta" else "BSQ_GEMM_GROUPED_PAIR", "1")
    counts, N, K = GROUPED_CASES[case]
    G = len(counts)
    off, ca, sa, cw, sw, Ad, Wd = _grouped_case_oracle(case)
    M = int(off[-1])
    A = upload_q(bsq, "mxfp8_e4m3", ca, sa)
    W = upload_q(bsq, "mxfp8_e4m3", cw, sw)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    guard = 64
    buf = torch.full((M + 2 * guard, N), -7.0, dtype=dt, device="cuda")
    C = buf[guard:guard + M]
    bsq.grouped_gemm_into(A, torch.from_numpy(off).cuda(), bsq.group_views(W, G), C)
    bsq.sync_status()
    host = buf.float().cpu().numpy()
    assert (host[:guard] == -7.0).all() and (host[guard + M:] == -7.0).all(), "write outside C"
    Ch = host[guard:guard + M]
    for g in range(G):
        lo, hi = off[g], off[g + 1]
        if hi == lo:
            continue
        ref, mag = oracle.gemm_full(Ad[lo:hi], Wd[g * N:(g + 1) * N])
        ok, err, tol = gemm_tol_ok(Ch[lo:hi], ref, mag, out == "bf16")
        assert ok.all(), (case, path, g, int((~ok).sum()))


def test_grouped_gemm_scattered_scales(bsq):
    """Experts whose scale buffers are separate allocations (not evenly
    spaced) take the single-CTA kernel; results match the oracle."""
    import torch
    counts = np.array([300, 129, 0, 500], dtype=np.int64)
    G, N, K = len(counts), 256, 512
    off = inputs.group_offsets(counts)
    xa = inputs.normal_bf16((int(off[-1]), K), 31)
    xw = inputs.normal_bf16((G * N, K), 32, std=0.02)
    ca, sa, _ = _q_oracle(xa, "mxfp8_e4m3")
    cw, sw, _ = _q_oracle(xw, "mxfp8_e4m3")
    A = upload_q(bsq, "mxfp8_e4m3", ca, sa)
    W = upload_q(bsq, "mxfp8_e4m3", cw, sw)
    views = bsq.group_views(W, G)
    # same codes; each expert's scales copied to its own allocation, in reverse order
    own = [v.scales.clone() for v in views[::-1]][::-1]
    scattered = [bsq.QTensor(v.fmt, v.rows, v.cols, v.codes, sc, v.tensor_scale) for v, sc in zip(views, own)]
    C = grouped_g(bsq, A, torch.from_numpy(off).cuda(), scattered, torch.float32).cpu().numpy()
    Ad = oracle.dequant_rows(ca, sa, "mxfp8_e4m3")
    Wd = oracle.dequant_rows(cw, sw, "mxfp8_e4m3")
    for g in range(G):
        lo, hi = off[g], off[g + 1]
        if hi == lo:
            continue
        ref, mag = oracle.gemm_full(Ad[lo:hi], Wd[g * N:(g + 1) * N])
        ok, err, tol = gemm_tol_ok(C[lo:hi], ref, mag, False)
        assert ok.all(), (g, int((~ok).sum()))


# ----------------------------------------------------------------- failures
def test_timeout_probe_reports_status(bsq):
    bsq.sync_status()
    bsq.debug_timeout_probe(2_000_000)          # 2 ms limit, nothing ever arrives
    with pytest.raises(bsq.BsqError) as ei:
        bsq.sync_status()
    assert ei.value.status == 5
    bsq.sync_status()                           # cleared; context still usable


@pytest.mark.parametrize("fmt,kernel", [("mxfp8_e4m3", 0), ("nvfp4", 0), ("mxfp4", 0), ("mxfp8_e4m3", 1),
                                        ("nvfp4", 1)])
@pytest.mark.parametrize("limit_ns", [2_000, 10_000])
def test_gemm_wait_limit_runs_out_then_recovers(bsq, fmt, kernel, limit_ns):
    """A GEMM whose waits are limited to a few microseconds gives up part-way
    (stage loads, scale copies and MMAs in flight), reports BSQ_ERR_TIMEOUT
    and leaves the context usable: the next GEMM on the same buffers is
    exact.  The waits run out; nothing faults."""
    import torch
    # a long K: one output tile takes tens of microseconds, far beyond the limit
    M, N, K = 512, 512, 32768
    x = inputs.normal_bf16((M, K), 31)
    w = inputs.normal_bf16((N, K), 32, std=0.02)
    ca, sa, ta = oracle.quantize_rows(x, fmt)
    cb, sb, tb = oracle.quantize_rows(w, fmt)
    A = upload_q(bsq, fmt, ca, sa, ta)
    B = upload_q(bsq, fmt, cb, sb, tb)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    bsq.sync_status()
    bsq.debug_gemm_timeout_into(A, B, C, limit_ns, kernel)
    with pytest.raises(bsq.BsqError) as ei:
        bsq.sync_status()
    assert ei.value.status == 5
    bsq.sync_status()                            # taken and cleared
    C.fill_(float("nan"))
    if kernel == 1:
        bsq.debug_gemm_timeout_into(A, B, C, 4_000_000_000, 1)
    else:
        bsq.gemm_into(A, B, C)
    bsq.sync_status()
    rows = np.arange(0, M, 7)
    Csub = C[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref, mag = oracle.gemm_full(oracle.dequant_rows(ca[rows], sa[rows], fmt, ta), oracle.dequant_rows(cb, sb, fmt, tb))
    ok, err, tol = gemm_tol_ok(Csub, ref, mag, False)
    assert ok.all(), f"{(~ok).sum()} outputs outside the bound after the timed-out GEMM"


@pytest.mark.parametrize("fmt", ["mxfp8_e4m3", "mxfp8_e5m2", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("src_off,codes_off", [(16, 0), (0, 16), (16, 16)])
def test_row_quantize_16_byte_aligned_buffers(bsq, fmt, src_off, codes_off):
    # the row kernels read and write 32 bytes per instruction when both
    # buffers are 32-byte aligned; 16-byte aligned buffers take the other path
    import torch
    R, C = 96, 1056
    x = inputs.outlier_activations_bf16((R, C), 71)
    buf = torch.empty(R * C + 64, dtype=torch.bfloat16, device="cuda")
    base = (-buf.data_ptr() // 2) % 16                      # first element on a 32-byte boundary
    xd = buf[base + src_off // 2:base + src_off // 2 + R * C].view(R, C)
    xd.copy_(dev_bf16(x))
    assert xd.data_ptr() % 32 == src_off
    out = poisoned_qtensor(bsq, fmt, R, C)
    if codes_off:
        cb = torch.full((out.codes.numel() + 64,), 0xAB, dtype=torch.uint8, device="cuda")
        cbase = (-cb.data_ptr()) % 32
        out.codes = cb[cbase + codes_off:cbase + codes_off + out.codes.numel()]
        assert out.codes.data_ptr() % 32 == codes_off
    bsq.quantize_into(xd, fmt, "row", out, None)
    assert_qtensor_equal(out, expected(x, fmt, "row")["row"], f"{fmt} src+{src_off} codes+{codes_off}")


def test_quantize_rejects_unaligned_cols(bsq):
    x = inputs.normal_bf16((96, 130), 1)
    with pytest.raises(bsq.BsqError) as ei:
        qz(bsq, dev_bf16(x), "mxfp8_e4m3", "col")
    assert ei.value.status == 3


def test_gemm_rejects_bad_args(bsq):
    import torch
    A = bsq.empty("mxfp8_e4m3", 128, 256)
    B = bsq.empty("mxfp8_e4m3", 128, 512)
    with pytest.raises(bsq.BsqError):
        bsq.gemm(A, B)
    Bn = bsq.empty("nvfp4", 128, 256)
    with pytest.raises(bsq.BsqError) as ei:
        bsq.gemm(A, Bn)
    assert ei.value.status == 2


@pytest.mark.parametrize("M,N,K,fmt", [(300, 520, 384, "mxfp8_e4m3"), (256, 256, 4096, "mxfp8_e5m2"),
                                       (130, 260, 640, "nvfp4"), (513, 257, 1056, "mxfp8_e4m3")])
def test_gemm_single_cta_tile_path(bsq, M, N, K, fmt, monkeypatch):
    """The dense GEMM normally runs on CTA pairs (256 x 256 tiles); the
    single-CTA 128 x 256 kernel (the grouped GEMM's) must agree as well."""
    monkeypatch.setenv("BSQ_GEMM_1CTA", "1")
    xa = inputs.loguniform_grad_bf16((M, K), 3) if fmt == "mxfp8_e5m2" else inputs.outlier_activations_bf16((M, K), 3)
    xb = inputs.normal_bf16((N, K), 4, std=0.02)
    fb = "mxfp8_e4m3" if fmt == "mxfp8_e5m2" else fmt
    _check_gemm(bsq, xa, fmt, xb, fb, "f32")


@pytest.mark.parametrize("kernel", ["pair", "1cta"])
@pytest.mark.parametrize("dtype_name", ["f32", "bf16"])
def test_gemm_nvfp4_tiny_tensor_scales(bsq, kernel, dtype_name, monkeypatch):
    """NVFP4 operands whose tensor amax is about 2^-58: each tensor scale
    amax / 2688 is a normal FP32 number, but their product is an FP32
    subnormal with about eleven significant bits, so an epilogue that formed it
    would leave the bound; applied one after the other they keep the
    outputs (about 2^-115, normal) within it."""
    if kernel == "1cta":
        monkeypatch.setenv("BSQ_GEMM_1CTA", "1")
    M, N, K = 300, 260, 512
    xa = inputs.normal_bf16((M, K), 11, std=2.0 ** -60)
    xb = inputs.normal_bf16((N, K), 12, std=2.0 ** -60)
    ta = oracle.quantize_rows(xa, "nvfp4")[2]
    tb = oracle.quantize_rows(xb, "nvfp4")[2]
    assert ta >= 2.0 ** -126 and tb >= 2.0 ** -126 and float(ta) * float(tb) < 2.0 ** -126
    C, ref = _check_gemm(bsq, xa, "nvfp4", xb, "nvfp4", dtype_name)
    assert np.abs(ref).max() > 2.0 ** -120 and np.isfinite(C).all()


def test_gemm_pair_tile_tails(bsq):
    """Tails of the 256 x 256 pair tile: the odd CTA's rows fully past M,
    the second B half past N, and a K tail inside the last stage."""
    for M, N, K in [(129, 129, 160), (100, 384, 4128), (384, 100, 96)]:
        xa = inputs.outlier_activations_bf16((M, K), 8)
        xb = inputs.normal_bf16((N, K), 9, std=0.02)
        _check_gemm(bsq, xa, "mxfp8_e4m3", xb, "mxfp8_e4m3", "f32")
        _check_gemm(bsq, xa, "nvfp4", xb, "nvfp4", "bf16")


# ------------------------------------------------ per-expert padded scales
def _padded_capacity(R, G):
    return (R + 127) // 128 * 128 + 128 * G


@pytest.mark.parametrize("case", sorted(GROUPED_CASES))
@pytest.mark.parametrize("align", [32, 16])
def test_repack_grouped_scale_layout(bsq, case, align):
    import torch
    counts, N, K = GROUPED_CASES[case]
    off = inputs.group_offsets(counts)
    R = int(off[-1])
    x = inputs.normal_bf16((R, K), 23)
    c4, s4 = oracle.mx_quantize_rows(x, "mxfp4")
    q4 = upload_q(bsq, "mxfp4", c4, s4)
    # stale bytes in the whole buffer: every byte of the capacity is written by the call
    q8 = codes_at(bsq.empty_grouped("mxfp8_e4m3", R, K, len(counts)), align)
    q8.scales.fill_(0xAB)
    q8.codes.fill_(0xAB)
    bsq.mxfp4_to_mxfp8_grouped_into(q4, q8, torch.from_numpy(off).cuda(), len(counts))
    c8, s8 = oracle.mxfp4_to_mxfp8_rows(c4, s4)
    assert np.array_equal(host_u8(q8.codes).reshape(R, K), c8)
    exp = oracle.swizzle_scales_grouped(s8, off, _padded_capacity(R, len(counts)))
    assert q8.scales.numel() == exp.size
    got = host_u8(q8.scales)
    assert np.array_equal(got, exp), f"{(got != exp).sum()} scale bytes differ"


@pytest.mark.parametrize("case", sorted(GROUPED_CASES))
@pytest.mark.parametrize("path", ["pair", "single_cta"])
def test_grouped_gemm_padded_scales(bsq, monkeypatch, case, path):
    """Grouped GEMM reading A's scales in the per-expert padded layout: tiles
    start at each expert's first row; results as the oracle, nothing written
    outside C."""
    import torch
    monkeypatch.setenv("BSQ_GEMM_1CTA" if path == "single_cta" else "BSQ_GEMM_GROUPED_PAIR", "1")
    counts, N, K = GROUPED_CASES[case]
    G = len(counts)
    off, ca, sa, cw, sw, Ad, Wd = _grouped_case_oracle(case)
    R = int(off[-1])
    A = bsq.empty("mxfp8_e4m3", R, K)
    A.codes.copy_(dev_u8(ca.ravel()))
    A.scales = dev_u8(oracle.swizzle_scales_grouped(sa, off, _padded_capacity(R, G)))
    W = upload_q(bsq, "mxfp8_e4m3", cw, sw)
    guard = 64
    buf = torch.full((R + 2 * guard, N), -7.0, dtype=torch.float32, device="cuda")
    C = buf[guard:guard + R]
    bsq.grouped_gemm_into(A, torch.from_numpy(off).cuda(), bsq.group_views(W, G), C, padded_scales=True)
    bsq.sync_status()
    host = buf.cpu().numpy()
    assert (host[:guard] == -7.0).all() and (host[guard + R:] == -7.0).all(), "write outside C"
    Ch = host[guard:guard + R]
    for g in range(G):
        lo, hi = off[g], off[g + 1]
        if hi == lo:
            continue
        ref, mag = oracle.gemm_full(Ad[lo:hi], Wd[g * N:(g + 1) * N])
        ok, err, tol = gemm_tol_ok(Ch[lo:hi], ref, mag, False)
        assert ok.all(), (case, path, g, int((~ok).sum()))
