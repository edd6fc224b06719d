"""Parity of the rows beyond the core path, against the oracle.

NVFP4 with delayed scaling: the tensor scale comes from an amax history of
previous steps ("FP8 Training Infrastructure", DelayedScaling recipe with
amax_history_len = 16, algorithm max); codes, scales, the tensor scale and
the updated history must equal the oracle's byte for byte."""
import numpy as np
import pytest

import oracle
from block_scaled_precision_03_gb300 import inputs
from _util import (dev_bf16, host_u8, codes_at, qz, qz_delayed, gemm_g, deq, grouped_g, repack_grouped, repack_col, repack_1x128, repack, poisoned_qtensor, guarded)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsq():
    import block_scaled_precision_03_gb300 as b
    b.lib()
    return b


def _abs_max(x_bits):
    f = (np.asarray(x_bits, np.uint32) << 16).view(np.float32)
    return float(np.abs(f[np.isfinite(f)]).max())


def _check_delayed(q, codes, scales, s_t, what):
    exp_c = oracle.storage_codes(codes, "nvfp4")
    got_c = host_u8(q.codes).reshape(exp_c.shape)
    assert np.array_equal(got_c, exp_c), f"{what}: {(got_c != exp_c).sum()} code bytes differ"
    got_s = host_u8(q.scales)
    assert np.array_equal(got_s, oracle.swizzle_scales(scales)), f"{what}: scales differ"
    assert np.float32(q.tensor_scale.cpu().numpy()[0]) == np.float32(s_t), what


@pytest.mark.parametrize("shape", [(256, 512), (304, 1040), (16, 16), (1008, 96)])
@pytest.mark.parametrize("axis", ["row", "col", "both"])
def test_delayed_nvfp4_matches_oracle(bsq, shape, axis):
    import torch
    R, C = shape
    x = inputs.outlier_activations_bf16(shape, 11)
    hist0 = np.float32([3.0, 0.0, 7.5, 1.0] + [0.0] * 12)
    h = torch.from_numpy(hist0.copy()).cuda()
    row, col = qz_delayed(bsq, dev_bf16(x), h, axis)
    exp = oracle.nvfp4_delayed_quantize(x, hist0, axis)
    if row is not None:
        _check_delayed(row, *exp["row"], exp["s_t"], f"row {shape}")
    if col is not None:
        _check_delayed(col, *exp["col"], exp["s_t"], f"col {shape}")
    np.testing.assert_array_equal(h.cpu().numpy(), exp["history"])
    bsq.sync_status()


def test_delayed_nvfp4_consecutive_steps(bsq):
    # three steps on different tensors share one history in stream order
    import torch
    hist = np.zeros(16, np.float32)
    h = torch.from_numpy(hist.copy()).cuda()
    for step, scale in enumerate((1.0, 8.0, 0.25)):
        x = inputs.normal_bf16((128, 256), 20 + step, std=scale)
        row, _ = qz_delayed(bsq, dev_bf16(x), h, "row")
        exp = oracle.nvfp4_delayed_quantize(x, hist, "row")
        _check_delayed(row, *exp["row"], exp["s_t"], f"step {step}")
        hist = exp["history"]
        np.testing.assert_array_equal(h.cpu().numpy(), hist)
    assert hist[0] == np.float32(_abs_max(x))


def test_delayed_nvfp4_saturates(bsq):
    import torch
    x = inputs.normal_bf16((64, 256), 30)
    hist0 = np.float32([_abs_max(x) / 64.0] + [0.0] * 15)
    h = torch.from_numpy(hist0.copy()).cuda()
    row, _ = qz_delayed(bsq, dev_bf16(x), h, "row")
    exp = oracle.nvfp4_delayed_quantize(x, hist0, "row")
    _check_delayed(row, *exp["row"], exp["s_t"], "saturating")
    v = deq(bsq, row, torch.float32).cpu().numpy()
    assert np.abs(v).max() == np.float32(6.0 * 448.0 * exp["s_t"])


def test_delayed_nvfp4_full_size_equals_just_in_time(bsq):
    # config 4's X (8192 x 4096): with its own amax in the history the one-pass
    # delayed path gives the two-pass result exactly
    import torch
    X = inputs.nvfp4_forward()["X"]
    xd = dev_bf16(X)
    jit, _ = qz(bsq, xd, "nvfp4", "row")
    h = torch.zeros(16, dtype=torch.float32, device="cuda")
    h[3] = oracle.tensor_amax(X)
    dl, _ = qz_delayed(bsq, xd, h, "row")
    assert torch.equal(jit.codes, dl.codes) and torch.equal(jit.scales, dl.scales)
    assert torch.equal(jit.tensor_scale, dl.tensor_scale)
    assert float(h[0]) == oracle.tensor_amax(X) and float(h[4]) == oracle.tensor_amax(X) and float(h[3]) == 0.0
    bsq.sync_status()


def test_delayed_nvfp4_empty_history_unit_scale(bsq):
    import torch
    x = inputs.normal_bf16((32, 64), 31)
    h = torch.zeros(16, dtype=torch.float32, device="cuda")
    row, _ = qz_delayed(bsq, dev_bf16(x), h, "row")
    assert float(row.tensor_scale.cpu()[0]) == 1.0
    c, s, _ = oracle.nvfp4_quantize_rows(x, 1.0)
    _check_delayed(row, c, s, 1.0, "unit scale")


# ------------------------------------------------------------ FP4RowToFP8Col
def _check_fp8col(out, codes8, scales8, what):
    got_c = host_u8(out.codes).reshape(codes8.shape)
    bad = np.argwhere(got_c != codes8)
    assert len(bad) == 0, f"{what}: {len(bad)} code bytes differ, first at {tuple(bad[0])}"
    assert np.array_equal(host_u8(out.scales), oracle.swizzle_scales(scales8)), f"{what}: scales differ"


@pytest.mark.parametrize("shape", [(128, 128), (96, 160), (32, 32), (416, 4160), (4128, 96)])
def test_fp4_row_to_fp8_col_random_codes_and_scales(bsq, shape):
    # every nibble, scale bytes over the whole range including 0, 254 and NaN
    from _util import upload_q
    R, C = shape
    rng = np.random.default_rng(R * 7 + C)
    c4 = rng.integers(0, 16, (R, C)).astype(np.uint8)
    s4 = rng.integers(0, 255, (R, C // 32)).astype(np.uint8)
    s4[rng.random(s4.shape) < 0.01] = 0xFF
    s4[0, 0], s4[-1, -1] = 0, 254
    q4 = upload_q(bsq, "mxfp4", c4, s4)
    out = repack_col(bsq, q4)
    c8, s8 = oracle.mxfp4_row_to_mxfp8_col(c4, s4)
    _check_fp8col(out, c8, s8, f"random {shape}")
    bsq.sync_status()


@pytest.mark.parametrize("kind", ["narrow", "spread14", "zero_columns", "sparse", "floor", "mixed"])
@pytest.mark.parametrize("align", [32, 16])
def test_fp4_row_to_fp8_col_scale_structures(bsq, kind, align):
    """Row scales within a few binades (the kernel's fast path, half products),
    spread to its limit, all-zero columns, sparse codes, scales at the E8M0
    floor, and blocks of both paths side by side in one launch."""
    from _util import upload_q
    R, C = 512, 256
    rng = np.random.default_rng(len(kind) * 131)
    c4 = rng.integers(0, 16, (R, C)).astype(np.uint8)
    base = rng.integers(20, 230, (R // 32, 1))
    spread = {"narrow": 3, "spread14": 14, "zero_columns": 2, "sparse": 6, "floor": 0, "mixed": 3}[kind]
    s_row = np.clip(np.repeat(base, 32, axis=0) + rng.integers(-spread, spread + 1, (R, 1)), 0, 254)
    if kind == "floor":
        s_row = rng.integers(0, 20, (R, 1))
    if kind == "zero_columns":
        c4[:, rng.choice(C, 40, replace=False)] = 0
        c4[:64, :96] = 8                                  # negative zeros
    if kind == "sparse":
        c4[rng.random((R, C)) < 0.7] = 0
    if kind == "mixed":
        s_row[::3] = rng.integers(0, 255, (len(s_row[::3]), 1))   # wide spread in some blocks
        s_row[100] = 0xFF                                          # one NaN row
    s4 = np.repeat(s_row, C // 32, axis=1).astype(np.uint8)
    q4 = upload_q(bsq, "mxfp4", c4, s4)
    out = codes_at(bsq.empty("mxfp8_e4m3", C, R), align)       # both store widths
    bsq.mxfp4_to_mxfp8_col_into(q4, out)
    c8, s8 = oracle.mxfp4_row_to_mxfp8_col(c4, s4)
    _check_fp8col(out, c8, s8, kind)
    bsq.sync_status()


@pytest.mark.parametrize("align", [32, 16])
def test_fp4_row_to_fp8_col_fast_path_edges(bsq, align):
    """Blocks at the edges of the kernel's half-precision path: row scales
    spread over exactly 0, 1, 13, 14 (the path's limit), 15 and 40 binades;
    code 0.5 in a row 14 binades below the block's largest scale (a
    subnormal half product); columns whose only nonzero codes sit in the
    lowest-scale rows (a column factor at and beyond its exponent limit),
    all-zero columns and columns of negative zeros beside full ones; scale
    bytes near 0 and 254."""
    from _util import upload_q
    R, C = 32 * 96, 128
    rng = np.random.default_rng(733)
    c4 = rng.integers(0, 16, (R, C)).astype(np.uint8)
    s_row = np.zeros(R, dtype=np.int64)
    spreads = [0, 1, 13, 14, 15, 40]
    for b in range(R // 32):
        d = spreads[b % len(spreads)]
        top = int(rng.integers(d + 2, 255)) if b % 7 else (d + 1 if b % 2 else 254)
        rows = slice(32 * b, 32 * b + 32)
        sr = top - rng.integers(0, d + 1, 32)
        sr[0], sr[31] = top, top - d
        s_row[rows] = sr
        low = np.flatnonzero(sr == top - d)                 # the block's lowest-scale rows
        blk = c4[rows]                                      # a view: edits land in c4
        mode = b % 5
        cols = rng.choice(C, 24, replace=False)
        if mode == 1:                                       # code 0.5 (magnitude 1) in the lowest rows only
            blk[:, cols] = 0
            blk[np.ix_(low, cols)] = rng.choice([1, 9], (len(low), len(cols)))
        elif mode == 2:                                     # small codes in the lowest rows only
            blk[:, cols] = 0
            blk[np.ix_(low, cols)] = rng.integers(1, 8, (len(low), len(cols)))
        elif mode == 3:                                     # all-zero and negative-zero columns
            blk[:, cols[:12]] = 0
            blk[:, cols[12:]] = 8
        elif mode == 4:                                     # only rows a few binades below the top
            mid = np.flatnonzero(sr <= top - min(d, 7))
            blk[:, cols] = 0
            if len(mid):
                blk[np.ix_(mid, cols)] = rng.integers(1, 16, (len(mid), len(cols)))
    s4 = np.repeat(np.clip(s_row, 0, 254)[:, None], C // 32, axis=1).astype(np.uint8)
    q4 = upload_q(bsq, "mxfp4", c4, s4)
    out = codes_at(bsq.empty("mxfp8_e4m3", C, R), align)
    bsq.mxfp4_to_mxfp8_col_into(q4, out)
    c8, s8 = oracle.mxfp4_row_to_mxfp8_col(c4, s4)
    _check_fp8col(out, c8, s8, f"fast-path edges, align {align}")
    bsq.sync_status()


def test_fp4_row_to_fp8_col_from_bf16(bsq):
    # the MoE path: BF16 activations -> MXFP4 rows (GPU) -> FP8 columns (GPU)
    x = inputs.normal_bf16((1024, 7168), 50)
    q4, _ = qz(bsq, dev_bf16(x), "mxfp4", "row")
    c4, s4 = oracle.mx_quantize_rows(x, "mxfp4")
    out = repack_col(bsq, q4)
    c8, s8 = oracle.mxfp4_row_to_mxfp8_col(c4, s4)
    _check_fp8col(out, c8, s8, "from bf16")


def test_fp4_row_to_fp8_col_full_size_sampled(bsq):
    # config 5's activations (32768 x 7168); the oracle checks four whole
    # 32-column groups (every row, every scale block of those columns)
    d = inputs.moe_grouped()
    A = d["A"]
    q4, _ = qz(bsq, dev_bf16(A), "mxfp4", "row")
    out = repack_col(bsq, q4)
    rng = np.random.default_rng(51)
    groups = np.sort(rng.choice(7168 // 32, size=4, replace=False))
    S_out = 32768 // 32
    codes_all = host_u8(out.codes).reshape(7168, 32768)
    sc_buf = host_u8(out.scales)
    for g in groups:
        cols = np.arange(32 * g, 32 * g + 32)
        c4, s4 = oracle.mx_quantize_rows(np.ascontiguousarray(A[:, cols]), "mxfp4")
        c8, s8 = oracle.mxfp4_row_to_mxfp8_col(c4, s4)
        assert np.array_equal(codes_all[cols], c8), f"group {g}: codes differ"
        r = cols[:, None]
        cc = np.arange(S_out)[None, :]
        off = ((r // 128) * (S_out // 4) + cc // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + cc % 4
        assert np.array_equal(sc_buf[off], s8), f"group {g}: scales differ"
    bsq.sync_status()


# ------------------------------------------------------- native MXFP4 GEMM
def _mx4_gemm_check(bsq, xa, xb, out, groups=None):
    """Oracle-quantized MXFP4 operands uploaded, GEMM on the device, compared
    with the FP64 product of the exactly dequantized operands."""
    import torch
    from _util import upload_q, gemm_tol_ok
    ca, sa = oracle.mx_quantize_rows(xa, "mxfp4")
    cb, sb = oracle.mx_quantize_rows(xb, "mxfp4")
    A = upload_q(bsq, "mxfp4", ca, sa)
    B = upload_q(bsq, "mxfp4", cb, sb)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    Ad = oracle.dequant_rows(ca, sa, "mxfp4")
    Bd = oracle.dequant_rows(cb, sb, "mxfp4")
    if groups is None:
        C = gemm_g(bsq, A, B, dt).float().cpu().numpy()
        pairs = [(slice(0, xa.shape[0]), slice(0, xb.shape[0]))]
    else:
        off = inputs.group_offsets(groups)
        N = xb.shape[0] // len(groups)
        C = grouped_g(bsq, A, torch.from_numpy(off).cuda(), bsq.group_views(B, len(groups)), dt)
        C = C.float().cpu().numpy()
        pairs = [(slice(off[g], off[g + 1]), slice(g * N, (g + 1) * N)) for g in range(len(groups)) if off[g + 1] > off[g]]
    for rows, brows in pairs:
        ref, mag = oracle.gemm_full(Ad[rows], Bd[brows])
        ok, err, tol = gemm_tol_ok(C[rows], ref, mag, out == "bf16")
        assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the bound (max err/tol {np.max(err / tol):.3g})"


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (1, 1, 32), (200, 300, 96), (257, 513, 4160), (64, 640, 1024),
                                   (300, 256, 7168)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gemm_mxfp4_shapes(bsq, M, N, K, out):
    xa = inputs.outlier_activations_bf16((M, K), 60)
    xb = inputs.normal_bf16((N, K), 61, std=0.02)
    _mx4_gemm_check(bsq, xa, xb, out)
    bsq.sync_status()


def test_grouped_gemm_mxfp4(bsq):
    counts = np.array([700, 0, 129, 1, 383, 256, 1000, 0, 31], dtype=np.int64)
    N, K = 256, 4160
    xa = inputs.normal_bf16((int(counts.sum()), K), 62)
    xb = inputs.normal_bf16((len(counts) * N, K), 63, std=0.02)
    _mx4_gemm_check(bsq, xa, xb, "f32", groups=counts)
    bsq.sync_status()


def test_gemm_mxfp4_single_scale_probe(bsq):
    """Codes all 1.0, one scale per (row, 32-block) drawn near 2^0: every
    scale byte must reach the MMA for the row and K-block it belongs to
    (each MMA reads a byte pair of a 4-byte scale word)."""
    import torch
    from _util import upload_q
    M, N, K = 128, 256, 512
    one = oracle.encode(oracle.E2M1, 1.0)
    ca = np.full((M, K), one, np.uint8)
    cb = np.full((N, K), one, np.uint8)
    rng = np.random.default_rng(64)
    sa = (127 + rng.integers(-3, 4, (M, K // 32))).astype(np.uint8)
    sb = (127 + rng.integers(-3, 4, (N, K // 32))).astype(np.uint8)
    C = gemm_g(bsq, upload_q(bsq, "mxfp4", ca, sa), upload_q(bsq, "mxfp4", cb, sb), torch.float32).cpu().numpy()
    ref = 32.0 * (np.exp2(sa.astype(np.float64) - 127) @ np.exp2(sb.astype(np.float64) - 127).T)
    np.testing.assert_array_equal(C, ref.astype(np.float32))


# ------------------------------------------------- MXFP4 -> FP8 1x128 blocks
@pytest.mark.parametrize("shape", [(64, 256), (33, 160), (1, 32), (300, 7168), (129, 4160)])
@pytest.mark.parametrize("spread", [0, 5, 14, 40, 254])
def test_1x128_random_codes_and_scales(bsq, shape, spread):
    """Every nibble; block scales up to `spread` binades below the row's
    largest (exact, subnormal and flushed shifts); ragged last groups; NaN."""
    from _util import upload_q
    R, C = shape
    rng = np.random.default_rng(R * 131 + C + spread)
    c4 = rng.integers(0, 16, (R, C)).astype(np.uint8)
    top = rng.integers(0, 255, (R, 1))
    s4 = np.clip(top - rng.integers(0, spread + 1, (R, C // 32)), 0, 254).astype(np.uint8)
    if spread == 40:
        s4[rng.random(s4.shape) < 0.02] = 0xFF
    q4 = upload_q(bsq, "mxfp4", c4, s4)
    codes, scales = repack_1x128(bsq, q4)
    c8, s8 = oracle.mxfp4_to_fp8_1x128(c4, s4)
    got = host_u8(codes)
    bad = np.argwhere(got != c8)
    assert len(bad) == 0, f"{len(bad)} codes differ, first at {tuple(bad[0])}"
    assert np.array_equal(host_u8(scales), s8)
    bsq.sync_status()


@pytest.mark.parametrize("align", [32, 16])
def test_1x128_from_bf16_both_store_widths(bsq, align):
    # the MoE activations' path: BF16 -> MXFP4 rows (GPU) -> FP8 1x128 (GPU)
    import torch
    x = inputs.outlier_activations_bf16((512, 7168), 61)
    q4, _ = qz(bsq, dev_bf16(x), "mxfp4", "row")
    c4, s4 = oracle.mx_quantize_rows(x, "mxfp4")
    buf = torch.full((512 * 7168 + 16,), 0xAB, dtype=torch.uint8, device="cuda")
    codes = (buf[16:] if align == 16 else buf[:-16]).view(512, 7168)
    assert codes.data_ptr() % 32 == (16 if align == 16 else 0)
    scales = torch.full((512, 56), 0xAB, dtype=torch.uint8, device="cuda")
    bsq.mxfp4_to_fp8_1x128_into(q4, codes, scales)
    c8, s8 = oracle.mxfp4_to_fp8_1x128(c4, s4)
    assert np.array_equal(host_u8(codes), c8) and np.array_equal(host_u8(scales), s8)


def test_1x128_full_size_sampled(bsq):
    # the MoE activations at full size (32768 x 7168): sampled rows, every group
    d = inputs.moe_grouped()
    A = d["A"]
    q4, _ = qz(bsq, dev_bf16(A), "mxfp4", "row")
    codes, scales = repack_1x128(bsq, q4)
    rows = np.sort(np.random.default_rng(62).choice(32768, 48, replace=False))
    c4, s4 = oracle.mx_quantize_rows(np.ascontiguousarray(A[rows]), "mxfp4")
    c8, s8 = oracle.mxfp4_to_fp8_1x128(c4, s4)
    import torch
    idx = torch.from_numpy(rows).cuda()
    assert np.array_equal(host_u8(codes.index_select(0, idx)), c8)
    assert np.array_equal(host_u8(scales.index_select(0, idx)), s8)
    bsq.sync_status()
