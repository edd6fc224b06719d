"""Full-size parity: every workload at its full size, in the launch
configuration the benchmark times.

Every code and scale byte of every quantized tensor (row-wise, column-wise,
re-encoded, per-expert padded scales) is compared with the oracle's
quantization of the whole tensor.  GEMM outputs are compared on 512 random
rows x every column of C (every row of the tiny linear) against the
oracle's FP64 reference over exactly dequantized operands, within
|C - ref| <= 1e-5 * sum|a b| plus BF16 output rounding.  All outputs start
as 0xAB bytes and GEMM outputs sit between guard bands."""
import numpy as np
import pytest

import oracle
from block_scaled_precision_03_gb300 import inputs
from _util import (dev_bf16, gemm_tol_ok, host_u8, qz, gemm_g, grouped_g, repack, repack_grouped)

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(12345)
GEMM_ROWS = 512


@pytest.fixture(scope="module")
def bsq():
    import block_scaled_precision_03_gb300 as b
    b.lib()
    return b


def _rows(n, k):
    return np.sort(RNG.choice(n, size=min(k, n), replace=False))


def _check_all(q, x_bits, fmt, s_t=None, what=""):
    """Every code and scale byte of the device tensor q equals the oracle's
    row-wise quantization of x_bits (for a column-wise output, pass the
    transpose); returns the oracle's (codes, row-major scales)."""
    if fmt == "nvfp4":
        c, s, _ = oracle.nvfp4_quantize_rows(x_bits, s_t)
    else:
        c, s = oracle.mx_quantize_rows(x_bits, fmt)
    exp_c = oracle.storage_codes(c, fmt).ravel()
    got_c = host_u8(q.codes)
    nbad = int((got_c != exp_c).sum())
    assert nbad == 0, f"{what}: {nbad} of {got_c.size} code bytes differ"
    exp_s = oracle.swizzle_scales(s)
    got_s = host_u8(q.scales)
    nbad = int((got_s != exp_s).sum())
    assert nbad == 0, f"{what}: {nbad} of {got_s.size} scale bytes differ"
    return c, s


def _check_gemm_rows(C_dev, A_codes, A_scales, fa, B_codes, B_scales, fb, m_rows, bf16, what,
                     ts_a=None, ts_b=None):
    """Rows m_rows of C_dev [M, N], every column, against the oracle: A_codes /
    A_scales are the oracle's codes of those A rows, B_* all of B."""
    import torch
    Ad = oracle.dequant_rows(A_codes, A_scales, fa, ts_a)
    Bd = oracle.dequant_rows(B_codes, B_scales, fb, ts_b)
    mi = torch.from_numpy(np.asarray(m_rows, np.int64)).cuda()
    Csub = C_dev.index_select(0, mi).float().cpu().numpy()
    ref, mag = oracle.gemm_full(Ad, Bd)
    ok, err, tol = gemm_tol_ok(Csub, ref, mag, bf16)
    assert ok.all(), (f"{what}: {(~ok).sum()} of {ok.size} outputs outside the bound "
                      f"(max err/tol {np.max(err / tol):.3g})")
    return float(np.max(err / tol))


def _t(x):
    return np.ascontiguousarray(x.T)


# ------------------------------------------------------------------ configs
def test_config1_tiny_linear_every_element(bsq):
    import torch
    d = inputs.tiny_linear()
    qa, _ = qz(bsq, dev_bf16(d["A"]), "mxfp8_e4m3", "row")
    qb, _ = qz(bsq, dev_bf16(d["B"]), "mxfp8_e4m3", "row")
    ca, sa = _check_all(qa, d["A"], "mxfp8_e4m3", what="A")
    cb, sb = _check_all(qb, d["B"], "mxfp8_e4m3", what="B")
    C = gemm_g(bsq, qa, qb, torch.float32)
    _check_gemm_rows(C, ca, sa, "mxfp8_e4m3", cb, sb, "mxfp8_e4m3", np.arange(256), False, "C")


def test_config2_llama_up_proj_forward(bsq):
    import torch
    d = inputs.llama_up_proj()
    X, W = d["X"], d["W"]
    qx, _ = qz(bsq, dev_bf16(X), "mxfp8_e4m3", "row")
    qw, _ = qz(bsq, dev_bf16(W), "mxfp8_e4m3", "row")
    cx, sx = _check_all(qx, X, "mxfp8_e4m3", what="X")
    cw, sw = _check_all(qw, W, "mxfp8_e4m3", what="W")
    Y = gemm_g(bsq, qx, qw, torch.bfloat16)
    mr = _rows(8192, GEMM_ROWS)
    _check_gemm_rows(Y, cx[mr], sx[mr], "mxfp8_e4m3", cw, sw, "mxfp8_e4m3", mr, True, "Y")
    bsq.sync_status()


def test_config3_llama_up_proj_backward(bsq):
    import torch
    d = inputs.llama_up_proj_backward()
    X, W, dY = d["X"], d["W"], d["dY"]
    qdy_r, qdy_c = qz(bsq, dev_bf16(dY), "mxfp8_e5m2", "both")
    _, qw_c = qz(bsq, dev_bf16(W), "mxfp8_e4m3", "col")
    _, qx_c = qz(bsq, dev_bf16(X), "mxfp8_e4m3", "col")
    c_dyr, s_dyr = _check_all(qdy_r, dY, "mxfp8_e5m2", what="dY row")
    c_dyc, s_dyc = _check_all(qdy_c, _t(dY), "mxfp8_e5m2", what="dY col")
    c_wc, s_wc = _check_all(qw_c, _t(W), "mxfp8_e4m3", what="W col")
    c_xc, s_xc = _check_all(qx_c, _t(X), "mxfp8_e4m3", what="X col")
    dX = gemm_g(bsq, qdy_r, qw_c, torch.bfloat16)          # [8192, 4096], K = 14336
    mr = _rows(8192, GEMM_ROWS)
    _check_gemm_rows(dX, c_dyr[mr], s_dyr[mr], "mxfp8_e5m2", c_wc, s_wc, "mxfp8_e4m3", mr, True, "dgrad")
    dW = gemm_g(bsq, qdy_c, qx_c, torch.bfloat16)          # [14336, 4096], K = 8192
    nr = _rows(14336, GEMM_ROWS)
    _check_gemm_rows(dW, c_dyc[nr], s_dyc[nr], "mxfp8_e5m2", c_xc, s_xc, "mxfp8_e4m3", nr, True, "wgrad")
    bsq.sync_status()


def test_config4_nvfp4_forward(bsq):
    import torch
    d = inputs.nvfp4_forward()
    for xk, wk in (("X", "W"), ("X2", "W2")):
        X, W = d[xk], d[wk]
        qx, _ = qz(bsq, dev_bf16(X), "nvfp4", "row")
        qw, _ = qz(bsq, dev_bf16(W), "nvfp4", "row")
        tx, tw = oracle.nvfp4_tensor_scale(X), oracle.nvfp4_tensor_scale(W)
        assert float(qx.tensor_scale.cpu()[0]) == tx and float(qw.tensor_scale.cpu()[0]) == tw
        cx, sx = _check_all(qx, X, "nvfp4", tx, what=xk)
        cw, sw = _check_all(qw, W, "nvfp4", tw, what=wk)
        Y = gemm_g(bsq, qx, qw, torch.bfloat16)
        mr = _rows(X.shape[0], GEMM_ROWS)
        _check_gemm_rows(Y, cx[mr], sx[mr], "nvfp4", cw, sw, "nvfp4", mr, True, f"Y {xk}", tx, tw)
    bsq.sync_status()


def test_config5_moe_grouped(bsq):
    import torch
    d = inputs.moe_grouped()
    A, W, off = d["A"], d["W"].reshape(-1, 7168), d["offsets"]
    G, N = 64, 2048
    assert d["counts"].min() > 0 and off[-1] == 32768
    q4, _ = qz(bsq, dev_bf16(A), "mxfp4", "row")
    q8 = repack(bsq, q4)
    qw, _ = qz(bsq, dev_bf16(W), "mxfp8_e4m3", "row")
    c4, s4 = _check_all(q4, A, "mxfp4", what="A mxfp4")
    c8, s8 = oracle.mxfp4_to_mxfp8_rows(c4, s4)
    assert np.array_equal(host_u8(q8.codes), c8.ravel()), "re-encoded codes differ"
    assert np.array_equal(host_u8(q8.scales), oracle.swizzle_scales(s8)), "re-encoded scales differ"
    offd = torch.from_numpy(off).cuda()
    # the benchmark's path: re-encode with per-expert padded scales, grouped GEMM reading them
    q8p = repack_grouped(bsq, q4, offd, G)
    assert torch.equal(q8p.codes, q8.codes)
    exp_p = oracle.swizzle_scales_grouped(s8, off, capacity_rows=q8p.scales.numel() // ((s8.shape[1] + 3) // 4 * 4))
    assert np.array_equal(host_u8(q8p.scales), exp_p), "padded re-encoded scales differ"
    Y = grouped_g(bsq, q8, offd, bsq.group_views(qw, G), torch.bfloat16)
    Yp = grouped_g(bsq, q8p, offd, bsq.group_views(qw, G), torch.bfloat16, padded_scales=True)
    # every weight byte, expert by expert, and for 512 random activation rows
    # (plus the first and last row of every expert) every output column
    mr = np.unique(np.concatenate([_rows(32768, GEMM_ROWS), off[1:-1] - 1, off[1:-1]]))
    groups = np.searchsorted(off, mr, side="right") - 1
    wc, ws = oracle.mx_quantize_rows(W, "mxfp8_e4m3")
    assert np.array_equal(host_u8(qw.codes), wc.ravel()), "expert weight codes differ"
    assert np.array_equal(host_u8(qw.scales), oracle.swizzle_scales(ws)), "expert weight scales differ"
    for name, out in (("plain", Y), ("padded", Yp)):
        for g in np.unique(groups):
            sel = np.flatnonzero(groups == g)
            rows_g = slice(g * N, (g + 1) * N)
            _check_gemm_rows(out[:, :], c8[mr[sel]], s8[mr[sel]], "mxfp8_e4m3", wc[rows_g], ws[rows_g],
                             "mxfp8_e4m3", mr[sel], True, f"{name} expert {g}")
    bsq.sync_status()
