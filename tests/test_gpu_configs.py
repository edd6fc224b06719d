"""Full-size parity: every workload at its full size, in the launch
configuration the benchmark times.

Quantized bytes are compared bit for bit on sampled rows (row-wise) and
sampled columns (column-wise), scales at their tiled positions; GEMM
outputs are compared on the sampled rows x sampled columns of C against the
oracle's FP64 reference over exactly dequantized operands.  The oracle
quantizes only the sampled rows (the NVFP4 tensor scale is computed by the
oracle over the whole tensor)."""
import numpy as np
import pytest

import oracle
from block_scaled_precision_03_gb300 import inputs
from _util import dev_bf16, gemm_tol_ok

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(12345)


@pytest.fixture(scope="module")
def bsq():
    import block_scaled_precision_03_gb300 as b
    b.lib()
    return b


def _rows(n, k):
    return np.sort(RNG.choice(n, size=min(k, n), replace=False))


def _gpu_rows_codes(q, rows, fmt):
    """Codes of the given rows of a device QTensor, unpacked to one per byte."""
    import torch
    per_row = q.cols // 2 if oracle.ELEM[fmt] == oracle.E2M1 else q.cols
    idx = torch.from_numpy(np.asarray(rows, dtype=np.int64)).cuda()
    got = q.codes.view(q.rows, per_row).index_select(0, idx).cpu().numpy()
    return oracle.unpack_fp4(got) if oracle.ELEM[fmt] == oracle.E2M1 else got


def _gpu_rows_scales(q, rows, fmt):
    S = q.cols // oracle.BLOCK[fmt]
    buf = q.scales.cpu().numpy()
    s_pad = (S + 3) // 4 * 4
    r = np.asarray(rows)[:, None]
    c = np.arange(S)[None, :]
    off = ((r // 128) * (s_pad // 4) + (c // 4)) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4)
    return buf[off]


def _check_rows(q, x_rows_bits, rows, fmt, s_t=None, what=""):
    """Oracle-quantize x_rows_bits (the sampled source rows) and compare."""
    if fmt == "nvfp4":
        c, s, _ = oracle.nvfp4_quantize_rows(x_rows_bits, s_t)
    else:
        c, s = oracle.mx_quantize_rows(x_rows_bits, fmt)
    gc = _gpu_rows_codes(q, rows, fmt)
    gs = _gpu_rows_scales(q, rows, fmt)
    bad = np.argwhere(gc != c)
    assert len(bad) == 0, f"{what}: {len(bad)} codes differ, first at sampled row {bad[0]}"
    assert np.array_equal(gs, s), f"{what}: scales differ"
    return c, s


def _check_gemm_samples(C_dev, A_codes, A_scales, fa, B_codes, B_scales, fb, m_rows, n_rows, bf16, what,
                        ts_a=None, ts_b=None):
    """C_dev [M, N] on the device; A_codes / A_scales are the oracle's codes
    of the sampled A rows m_rows (all K), B likewise for n_rows."""
    import torch
    Ad = oracle.dequant_rows(A_codes, A_scales, fa, ts_a)
    Bd = oracle.dequant_rows(B_codes, B_scales, fb, ts_b)
    mi = torch.from_numpy(np.asarray(m_rows, np.int64)).cuda()
    ni = torch.from_numpy(np.asarray(n_rows, np.int64)).cuda()
    Csub = C_dev.index_select(0, mi).index_select(1, ni).float().cpu().numpy()
    ref, mag = oracle.gemm_full(Ad, Bd)
    ok, err, tol = gemm_tol_ok(Csub, ref, mag, bf16)
    assert ok.all(), f"{what}: {(~ok).sum()} of {ok.size} sampled outputs outside the bound (max err/tol {np.max(err / tol):.3g})"


def _tensors(bsq, x, fmt, axis):
    return bsq.quantize(dev_bf16(x), fmt, axis)


# ------------------------------------------------------------------ configs
def test_config1_tiny_linear_every_element(bsq):
    import torch
    d = inputs.tiny_linear()
    qa, _ = _tensors(bsq, d["A"], "mxfp8_e4m3", "row")
    qb, _ = _tensors(bsq, d["B"], "mxfp8_e4m3", "row")
    ca, sa = _check_rows(qa, d["A"], np.arange(256), "mxfp8_e4m3", what="A")
    cb, sb = _check_rows(qb, d["B"], np.arange(256), "mxfp8_e4m3", what="B")
    C = bsq.gemm(qa, qb, torch.float32)
    _check_gemm_samples(C, ca, sa, "mxfp8_e4m3", cb, sb, "mxfp8_e4m3", np.arange(256), np.arange(256), False, "C")


def test_config2_llama_up_proj_forward(bsq):
    import torch
    d = inputs.llama_up_proj()
    X, W = d["X"], d["W"]
    qx, _ = _tensors(bsq, X, "mxfp8_e4m3", "row")
    qw, _ = _tensors(bsq, W, "mxfp8_e4m3", "row")
    mr, nr = _rows(8192, 48), _rows(14336, 64)
    cx, sx = _check_rows(qx, X[mr], mr, "mxfp8_e4m3", what="X")
    cw, sw = _check_rows(qw, W[nr], nr, "mxfp8_e4m3", what="W")
    Y = bsq.gemm(qx, qw, torch.bfloat16)
    _check_gemm_samples(Y, cx, sx, "mxfp8_e4m3", cw, sw, "mxfp8_e4m3", mr, nr, True, "Y")
    bsq.sync_status()


def test_config3_llama_up_proj_backward(bsq):
    import torch
    d = inputs.llama_up_proj_backward()
    X, W, dY = d["X"], d["W"], d["dY"]
    qdy_r, qdy_c = _tensors(bsq, dY, "mxfp8_e5m2", "both")
    _, qw_c = _tensors(bsq, W, "mxfp8_e4m3", "col")
    _, qx_c = _tensors(bsq, X, "mxfp8_e4m3", "col")
    mr = _rows(8192, 48)           # rows of dY / dX
    kr = _rows(4096, 48)           # columns of W / X = rows of W^T, X^T
    nr = _rows(14336, 48)          # columns of dY = rows of dY^T
    c_dyr, s_dyr = _check_rows(qdy_r, dY[mr], mr, "mxfp8_e5m2", what="dY row")
    c_dyc, s_dyc = _check_rows(qdy_c, np.ascontiguousarray(dY[:, nr].T), nr, "mxfp8_e5m2", what="dY col")
    c_wc, s_wc = _check_rows(qw_c, np.ascontiguousarray(W[:, kr].T), kr, "mxfp8_e4m3", what="W col")
    c_xc, s_xc = _check_rows(qx_c, np.ascontiguousarray(X[:, kr].T), kr, "mxfp8_e4m3", what="X col")
    dX = bsq.gemm(qdy_r, qw_c, torch.bfloat16)          # [8192, 4096], K = 14336
    _check_gemm_samples(dX, c_dyr, s_dyr, "mxfp8_e5m2", c_wc, s_wc, "mxfp8_e4m3", mr, kr, True, "dgrad")
    dW = bsq.gemm(qdy_c, qx_c, torch.bfloat16)          # [14336, 4096], K = 8192
    _check_gemm_samples(dW, c_dyc, s_dyc, "mxfp8_e5m2", c_xc, s_xc, "mxfp8_e4m3", nr, kr, True, "wgrad")
    bsq.sync_status()


def test_config4_nvfp4_forward(bsq):
    import torch
    d = inputs.nvfp4_forward()
    for xk, wk in (("X", "W"), ("X2", "W2")):
        X, W = d[xk], d[wk]
        qx, _ = _tensors(bsq, X, "nvfp4", "row")
        qw, _ = _tensors(bsq, W, "nvfp4", "row")
        tx, tw = oracle.nvfp4_tensor_scale(X), oracle.nvfp4_tensor_scale(W)
        assert float(qx.tensor_scale.cpu()[0]) == tx and float(qw.tensor_scale.cpu()[0]) == tw
        mr, nr = _rows(X.shape[0], 48), _rows(W.shape[0], 48)
        cx, sx = _check_rows(qx, X[mr], mr, "nvfp4", tx, what=f"{xk}")
        cw, sw = _check_rows(qw, W[nr], nr, "nvfp4", tw, what=f"{wk}")
        Y = bsq.gemm(qx, qw, torch.bfloat16)
        _check_gemm_samples(Y, cx, sx, "nvfp4", cw, sw, "nvfp4", mr, nr, True, f"Y {xk}", tx, tw)
    bsq.sync_status()


def test_config5_moe_grouped(bsq):
    import torch
    d = inputs.moe_grouped()
    A, W, off = d["A"], d["W"].reshape(-1, 7168), d["offsets"]
    G, N = 64, 2048
    assert d["counts"].min() > 0 and off[-1] == 32768
    q4, _ = _tensors(bsq, A, "mxfp4", "row")
    q8 = bsq.mxfp4_to_mxfp8(q4)
    qw, _ = _tensors(bsq, W, "mxfp8_e4m3", "row")
    # activations: MXFP4 codes, then the re-encoded MXFP8 codes, on sampled rows
    # (random rows plus the first and last row of every expert)
    mr = np.unique(np.concatenate([_rows(32768, 40), off[1:-1] - 1, off[1:-1]]))
    c4, s4 = _check_rows(q4, A[mr], mr, "mxfp4", what="A mxfp4")
    c8, s8 = oracle.mxfp4_to_mxfp8_rows(c4, s4)
    assert np.array_equal(_gpu_rows_codes(q8, mr, "mxfp8_e4m3"), c8)
    assert np.array_equal(_gpu_rows_scales(q8, mr, "mxfp8_e4m3"), s8)
    offd = torch.from_numpy(off).cuda()
    Y = bsq.grouped_gemm(q8, offd, bsq.group_views(qw, G), torch.bfloat16)
    # the benchmark's path: re-encode with per-expert padded scales, grouped GEMM reading them
    q8p = bsq.mxfp4_to_mxfp8_grouped(q4, offd, G)
    assert torch.equal(q8p.codes, q8.codes)
    Yp = bsq.grouped_gemm(q8p, offd, bsq.group_views(qw, G), torch.bfloat16, padded_scales=True)
    # for each sampled A row, its expert's weights on sampled output columns
    nr = _rows(N, 24)
    groups = np.searchsorted(off, mr, side="right") - 1
    ncols = torch.from_numpy(nr).cuda()
    for name, out in (("plain", Y), ("padded", Yp)):
        Yn = out.index_select(1, ncols)
        for g in np.unique(groups):
            sel = np.flatnonzero(groups == g)
            wr = g * N + nr
            cw, sw = _check_rows(qw, W[wr], wr, "mxfp8_e4m3", what=f"W_{g}")
            _check_gemm_samples(Yn, c8[sel], s8[sel], "mxfp8_e4m3", cw, sw, "mxfp8_e4m3", mr[sel],
                                np.arange(len(nr)), True, f"{name} expert {g}")
    bsq.sync_status()
