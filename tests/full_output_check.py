#!/usr/bin/env python3
"""Full-output GEMM check of every workload, run once on a GPU and recorded.

For each GEMM of the benchmark step (the forward, dgrad and wgrad MXFP8
GEMMs of the Llama-3-8B up-projection, the two NVFP4 forward GEMMs and the
64-expert MoE grouped GEMM), in the launch configuration the benchmark
uses, this compares EVERY output element with the oracle: the oracle
quantizes the BF16 inputs itself, dequantizes exactly, and forms
ref = sum_k a_k b_k and mag = sum_k |a_k b_k| in FP64 (oracle.gemm_full_matmul);
an output passes when |C - ref| <= 1e-5 mag (1 + 2^-8) + 2^-8 |ref| (BF16
output).  Before the GEMMs, every quantized byte is compared with the
oracle's.  Prints one line per GEMM: outputs checked, failures, max err/tol.

Run: python tests/full_output_check.py  (needs a CUDA device; a few minutes)
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np
import torch

import oracle
import block_scaled_precision_03_gb300 as bsq
from block_scaled_precision_03_gb300 import inputs
from _util import dev_bf16, host_u8, gemm_tol_ok

CHUNK = 1024


def quantized(x, fmt, axis):
    """Device quantization of x plus the oracle's codes / scales of the
    requested orientation, after a byte-for-byte comparison."""
    row, col = bsq.quantize(dev_bf16(x), fmt, axis)
    q = row if axis == "row" else col
    src = x if axis == "row" else np.ascontiguousarray(x.T)
    c, s, t = oracle.quantize_rows(src, fmt)
    assert np.array_equal(host_u8(q.codes), oracle.storage_codes(c, fmt).ravel()), f"{fmt} {axis} codes"
    assert np.array_equal(host_u8(q.scales), oracle.swizzle_scales(s)), f"{fmt} {axis} scales"
    return q, c, s, t


def check(name, C_dev, ca, sa, fa, ta, cb, sb, fb, tb):
    Bd = oracle.dequant_rows(cb, sb, fb, tb)
    M = C_dev.shape[0]
    bad, worst = 0, 0.0
    for m0 in range(0, M, CHUNK):
        m1 = min(M, m0 + CHUNK)
        Ad = oracle.dequant_rows(ca[m0:m1], sa[m0:m1], fa, ta)
        ref, mag = oracle.gemm_full_matmul(Ad, Bd)
        C = C_dev[m0:m1].float().cpu().numpy()
        ok, err, tol = gemm_tol_ok(C, ref, mag, True)
        bad += int((~ok).sum())
        worst = max(worst, float(np.max(err / tol)))
    print(f"{name}: {C_dev.numel()} outputs, {bad} outside the bound, max err/tol {worst:.4f}", flush=True)
    return bad


def main():
    assert torch.cuda.is_available()
    fails = 0
    d = inputs.llama_up_proj_backward()
    X, W, dY = d["X"], d["W"], d["dY"]
    qx, cx, sx, _ = quantized(X, "mxfp8_e4m3", "row")
    qw, cw, sw, _ = quantized(W, "mxfp8_e4m3", "row")
    fails += check("fwd Y = X W^T 8192x14336x4096", bsq.gemm(qx, qw, torch.bfloat16), cx, sx, "mxfp8_e4m3", None,
                   cw, sw, "mxfp8_e4m3", None)
    del qx, qw
    qdy, cdy, sdy, _ = quantized(dY, "mxfp8_e5m2", "row")
    qwc, cwc, swc, _ = quantized(W, "mxfp8_e4m3", "col")
    fails += check("dgrad dX = dY W 8192x4096x14336", bsq.gemm(qdy, qwc, torch.bfloat16), cdy, sdy, "mxfp8_e5m2", None,
                   cwc, swc, "mxfp8_e4m3", None)
    del qdy, qwc
    qdyc, cdyc, sdyc, _ = quantized(dY, "mxfp8_e5m2", "col")
    qxc, cxc, sxc, _ = quantized(X, "mxfp8_e4m3", "col")
    fails += check("wgrad dW = dY^T X 14336x4096x8192", bsq.gemm(qdyc, qxc, torch.bfloat16), cdyc, sdyc, "mxfp8_e5m2",
                   None, cxc, sxc, "mxfp8_e4m3", None)
    del qdyc, qxc, d, X, W, dY
    nv = inputs.nvfp4_forward()
    for xk, wk, name in (("X", "W", "nvfp4 Y = X W^T 8192x4096x4096"), ("X2", "W2", "nvfp4 Y' = X' W'^T 8192x4096x14336")):
        qa, ca, sa, ta = quantized(nv[xk], "nvfp4", "row")
        qb, cb, sb, tb = quantized(nv[wk], "nvfp4", "row")
        fails += check(name, bsq.gemm(qa, qb, torch.bfloat16), ca, sa, "nvfp4", ta, cb, sb, "nvfp4", tb)
    del nv
    m = inputs.moe_grouped()
    A, Wm, off = m["A"], m["W"].reshape(-1, 7168), m["offsets"]
    q4, c4, s4, _ = quantized(A, "mxfp4", "row")
    offd = torch.from_numpy(off).cuda()
    q8 = bsq.mxfp4_to_mxfp8_grouped(q4, offd, 64)
    c8, s8 = oracle.mxfp4_to_mxfp8_rows(c4, s4)
    assert np.array_equal(host_u8(q8.codes), c8.ravel())
    qwm, cwm, swm, _ = quantized(Wm, "mxfp8_e4m3", "row")
    Y = bsq.grouped_gemm(q8, offd, bsq.group_views(qwm, 64), torch.bfloat16, padded_scales=True)
    bad, total, worst = 0, 0, 0.0
    for g in range(64):
        lo, hi = int(off[g]), int(off[g + 1])
        Bd = oracle.dequant_rows(cwm[g * 2048:(g + 1) * 2048], swm[g * 2048:(g + 1) * 2048], "mxfp8_e4m3")
        Ad = oracle.dequant_rows(c8[lo:hi], s8[lo:hi], "mxfp8_e4m3")
        ref, mag = oracle.gemm_full_matmul(Ad, Bd)
        ok, err, tol = gemm_tol_ok(Y[lo:hi].float().cpu().numpy(), ref, mag, True)
        bad += int((~ok).sum())
        total += ok.size
        worst = max(worst, float(np.max(err / tol)))
    print(f"moe grouped 32768x2048x7168 (64 experts): {total} outputs, {bad} outside the bound, max err/tol {worst:.4f}",
          flush=True)
    fails += bad
    bsq.sync_status()
    print("full-output check:", "PASS" if fails == 0 else f"FAIL ({fails} outputs)")
    return 0 if fails == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
