#!/usr/bin/env python3
"""Benchmark of the block-scaled low-precision linear layer on GB300.

One step is one pass of the whole hot path over one synthetic batch, with
every input resident in HBM when the timed region starts:

  forward  (Llama-3-8B MLP up-projection, MXFP8 E4M3)
      quantize X[8192,4096] and W[14336,4096] both ways in one read each
      (rows for the forward, columns kept for the backward); Y = X W^T
      (BF16 out)
  backward (MXFP8, gradients E5M2)
      quantize dY[8192,14336] both (row + column);
      dX = dY W (8192x4096, K=14336); dW = dY^T X (14336x4096, K=8192)
  NVFP4 forward
      quantize X[8192,4096], W[4096,4096], X'[8192,14336], W'[4096,14336]
      (tensor amax + 16-block quantize); Y = X W^T, Y' = X' W'^T
  MoE grouped (64 experts, 32768 rows, Zipf(1.1) counts, K=7168, N=2048)
      quantize activations to MXFP4, re-encode MXFP4 -> MXFP8, quantize the
      expert weights to E4M3, grouped GEMM (BF16 out)

value = block-scaled GEMM FLOPs of the step / device time of the whole step
(quantize + re-encode + GEMMs), TFLOP/s; the timed steps replay CUDA graphs
of the step.  The dominant kernel (the forward FP8 GEMM) is timed with CUDA
events inside the timed region for the roofline; the per-op table comes from
a separate op-by-op pass with an event pair per op; both are reported
against the measured peaks.  e2e repeats the step through the same C ABI with the BF16
inputs copied from pinned host memory and the outputs read back, every step.

Run: python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Under torchrun each rank runs its own replica of the step (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantize GB/s vs HBM peak; block-scaled GEMM TFLOP/s vs dense FP8/FP4 peak"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--small", action="store_true", help="1/8-size shapes (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed steps op by op on the stream instead of replaying CUDA graphs")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-reps", type=int, default=12)
    ap.add_argument("--part", default="all", choices=["all", "fwd", "bwd", "nv", "moe"],
                    help="run one part of the step only (profiling)")
    ap.add_argument("--cpu-leg", default="", choices=["", "rows", "gemm"],
                    help=argparse.SUPPRESS)      # internal: the CPU baseline, run in its own process
    return ap.parse_args()


def peaks():
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        p.update({k: float(m[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")})
        p["source"] = "measured"
    except Exception:
        pass
    # nominal dense rates: BF16 2.25, FP8 4.5, FP4 13.5 PFLOP/s -> FP8 = 2x, FP4 = 6x the BF16 rate
    p["fp8_tflops"] = 2 * p["bf16_tflops"]
    p["fp4_tflops"] = 6 * p["bf16_tflops"]
    return p


# ----------------------------------------------------------------- shapes
def shapes(small: bool):
    d = 8 if small else 1
    return {
        "fwd": dict(M=8192 // d, N=14336 // d, K=4096),
        "nv": dict(M=8192 // d, N=4096 // d, K=4096, K2=14336),
        "moe": dict(rows=32768 // d, experts=64, K=7168, N=2048 // d if small else 2048),
    }


def make_inputs(sh, part="all"):
    from block_scaled_precision_03_gb300 import inputs
    f, n, m = sh["fwd"], sh["nv"], sh["moe"]
    h = {}
    if part in ("all", "fwd", "bwd"):
        h["X"] = inputs.outlier_activations_bf16((f["M"], f["K"]), 0)
        h["W"] = inputs.normal_bf16((f["N"], f["K"]), 1, std=0.02)
    if part in ("all", "bwd"):
        h["dY"] = inputs.loguniform_grad_bf16((f["M"], f["N"]), 2)
    if part in ("all", "nv"):
        nv = inputs.nvfp4_forward(n["M"], n["N"], n["K"], n["K2"], seed=10)
        h.update({"X4": nv["X"], "W4": nv["W"], "X42": nv["X2"], "W42": nv["W2"]})
    if part in ("all", "moe"):
        moe = inputs.moe_grouped(m["rows"], m["experts"], m["K"], m["N"], seed=20)
        h.update({"A_moe": moe["A"], "W_moe": moe["W"].reshape(-1, m["K"]), "offsets": moe["offsets"],
                  "counts": moe["counts"]})
    return h


# ------------------------------------------------------------- GPU step
class Step:
    """Device buffers and the ordered list of C-ABI calls of one step."""

    def __init__(self, host, sh, part="all"):
        import numpy as np
        import torch
        import block_scaled_precision_03_gb300 as bsq
        self.bsq, self.torch, self.sh = bsq, torch, sh
        bsq.lib()

        def dev(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

        self.host = host
        self.inp = {k: dev(host[k]) for k in ("X", "W", "dY", "X4", "W4", "X42", "W42", "A_moe", "W_moe")
                    if k in host}
        self.offsets = torch.from_numpy(host["offsets"]).cuda() if "offsets" in host else None
        self.moe_counts = np.diff(host["offsets"]).tolist() if "offsets" in host else None
        self.moe_kn = (sh["moe"]["K"], sh["moe"]["N"])
        want = {"all": ("fwd", "bwd", "nv", "moe")}.get(part, (part,))
        f, n, m = sh["fwd"], sh["nv"], sh["moe"]
        M, N, K = f["M"], f["N"], f["K"]
        E = bsq.empty
        o = {}
        if "fwd" in want or "bwd" in want:
            o["Xq"] = E("mxfp8_e4m3", M, K)
            o["Wq"] = E("mxfp8_e4m3", N, K)
            o["Wc"] = E("mxfp8_e4m3", K, N)
            o["Xc"] = E("mxfp8_e4m3", K, M)
            o["Y"] = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        if "bwd" in want:
            o["dYr"] = E("mxfp8_e5m2", M, N)
            o["dYc"] = E("mxfp8_e5m2", N, M)
            o["dX"] = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
            o["dW"] = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
        if "nv" in want:
            o["X4q"] = E("nvfp4", n["M"], n["K"])
            o["W4q"] = E("nvfp4", n["N"], n["K"])
            o["X42q"] = E("nvfp4", n["M"], n["K2"])
            o["W42q"] = E("nvfp4", n["N"], n["K2"])
            o["Y4"] = torch.empty((n["M"], n["N"]), dtype=torch.bfloat16, device="cuda")
            o["Y42"] = torch.empty((n["M"], n["N"]), dtype=torch.bfloat16, device="cuda")
        if "moe" in want:
            o["A4"] = E("mxfp4", m["rows"], m["K"])
            # the re-encoded activations carry their scales in the per-expert
            # padded layout, so the grouped GEMM's tiles start at expert boundaries
            o["A8"] = bsq.empty_grouped("mxfp8_e4m3", m["rows"], m["K"], m["experts"])
            o["Wm"] = E("mxfp8_e4m3", m["experts"] * m["N"], m["K"])
            o["Ym"] = torch.empty((m["rows"], m["N"]), dtype=torch.bfloat16, device="cuda")
        self.out = o
        self.wm_groups = bsq.group_views(o["Wm"], m["experts"]) if "moe" in want else None
        i = self.inp
        q = bsq.quantize_into
        # (name, row, kind, fn, bytes, flops, kernels)
        B_ROW8, B_ROW4, B_BOTH, B_NV, B_REPACK = 2 + 1 + 1 / 32, 2 + 0.5 + 1 / 32, 2 + 2 * (1 + 1 / 32), \
            2 + 2 + 0.5 + 1 / 16, 0.5 + 1 / 32 + 1 + 1 / 32
        mn = m["rows"] * m["K"]
        # X and W are quantized once, both ways: the rows feed the forward GEMM,
        # the columns (the transposed operands) the dgrad and wgrad GEMMs
        ops = [
            ("quant X e4m3 both", "a2", "quant", lambda: q(i["X"], "mxfp8_e4m3", "both", o["Xq"], o["Xc"]), M * K * B_BOTH, 0, 1),
            ("quant W e4m3 both", "a2", "quant", lambda: q(i["W"], "mxfp8_e4m3", "both", o["Wq"], o["Wc"]), N * K * B_BOTH, 0, 1),
            ("gemm fwd Y=XW^T", "a4", "gemm8", lambda: bsq.gemm_into(o["Xq"], o["Wq"], o["Y"]), 0, 2 * M * N * K, 1),
            ("quant dY e5m2 both", "a2", "quant", lambda: q(i["dY"], "mxfp8_e5m2", "both", o["dYr"], o["dYc"]), M * N * B_BOTH, 0, 1),
            ("gemm dgrad dX=dY W", "a4", "gemm8", lambda: bsq.gemm_into(o["dYr"], o["Wc"], o["dX"]), 0, 2 * M * K * N, 1),
            ("gemm wgrad dW=dY^T X", "a4", "gemm8", lambda: bsq.gemm_into(o["dYc"], o["Xc"], o["dW"]), 0, 2 * N * K * M, 1),
            ("quant X nvfp4", "a3", "quant", lambda: q(i["X4"], "nvfp4", "row", o["X4q"], None), n["M"] * n["K"] * B_NV, 0, 2),
            ("quant W nvfp4", "a3", "quant", lambda: q(i["W4"], "nvfp4", "row", o["W4q"], None), n["N"] * n["K"] * B_NV, 0, 2),
            ("quant X' nvfp4", "a3", "quant", lambda: q(i["X42"], "nvfp4", "row", o["X42q"], None), n["M"] * n["K2"] * B_NV, 0, 2),
            ("quant W' nvfp4", "a3", "quant", lambda: q(i["W42"], "nvfp4", "row", o["W42q"], None), n["N"] * n["K2"] * B_NV, 0, 2),
            ("gemm nvfp4 Y=XW^T", "a4", "gemm4", lambda: bsq.gemm_into(o["X4q"], o["W4q"], o["Y4"]), 0, 2 * n["M"] * n["N"] * n["K"], 1),
            ("gemm nvfp4 Y'=X'W'^T", "a4", "gemm4", lambda: bsq.gemm_into(o["X42q"], o["W42q"], o["Y42"]), 0, 2 * n["M"] * n["N"] * n["K2"], 1),
            ("quant A_moe mxfp4 row", "a1", "quant", lambda: q(i["A_moe"], "mxfp4", "row", o["A4"], None), mn * B_ROW4, 0, 1),
            ("repack mxfp4->mxfp8", "a5", "repack",
             lambda: bsq.mxfp4_to_mxfp8_grouped_into(o["A4"], o["A8"], self.offsets, m["experts"]), mn * B_REPACK, 0, 1),
            ("quant W_moe e4m3 row", "a1", "quant", lambda: q(i["W_moe"], "mxfp8_e4m3", "row", o["Wm"], None),
             m["experts"] * m["N"] * m["K"] * B_ROW8, 0, 1),
            ("grouped gemm moe", "a6", "gemm8", lambda: bsq.grouped_gemm_into(o["A8"], self.offsets, self.wm_groups, o["Ym"],
                                                                               padded_scales=True),
             0, 2 * m["rows"] * m["N"] * m["K"], 1),
        ]
        part_of = ["fwd"] * 3 + ["bwd"] * 3 + ["nv"] * 6 + ["moe"] * 4
        if part == "bwd":
            want = ("fwd", "bwd")      # the backward quantizes from the forward inputs
        ops = [op for op, pt in zip(ops, part_of) if pt in want]
        self.ops = ops
        # Rows beyond the core path, timed on their own after the step (not
        # part of the step's time or FLOPs).  NEXT-3: NVFP4 with delayed
        # scaling, one pass (2.5625 B per element), the amax history holding
        # the tensor's own amax as in steady state.
        self.extra_ops = []
        if "fwd" in want:
            # the same quantizes one layout at a time (rows a1 and a2 on X and W;
            # the outputs are the step's own, rewritten with the same bytes)
            self.extra_ops += [
                ("quant X e4m3 row", "a1", "quant", lambda: q(i["X"], "mxfp8_e4m3", "row", o["Xq"], None), M * K * B_ROW8, 0, 1),
                ("quant W e4m3 row", "a1", "quant", lambda: q(i["W"], "mxfp8_e4m3", "row", o["Wq"], None), N * K * B_ROW8, 0, 1),
                ("quant X e4m3 col", "a2", "quant", lambda: q(i["X"], "mxfp8_e4m3", "col", None, o["Xc"]), M * K * B_ROW8, 0, 1),
                ("quant W e4m3 col", "a2", "quant", lambda: q(i["W"], "mxfp8_e4m3", "col", None, o["Wc"]), N * K * B_ROW8, 0, 1),
            ]
            # NEXT-4, dense: the forward GEMM on MXFP4 x MXFP4 operands
            # (quantized once here; the timed op is the GEMM alone)
            o["Xq4"] = E("mxfp4", M, K)
            o["Wq4"] = E("mxfp4", N, K)
            q(i["X"], "mxfp4", "row", o["Xq4"], None)
            q(i["W"], "mxfp4", "row", o["Wq4"], None)
            self.extra_ops.append(("gemm fwd mxfp4 Y=XW^T", "NEXT-4", "gemm4",
                                   lambda: bsq.gemm_into(o["Xq4"], o["Wq4"], o["Y"]), 0, 2 * M * N * K, 1))
        if "moe" in want:
            # NEXT-1: FP4RowToFP8Col of the MoE activations (the wgrad operand),
            # from the MXFP4 rows the step produced; read 0.53125 + write 1.03125 B
            o["A8c"] = E("mxfp8_e4m3", m["K"], m["rows"])
            self.extra_ops.append(("fp4row->fp8col A_moe", "NEXT-1", "repack",
                                   lambda: bsq.mxfp4_to_mxfp8_col_into(o["A4"], o["A8c"]), mn * B_REPACK, 0, 1))
            # NEXT-2: MXFP4 -> FP8 E4M3 with 1x128 blocks (the Hopper FP8 block) of
            # the MoE activations; read 0.53125 + write 1 + 1/128 B per element
            o["A8h"] = torch.empty((m["rows"], m["K"]), dtype=torch.uint8, device="cuda")
            o["A8hs"] = torch.empty((m["rows"], (m["K"] + 127) // 128), dtype=torch.uint8, device="cuda")
            self.extra_ops.append(("mxfp4->fp8 1x128 A_moe", "NEXT-2", "repack",
                                   lambda: bsq.mxfp4_to_fp8_1x128_into(o["A4"], o["A8h"], o["A8hs"]),
                                   mn * (0.5 + 1 / 32 + 1 + 1 / 128), 0, 1))
            # NEXT-4: the MoE GEMM on MXFP4 x MXFP4 natively (weights quantized to
            # MXFP4 as well), against the step's repack + MXFP8 grouped GEMM
            o["Wm4"] = E("mxfp4", m["experts"] * m["N"], m["K"])
            o["Ym4"] = torch.empty((m["rows"], m["N"]), dtype=torch.bfloat16, device="cuda")
            self.wm4_groups = bsq.group_views(o["Wm4"], m["experts"])
            self.extra_ops += [
                ("quant W_moe mxfp4 row", "NEXT-4", "quant", lambda: q(i["W_moe"], "mxfp4", "row", o["Wm4"], None),
                 m["experts"] * m["N"] * m["K"] * B_ROW4, 0, 1),
                ("grouped gemm moe mxfp4", "NEXT-4", "gemm4", lambda: bsq.grouped_gemm_into(o["A4"], self.offsets,
                                                                                           self.wm4_groups, o["Ym4"]),
                 0, 2 * m["rows"] * m["N"] * m["K"], 1),
            ]
        if "nv" in want:
            B_NV1 = 2 + 0.5 + 1 / 16
            qd = bsq.quantize_nvfp4_delayed_into
            self.hist = {}
            for k in ("X4", "W4", "X42", "W42"):
                f = (np.asarray(host[k], np.uint32) << 16).view(np.float32)
                h = torch.zeros(16, dtype=torch.float32, device="cuda")
                h[0] = float(np.abs(f[np.isfinite(f)]).max())
                self.hist[k] = h
            o["X4d"] = E("nvfp4", n["M"], n["K"])
            o["W4d"] = E("nvfp4", n["N"], n["K"])
            o["X42d"] = E("nvfp4", n["M"], n["K2"])
            o["W42d"] = E("nvfp4", n["N"], n["K2"])
            hs = self.hist
            self.extra_ops += [
                ("quant X nvfp4 delayed", "NEXT-3", "quant", lambda: qd(i["X4"], "row", o["X4d"], None, hs["X4"]),
                 n["M"] * n["K"] * B_NV1, 0, 2),
                ("quant W nvfp4 delayed", "NEXT-3", "quant", lambda: qd(i["W4"], "row", o["W4d"], None, hs["W4"]),
                 n["N"] * n["K"] * B_NV1, 0, 2),
                ("quant X' nvfp4 delayed", "NEXT-3", "quant", lambda: qd(i["X42"], "row", o["X42d"], None, hs["X42"]),
                 n["M"] * n["K2"] * B_NV1, 0, 2),
                ("quant W' nvfp4 delayed", "NEXT-3", "quant", lambda: qd(i["W42"], "row", o["W42d"], None, hs["W42"]),
                 n["N"] * n["K2"] * B_NV1, 0, 2),
            ]
        self.flops = sum(op[5] for op in ops)
        self.kernels = sum(op[6] for op in ops)

    def run(self, events=None):
        for j, op in enumerate(self.ops):
            if events is not None:
                events[j][0].record()
            op[3]()
            if events is not None:
                events[j][1].record()

    # Independent quantizes that run side by side: op -> (side stream, the op
    # it starts beside, the op that waits for it).  Each side op goes to its
    # side stream when the main stream reaches its partner, and the op that
    # reads its output waits for that stream; the GEMMs themselves run alone.
    # The four NVFP4 quantizes run at once: X on the main stream, W then W' on
    # side stream 0, X' on side stream 1.
    SIDE = {"quant W e4m3 both": (0, "quant X e4m3 both", "gemm fwd Y=XW^T"),
            "quant W nvfp4": (0, "quant X nvfp4", "gemm nvfp4 Y=XW^T"),
            "quant X' nvfp4": (1, "quant X nvfp4", "gemm nvfp4 Y'=X'W'^T"),
            "quant W' nvfp4": (0, "quant X nvfp4", "gemm nvfp4 Y'=X'W'^T"),
            "quant W_moe e4m3 row": (0, "quant A_moe mxfp4 row", "grouped gemm moe")}

    def run_overlapped(self, timed=None, jr=None):
        """The step with the SIDE quantizes on side streams (the timed steps);
        `timed`: an event pair recorded around op `jr`."""
        torch = self.torch
        if not hasattr(self, "side_streams"):
            self.side_streams = [torch.cuda.Stream() for _ in range(2)]
        cur = torch.cuda.current_stream()
        by_name = {op[0]: j for j, op in enumerate(self.ops)}
        starts, joins = {}, {}
        for side, (lane, partner, reader) in self.SIDE.items():
            if side in by_name and partner in by_name and reader in by_name:
                starts.setdefault(partner, []).append((lane, side))
                joins.setdefault(reader, set()).add(lane)
        moved = {side for sides in starts.values() for _, side in sides}
        used = set()
        for j, op in enumerate(self.ops):
            name = op[0]
            if name in moved:
                continue
            for lane in sorted(joins.get(name, ())):
                cur.wait_stream(self.side_streams[lane])
            for lane, side in starts.get(name, ()):
                used.add(lane)
                self.side_streams[lane].wait_stream(cur)
                with torch.cuda.stream(self.side_streams[lane]):
                    self.ops[by_name[side]][3]()
            if j == jr and timed is not None:
                timed[0].record()
            op[3]()
            if j == jr and timed is not None:
                timed[1].record()
        # (a stream that took no work here must not be joined inside a capture)
        for lane in sorted(used):
            cur.wait_stream(self.side_streams[lane])

    # e2e: host (pinned) -> device copies of every BF16 input, the step, and a
    # device -> host read of every output, all inside the timed region.  The
    # host link (about 210 GB/s in, 190 GB/s out on this machine, the same for
    # copy engines and for SM loads of pinned memory) bounds this number, so
    # the copies are pipelined: inputs go up on one copy stream in the order
    # the ops need them, each op waits only for its own inputs, and each
    # output goes down on a second copy stream as soon as its GEMM finished.
    NEEDS = {"quant X e4m3 both": ("X",), "quant W e4m3 both": ("W",), "quant dY e5m2 both": ("dY",),
             "quant X nvfp4": ("X4",),
             "quant W nvfp4": ("W4",), "quant X' nvfp4": ("X42",), "quant W' nvfp4": ("W42",),
             "quant A_moe mxfp4 row": ("A_moe",), "quant W_moe e4m3 row": ("W_moe",),
             "repack mxfp4->mxfp8": ("offsets",), "grouped gemm moe": ("offsets",)}
    PRODUCES = {"gemm fwd Y=XW^T": "Y", "gemm dgrad dX=dY W": "dX", "gemm wgrad dW=dY^T X": "dW",
                "gemm nvfp4 Y=XW^T": "Y4", "gemm nvfp4 Y'=X'W'^T": "Y42", "grouped gemm moe": "Ym"}

    # e2e op order: the host link bounds the pass (3.2 GB up), so the inputs
    # go up largest-consumer first and the step ends soon after the last one
    # lands: the MoE part (2.35 GB of inputs) first, the 33.5 MB NVFP4 weight
    # and its GEMM last, the other NVFP4 GEMM just before, so that its output
    # goes down while the last two inputs come up.  Each op still waits only
    # for its own inputs.
    E2E_ORDER = ("quant A_moe mxfp4 row", "repack mxfp4->mxfp8", "quant W_moe e4m3 row", "grouped gemm moe",
                 "quant X e4m3 both", "quant W e4m3 both", "gemm fwd Y=XW^T", "quant dY e5m2 both",
                 "gemm dgrad dX=dY W", "gemm wgrad dW=dY^T X",
                 "quant X' nvfp4", "quant W' nvfp4", "gemm nvfp4 Y'=X'W'^T", "quant X nvfp4",
                 "quant W nvfp4", "gemm nvfp4 Y=XW^T")

    def setup_e2e(self):
        import numpy as np
        torch = self.torch
        self.pinned_in = {k: torch.from_numpy(np.ascontiguousarray(self.host[k]).view(np.int16))
                          .view(torch.bfloat16).pin_memory() for k in self.inp}
        outs = [k for k in ("Y", "dX", "dW", "Y4", "Y42", "Ym") if k in self.out]
        self.pinned_out = {k: torch.empty(self.out[k].shape, dtype=torch.bfloat16).pin_memory() for k in outs}
        self.pinned_offsets = None
        if getattr(self, "offsets", None) is not None:
            self.pinned_offsets = self.offsets.cpu().pin_memory()     # expert row offsets (int64)
        self.h2d = sum(t.numel() * 2 for t in self.pinned_in.values())
        self.h2d += 0 if self.pinned_offsets is None else self.pinned_offsets.numel() * 8
        self.d2h = sum(t.numel() * 2 for t in self.pinned_out.values())
        rank_of = {name: i for i, name in enumerate(self.E2E_ORDER)}
        self.e2e_ops = sorted(self.ops, key=lambda op: rank_of.get(op[0], len(rank_of)))
        # inputs in order of first use
        order = []
        for op in self.e2e_ops:
            for k in self.NEEDS.get(op[0], ()):
                if k in self.pinned_in and k not in order:
                    order.append(k)
        self.copy_order = order + [k for k in self.pinned_in if k not in order]
        self.h2d_stream = torch.cuda.Stream()
        self.d2h_stream = torch.cuda.Stream()

    def run_e2e(self):
        torch = self.torch
        cur = torch.cuda.current_stream()
        # the previous step's ops are done with the input buffers before new data lands
        self.h2d_stream.wait_stream(cur)
        ready = {}
        with torch.cuda.stream(self.h2d_stream):
            # the expert offsets (520 bytes) first: the re-encode and the grouped GEMM read them
            if self.pinned_offsets is not None:
                self.offsets.copy_(self.pinned_offsets, non_blocking=True)
                ready["offsets"] = torch.cuda.Event()
                ready["offsets"].record()
            for k in self.copy_order:
                self.inp[k].copy_(self.pinned_in[k], non_blocking=True)
                ready[k] = torch.cuda.Event()
                ready[k].record()
        for op in self.e2e_ops:
            for k in self.NEEDS.get(op[0], ()):
                if k in ready:
                    cur.wait_event(ready[k])
            op[3]()
            k = self.PRODUCES.get(op[0])
            if k in self.pinned_out:
                done = torch.cuda.Event()
                done.record(cur)
                self.d2h_stream.wait_event(done)
                with torch.cuda.stream(self.d2h_stream):
                    self.pinned_out[k].copy_(self.out[k], non_blocking=True)
        # the step ends when every output is in host memory
        cur.wait_stream(self.d2h_stream)


# ------------------------------------------------------------- clocks
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        mx = max(float(r[2]) for r in rows)
        load = [s for s, r in zip(sm, rows) if float(r[3]) > 300.0] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- CPU oracle
def cpu_forward_slice(host, rows=64, wrows=2048):
    """The oracle's forward on a slice: quantize X[:rows] and W[:wrows] (E4M3),
    dequantize, FP64 GEMM.  Returns (seconds, flops)."""
    import oracle
    X, W = host["X"][:rows], host["W"][:wrows]
    t0 = time.perf_counter()
    cx, sx = oracle.mx_quantize_rows(X, "mxfp8_e4m3")
    cw, sw = oracle.mx_quantize_rows(W, "mxfp8_e4m3")
    A = oracle.dequant_rows(cx, sx, "mxfp8_e4m3")
    B = oracle.dequant_rows(cw, sw, "mxfp8_e4m3")
    oracle.gemm_full(A, B)
    return time.perf_counter() - t0, 2.0 * rows * wrows * X.shape[1]


# Rows of the step timed on the oracle, single-threaded, on a bounded sample:
# (name, sample rows, row length, algorithmic bytes per element) -- the bytes
# are the same per-element figures the GPU rows use.
CPU_ROWS = (("quant X e4m3 row", 512, 4096, 2 + 1 + 1 / 32),
            ("quant X nvfp4", 512, 4096, 2 + 2 + 0.5 + 1 / 16),
            ("quant A_moe mxfp4 row", 256, 7168, 2 + 0.5 + 1 / 32),
            ("repack mxfp4->mxfp8", 256, 7168, 0.5 + 1 / 32 + 1 + 1 / 32))


def cpu_rows_leg(min_seconds=2.0):
    """The oracle's quantize and re-encode on a bounded sample of each row's
    tensor (same distribution and row length), GB/s of algorithmic bytes.
    Runs in its own process with OMP_NUM_THREADS=1."""
    import oracle
    from block_scaled_precision_03_gb300 import inputs
    out = {}
    for name, rows, cols, bpe in CPU_ROWS:
        if name == "quant X e4m3 row":
            x = inputs.outlier_activations_bf16((rows, cols), 0)
            fn = lambda: oracle.mx_quantize_rows(x, "mxfp8_e4m3")
        elif name == "quant X nvfp4":
            x = inputs.normal_bf16((rows, cols), 10)
            fn = lambda: oracle.nvfp4_quantize_rows(x)          # tensor amax, then the blocks
        elif name == "quant A_moe mxfp4 row":
            x = inputs.normal_bf16((rows, cols), 21)
            fn = lambda: oracle.mx_quantize_rows(x, "mxfp4")
        else:
            c4, s4 = oracle.mx_quantize_rows(inputs.normal_bf16((rows, cols), 21), "mxfp4")
            fn = lambda: oracle.mxfp4_to_mxfp8_rows(c4, s4)
        fn()
        n, t0 = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            dt = time.perf_counter() - t0
            if dt >= min_seconds:
                break
        out[name] = {"gbs": round(rows * cols * bpe * n / dt / 1e9, 4), "threads": 1,
                     "sample": f"{rows}x{cols} of the same distribution", "seconds": round(dt, 2)}
    return out


def cpu_gemm_leg(reps):
    from block_scaled_precision_03_gb300 import inputs
    host = {"X": inputs.outlier_activations_bf16((CPU_ROWS_X, 4096), 0),
            "W": inputs.normal_bf16((2048, 4096), 1, std=0.02)}
    ts = [cpu_forward_slice(host, CPU_ROWS_X) for _ in range(max(1, reps))]
    t_tot = sum(t for t, _ in ts)
    return {"value": ts[0][1] * len(ts) / t_tot / 1e12, "seconds": round(t_tot, 2)}


def run_cpu_leg(leg, reps, threads=None):
    """One CPU-baseline leg in a child process (the GPU process never loads
    the oracle); returns its JSON result or None."""
    env = dict(os.environ)
    if threads is not None:
        env["OMP_NUM_THREADS"] = str(threads)
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-leg", leg, "--cpu-reps", str(reps)],
                           env=env, capture_output=True, text=True, timeout=600)
        for line in r.stdout.splitlines()[::-1]:
            if line.startswith("{"):
                return json.loads(line)
    except Exception:
        pass
    return None


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_sample(rows, wrows):
    return (f"oracle forward slice: E4M3 quantize of X[:{rows},4096] and W[:{wrows},4096], exact dequantize, "
            f"FP64 GEMM {rows}x{wrows}x4096")


CPU_ROWS_X = 512
CPU_SAMPLE = cpu_sample(CPU_ROWS_X, 2048)
REF_ROWS, REF_WROWS = 64, 256      # one reference-arm step: a bounded slice (~0.1 s of CPU work)


def workload_config(args, world):
    return {"workload": "llama3-8b block-scaled linear layer step: MXFP8 fwd 8192x14336x4096 + "
                        "MXFP8 bwd (dgrad, wgrad) + NVFP4 fwd (4096/14336) + MoE 64-expert grouped "
                        "(MXFP4 -> MXFP8 repack, 32768x2048x7168)" + (" [1/8 size]" if args.small else "")
                        + ("" if args.part == "all" else f" [part {args.part}]"),
            "parallelism": f"replica x{world}",
            "l2": "inputs larger than L2: each step streams ~9 GB, evicting the previous step's data",
            "value_def": "GEMM FLOPs / whole-step device time"}


# ------------------------------------------------------------------ main
def dist_setup(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def attainable(step, ms, pk, fp4):
    """Attainable time of the grouped MoE GEMM: per expert the larger of its
    compute time at the tensor peak (FP8, or FP4 for MXFP4 operands) and the
    time to stream its weights, activations (codes and E8M0 scales per 32)
    and BF16 output at the HBM rate; small experts are bound by their
    weights."""
    K_, N_ = step.moe_kn
    code = 0.5 if fp4 else 1.0
    peak = pk["fp4_tflops"] if fp4 else pk["fp8_tflops"]
    t_bound = 0.0
    for cnt in step.moe_counts:
        fl = 2.0 * cnt * N_ * K_
        by = N_ * K_ * (code + 1 / 32) + cnt * K_ * (code + 1 / 32) + cnt * N_ * 2
        t_bound += max(fl / (peak * 1e12), by / (pk["hbm_gbs"] * 1e9))
    return {"attainable_ms": round(t_bound * 1e3, 4), "frac_attainable": round(t_bound * 1e3 / ms, 4)}


def reduce_max(x: float, device="cpu") -> float:
    """Max of x over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores: each step is the
    bounded forward slice of the same workload."""
    if rank != 0:
        return
    sh = shapes(args.small)
    from block_scaled_precision_03_gb300 import inputs
    f = sh["fwd"]
    host = {"X": inputs.outlier_activations_bf16((REF_ROWS, f["K"]), 0),
            "W": inputs.normal_bf16((REF_WROWS, f["K"]), 1, std=0.02)}
    for _ in range(args.warmup):
        cpu_forward_slice(host, REF_ROWS, REF_WROWS)
    ts, fl = [], 0.0
    for _ in range(args.steps):
        t, fl = cpu_forward_slice(host, REF_ROWS, REF_WROWS)
        ts.append(t)
    total = sum(ts)
    value = fl * args.steps / total / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args, world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": cpu_sample(REF_ROWS, REF_WROWS) + " per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.cpu_leg:
        res = cpu_rows_leg() if args.cpu_leg == "rows" else cpu_gemm_leg(args.cpu_reps)
        print(json.dumps(res), flush=True)
        return
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    import torch.distributed as dist
    assert torch.cuda.is_available(), "bench needs a CUDA device"
    torch.cuda.set_device(local)
    pk = peaks()
    sh = shapes(args.small)
    host = make_inputs(sh, args.part)
    step = Step(host, sh, args.part)
    nops = len(step.ops)

    def barrier():
        if world > 1:
            dist.barrier()

    # The roofline kernel: the forward FP8 GEMM (2*M*N*K FLOPs per launch over
    # its average event time), else the first GEMM of the step.
    fwd = next((j for j, op in enumerate(step.ops) if op[0].startswith("gemm fwd")), None)
    jr = fwd if fwd is not None else next((j for j, op in enumerate(step.ops) if op[2] == "gemm8"),
                                          next((j for j, op in enumerate(step.ops) if op[5]), 0))

    # The timed steps replay CUDA graphs of the step (one launch per graph
    # instead of one per kernel): graphs of G = min(10, K) steps, replayed
    # K // G times, and one of a single step for the K % G left over and the
    # warm-up.  Only the last G timed steps carry event pairs, on the roofline
    # kernel (external event nodes, which can be read after the replay, but
    # cost ~8 us each inside a graph); an event pair per op costs ~70 us of a
    # 2.4 ms step, so the per-op table comes from a separate pass after the
    # timed region.  --no-graph (or a
    # PyTorch without external events) launches the timed steps op by op,
    # with the same single event pair per step.
    def run_timed(pair):
        step.run_overlapped(pair, jr)

    launch_mode = "stream, op by op"
    graphs = None
    step.run()                 # first calls outside any capture (lazy set-up in the library)
    torch.cuda.synchronize()
    if not args.no_graph and args.steps > 0:
        try:
            G = min(10, args.steps)
            evG = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)] for _ in range(G)]
            gG, gP, g1 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            # thread-local capture: other threads of the process (NCCL's watchdog
            # under torchrun) may keep making CUDA calls meanwhile
            with torch.cuda.graph(gG, capture_error_mode="thread_local"):
                for s_ in range(G):
                    run_timed(evG[s_])
            with torch.cuda.graph(gP, capture_error_mode="thread_local"):
                for s_ in range(G):
                    step.run_overlapped()
            with torch.cuda.graph(g1, capture_error_mode="thread_local"):
                step.run_overlapped()
            torch.cuda.synchronize()
            graphs = (G, gG, gP, g1, evG)
            launch_mode = f"CUDA graph replay ({G} steps per graph)"
        except (TypeError, RuntimeError) as exc:
            print(f"[bench] CUDA graph capture unavailable ({exc}); launching op by op", file=sys.stderr)
            graphs = None
            torch.cuda.synchronize()
    for _ in range(max(args.warmup, 0) - 1):
        if graphs is not None:
            graphs[3].replay()
        else:
            step.run()
    torch.cuda.synchronize()

    # ---- timed region: K steps
    evK = None
    if graphs is None:
        evK = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local)
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    start.record()
    if graphs is not None:
        # the last G timed steps carry the roofline kernel's event nodes
        G, gG, gP, g1, evG = graphs
        for _ in range(args.steps % G):
            g1.replay()
        for _ in range(args.steps // G - 1):
            gP.replay()
        gG.replay()
    else:
        for s_ in range(args.steps):
            run_timed(evK[s_])
    stop.record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    elapsed_ms = reduce_max(start.elapsed_time(stop), "cuda")
    ms_step = elapsed_ms / args.steps
    value = world * step.flops / (ms_step * 1e-3) / 1e12
    timed_pairs = graphs[4] if graphs is not None else evK
    roof_ms = statistics.mean(a.elapsed_time(b) for a, b in timed_pairs)

    # ---- per-op table: a separate pass after the timed region, op by op
    # with an event pair per op
    nrows = max(1, min(args.steps, 100))
    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(nops)]
          for _ in range(nrows)]
    torch.cuda.synchronize()
    for s_ in range(nrows):
        step.run(ev[s_])
    torch.cuda.synchronize()
    op_ms = [statistics.mean(ev[s_][j][0].elapsed_time(ev[s_][j][1]) for s_ in range(nrows)) for j in range(nops)]
    rows, agg = {}, {}
    for (name, row, kind, _, nbytes, flops, nk), ms in zip(step.ops, op_ms):
        if flops:
            peak = pk["fp4_tflops"] if kind == "gemm4" else pk["fp8_tflops"]
            ach = flops / (ms * 1e-3) / 1e12
            rec = {"ms": round(ms, 4), "tflops": round(ach, 1), "frac": round(ach / peak, 4)}
        else:
            ach = nbytes / (ms * 1e-3) / 1e9
            rec = {"ms": round(ms, 4), "gbs": round(ach, 1), "frac": round(ach / pk["hbm_gbs"], 4),
                   "frac_spec_8tbs": round(ach / 8000.0, 4)}
        if kind == "quant" and row == "a3":
            # the NVFP4 bytes above count the amax pass; also the one-read minimum
            one = nbytes * (2 + 0.5 + 1 / 16) / (2 + 2 + 0.5 + 1 / 16)
            rec["frac_one_read"] = round(one / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)
        if name == "grouped gemm moe" and step.moe_counts is not None:
            rec.update(attainable(step, ms, pk, fp4=False))
        rows[name] = dict(row=row, **rec)
        a = agg.setdefault(kind, [0.0, 0.0, 0.0])
        a[0] += ms
        a[1] += nbytes
        a[2] += flops
    for kind in ("quant", "repack", "gemm8", "gemm4"):
        agg.setdefault(kind, [1e-30, 0.0, 0.0])

    # rows beyond the core path: each timed alone, cycling through all of
    # them so that every input has left L2 before it is read again
    rows_next = {}
    if step.extra_ops:
        reps = 20
        for _ in range(3):
            for op in step.extra_ops:
                op[3]()
        xev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in step.extra_ops] for _ in range(reps)]
        torch.cuda.synchronize()
        for r in range(reps):
            for j, op in enumerate(step.extra_ops):
                xev[r][j][0].record()
                op[3]()
                xev[r][j][1].record()
        torch.cuda.synchronize()
        for j, (name, row, kind, _, nbytes, flops, nk) in enumerate(step.extra_ops):
            ms = statistics.mean(xev[r][j][0].elapsed_time(xev[r][j][1]) for r in range(reps))
            if flops:
                ach = flops / (ms * 1e-3) / 1e12
                peak = pk["fp4_tflops"] if kind == "gemm4" else pk["fp8_tflops"]
                rows_next[name] = {"row": row, "ms": round(ms, 4), "tflops": round(ach, 1), "frac": round(ach / peak, 4)}
                if name == "grouped gemm moe mxfp4" and step.moe_counts is not None:
                    rows_next[name].update(attainable(step, ms, pk, fp4=True))
            else:
                ach = nbytes / (ms * 1e-3) / 1e9
                rows_next[name] = {"row": row, "ms": round(ms, 4), "gbs": round(ach, 1),
                                   "frac": round(ach / pk["hbm_gbs"], 4), "frac_spec_8tbs": round(ach / 8000.0, 4)}
    q_ms, q_bytes = agg["quant"][0] + agg["repack"][0], agg["quant"][1] + agg["repack"][1]
    g8_ms, g8_fl = agg["gemm8"][0], agg["gemm8"][2]
    g4_ms, g4_fl = agg["gemm4"][0], agg["gemm4"][2]
    g8 = g8_fl / (g8_ms * 1e-3) / 1e12
    # roofline of the dominant kernel (FP8 GEMM), taken on its largest launch
    # inside the timed region
    ach = step.ops[jr][5] / (roof_ms * 1e-3) / 1e12
    fp4_gemm = step.ops[jr][2] == "gemm4"
    rpeak = pk["fp4_tflops"] if fp4_gemm else pk["fp8_tflops"]
    roofline = {"bound": "tensor", "achieved": round(ach, 1), "peak": rpeak, "unit": "TFLOP/s",
                "frac": round(ach / rpeak, 4), "traffic": None,
                "kernel": ("gemm2_kernel<nvfp4> (CTA pair, tcgen05 mxf4nvf4 block_scale)" if fp4_gemm else
                           "gemm2_kernel<fp8> (CTA pair, tcgen05 mxf8f6f4 block_scale)") + ", launch: " + step.ops[jr][0],
                "flops_per_launch": step.ops[jr][5], "ms_per_launch": round(roof_ms, 4),
                "peak_note": f"{'6' if fp4_gemm else '2'}x {pk['source']} bf16 burst {pk['bf16_tflops']} TFLOP/s "
                             f"(nominal dense FP8 = 2x, FP4 = 6x the BF16 rate)",
                "frac_vs_sustained": round(ach / ((6 if fp4_gemm else 2) * pk["bf16_tflops_sustained"]), 4),
                "all_fp8_gemm_launches_tflops": round(g8, 1)}
    traffic = None if fp4_gemm else _profile_traffic()
    if traffic is not None:
        roofline["traffic"] = traffic

    # ---- e2e through the same C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        step.setup_e2e()
        step.run_e2e()
        torch.cuda.synchronize()
        ke = max(1, min(args.steps, 5))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        s0.record()
        for _ in range(ke):
            step.run_e2e()
        s1.record()
        torch.cuda.synchronize()
        barrier()
        e_ms = reduce_max(s0.elapsed_time(s1) / ke, "cuda")
        e2e = {"value": round(world * step.flops / (e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(e_ms, 3), "steps": ke,
               "h2d_bytes_per_step": step.h2d, "d2h_bytes_per_step": step.d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        g = run_cpu_leg("gemm", args.cpu_reps)
        rows_cpu = run_cpu_leg("rows", 1, threads=1)
        if g is not None:
            cpu = {"value": g["value"], "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                   "sample": CPU_SAMPLE, "seconds": g["seconds"], "process": "child process (oracle not in the GPU process)",
                   "rows": rows_cpu, "rows_note": "single-threaded oracle quantize / re-encode, GB/s of the same "
                                                  "algorithmic bytes as the GPU rows"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3/e5m2/e2m1 codes, f32 accumulate", "data": "synthetic",
            "config": dict(workload_config(args, world), launch=launch_mode),
            "quantize_gbs": round(q_bytes / (q_ms * 1e-3) / 1e9, 1),
            "quantize_frac": round(q_bytes / (q_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "gemm_fp8_tflops": round(g8, 1), "gemm_nvfp4_tflops": round(g4_fl / (g4_ms * 1e-3) / 1e12, 1),
            "roofline": roofline, "rows": rows, "rows_next": rows_next, "gpu_launches": step.kernels * args.steps,
            "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
            "peaks": {k: pk[k] for k in ("hbm_gbs", "fp8_tflops", "fp4_tflops", "source")},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# sources the FP8 GEMM launch is built from; the profile that gives its DRAM
# traffic names their hash, taken with comments and blank space removed
KERNEL_SOURCES = ("gemm2.cu", "tcgen05.cuh", "epilogue.cuh", "common.cuh", "tmap.h")


def kernel_source_hash() -> str:
    """sha256[:16] of the GEMM sources with // and /* */ comments and all
    white space removed (comment edits leave it unchanged)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        src = open(os.path.join(ROOT, "block_scaled_precision_03_gb300", "csrc", name)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(re.sub(r"\s+", "", src).encode())
    return h.hexdigest()[:16]


def _profile_traffic():
    """DRAM bytes per launch of the FP8 GEMM from the committed ncu summary,
    only if that summary was taken on the current GEMM sources."""
    try:
        vals = {}
        with open(os.path.join(ROOT, "profiles", "gemm2_fp8_fwd_8192x14336x4096.md")) as f:
            for line in f:
                if ":" in line and line.startswith("- "):
                    k, v = line[2:].rsplit(":", 1)
                    vals[k.strip()] = v.strip().strip("`")
        if vals.get("kernel source sha256[:16]") != kernel_source_hash():
            return None
        return float(vals["dram bytes per full launch"])
    except Exception:
        return None


if __name__ == "__main__":
    main()
