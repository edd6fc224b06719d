"""The library's calls captured in a CUDA graph.

One sequence of calls covering every kind of work a step launches (MXFP8
quantize both ways, NVFP4 just-in-time quantize: the scale-slot memset, the
amax pass and the quantize kernel that runs as its programmatic dependent;
the FP8 and NVFP4 GEMMs; MXFP4 quantize, the grouped MXFP4 -> MXFP8 re-encode
with its padding memset and the grouped GEMM; NVFP4 delayed scaling, whose
history update runs as the pass's programmatic dependent) is launched once on
the stream and once captured into a graph.  Every replay of the graph, into
outputs poisoned with 0xAB before it, must leave the same bytes as the stream
launch; the stream's quantized outputs are also checked against the oracle,
so the graph is tied to the parity of the rest of the suite."""
import numpy as np
import pytest

from block_scaled_precision_03_gb300 import inputs
from _util import dev_bf16, expected, assert_qtensor_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsq():
    import block_scaled_precision_03_gb300 as b
    b.lib()
    return b


def _outputs(bsq, torch, experts, rows_moe):
    E = bsq.empty
    o = {
        "Xq": E("mxfp8_e4m3", 256, 512), "Xc": E("mxfp8_e4m3", 512, 256),
        "Wq": E("mxfp8_e4m3", 384, 512), "Wc": E("mxfp8_e4m3", 512, 384),
        "X4": E("nvfp4", 256, 512), "W4": E("nvfp4", 256, 512),
        "A4": E("mxfp4", rows_moe, 512), "A8": bsq.empty_grouped("mxfp8_e4m3", rows_moe, 512, experts),
        "Wm": E("mxfp8_e4m3", experts * 256, 512), "Xd": E("nvfp4", 256, 512),
        "Y": torch.empty((256, 384), dtype=torch.bfloat16, device="cuda"),
        "Y4": torch.empty((256, 256), dtype=torch.float32, device="cuda"),
        "Ym": torch.empty((rows_moe, 256), dtype=torch.bfloat16, device="cuda"),
    }
    return o


def _poison(o, torch):
    for v in o.values():
        if isinstance(v, torch.Tensor):
            v.view(torch.uint8).fill_(0xAB)
        else:
            v.codes.fill_(0xAB)
            v.scales.fill_(0xAB)
            if v.tensor_scale is not None:
                v.tensor_scale.view(torch.uint8).fill_(0xAB)


def _bytes(o, torch):
    out = {}
    for k, v in o.items():
        if isinstance(v, torch.Tensor):
            out[k] = v.view(torch.uint8).cpu().numpy().copy()
        else:
            out[k + ".codes"] = v.codes.cpu().numpy().copy()
            out[k + ".scales"] = v.scales.cpu().numpy().copy()
            if v.tensor_scale is not None:
                out[k + ".ts"] = v.tensor_scale.view(torch.uint8).cpu().numpy().copy()
    return out


def test_graph_replay_equals_stream_launch(bsq):
    import torch
    experts, counts = 4, np.array([300, 5, 0, 395])
    rows_moe = int(counts.sum())
    x_bits, x4_bits = inputs.normal_bf16((256, 512), 1), inputs.normal_bf16((256, 512), 3)
    X = dev_bf16(x_bits)
    W = dev_bf16(inputs.normal_bf16((384, 512), 2, std=0.02))
    X4 = dev_bf16(x4_bits)
    W4 = dev_bf16(inputs.normal_bf16((256, 512), 4, std=0.02))
    A = dev_bf16(inputs.normal_bf16((rows_moe, 512), 5))
    Wm = dev_bf16(inputs.normal_bf16((experts * 256, 512), 6, std=0.02))
    offsets = torch.from_numpy(inputs.group_offsets(counts)).cuda()
    hist0 = torch.zeros(16, dtype=torch.float32, device="cuda")
    hist0[0] = 3.5
    hist = hist0.clone()

    def sequence(o):
        q = bsq.quantize_into
        q(X, "mxfp8_e4m3", "both", o["Xq"], o["Xc"])
        q(W, "mxfp8_e4m3", "both", o["Wq"], o["Wc"])
        bsq.gemm_into(o["Xq"], o["Wq"], o["Y"])
        q(X4, "nvfp4", "row", o["X4"], None)
        q(W4, "nvfp4", "row", o["W4"], None)
        bsq.gemm_into(o["X4"], o["W4"], o["Y4"])
        q(A, "mxfp4", "row", o["A4"], None)
        bsq.mxfp4_to_mxfp8_grouped_into(o["A4"], o["A8"], offsets, experts)
        q(Wm, "mxfp8_e4m3", "row", o["Wm"], None)
        bsq.grouped_gemm_into(o["A8"], offsets, bsq.group_views(o["Wm"], experts), o["Ym"], padded_scales=True)
        bsq.quantize_nvfp4_delayed_into(X4, "row", o["Xd"], None, hist)

    # on the stream
    o_s = _outputs(bsq, torch, experts, rows_moe)
    _poison(o_s, torch)
    sequence(o_s)
    torch.cuda.synchronize()
    bsq.sync_status()
    ref = _bytes(o_s, torch)
    hist_ref = hist.cpu().numpy().copy()

    # the stream's quantized outputs against the oracle
    exp = expected(x_bits, "mxfp8_e4m3", "both")
    assert_qtensor_equal(o_s["Xq"], exp["row"], "X rows")
    assert_qtensor_equal(o_s["Xc"], exp["col"], "X cols")
    assert_qtensor_equal(o_s["X4"], expected(x4_bits, "nvfp4", "row")["row"], "X NVFP4 rows")

    # captured once, replayed twice into poisoned outputs, the history reset
    # before each replay as it stood before the stream launch
    o_g = _outputs(bsq, torch, experts, rows_moe)
    _poison(o_g, torch)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sequence(o_g)
    torch.cuda.synchronize()
    for rep in range(2):
        _poison(o_g, torch)
        hist.copy_(hist0)
        g.replay()
        torch.cuda.synchronize()
        bsq.sync_status()
        got = _bytes(o_g, torch)
        for k, v in ref.items():
            assert np.array_equal(got[k], v), f"replay {rep}: {k}: {(got[k] != v).sum()} bytes differ"
        assert np.array_equal(hist.cpu().numpy(), hist_ref), f"replay {rep}: amax history differs"
