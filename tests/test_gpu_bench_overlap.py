"""The benchmark's timed step puts independent quantizes on side streams and
replays the step as a CUDA graph; its outputs must be the same bytes as the
step launched op by op on one stream (1/8-size shapes)."""
import os
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_overlapped_step_equals_sequential_step():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    sh = bench.shapes(True)
    step = bench.Step(bench.make_inputs(sh, "all"), sh, "all")
    # outputs the step writes (the rest belong to rows timed after it)
    keys = ["Xq", "Xc", "Wq", "Wc", "Y", "dYr", "dYc", "dX", "dW", "X4q", "W4q", "X42q", "W42q", "Y4", "Y42",
            "A4", "A8", "Wm", "Ym"]
    written = {k: step.out[k] for k in keys}

    def poison():
        for v in written.values():
            if isinstance(v, torch.Tensor):
                v.view(torch.uint8).fill_(0xAB)
            else:
                v.codes.fill_(0xAB)
                v.scales.fill_(0xAB)
                if v.tensor_scale is not None:
                    v.tensor_scale.view(torch.uint8).fill_(0xAB)

    def snap():
        out = {}
        for k, v in written.items():
            if isinstance(v, torch.Tensor):
                out[k] = v.view(torch.uint8).clone()
            else:
                out[k + ".codes"] = v.codes.clone()
                out[k + ".scales"] = v.scales.clone()
                if v.tensor_scale is not None:
                    out[k + ".ts"] = v.tensor_scale.clone()
        return out

    poison()
    step.run()
    torch.cuda.synchronize()
    ref = snap()

    poison()
    step.run_overlapped()
    torch.cuda.synchronize()
    got = snap()
    assert [k for k in ref if not torch.equal(ref[k], got[k])] == []

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        step.run_overlapped()
    for _ in range(2):
        poison()
        g.replay()
        torch.cuda.synchronize()
        got = snap()
        assert [k for k in ref if not torch.equal(ref[k], got[k])] == []
