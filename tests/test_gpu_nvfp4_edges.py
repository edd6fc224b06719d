"""NVFP4 quantize at the rounding boundaries, against the oracle, byte for byte.

The kernels reach the recipe's two FP32 quotients, (amax_b / 6) / s_t for the
UE4M3 block scale and x / d for the E2M1 codes, through reciprocals and take
an exact IEEE division only when the fast result lies near a rounding
boundary of the target format.  These tests put quotients on those
boundaries:

* just-in-time scaling: every quotient reachable from BF16 inputs in one
  binade of the tensor scale (all 128 tensor-amax mantissas; every BF16
  block maximum; every BF16 element under every scale code), row-wise, and
  column-wise on a sample of the transposed tensors;
* delayed scaling, whose FP32 history places the tensor scale freely: block
  and element quotients on every UE4M3 midpoint and every E2M1 edge (the
  midpoints and the saturation point 6), 0 to 3 ulps either side;
* a tensor amax far below 2688 * 2^-126, where s_t is an FP32 subnormal and
  1 / s_t overflows, just in time and delayed.

Inputs come from _nvfp4_edges (search in numpy, no oracle arithmetic);
expected bytes from the oracle."""
import numpy as np
import pytest

import oracle
import _nvfp4_edges as E
from _util import dev_bf16, expected, assert_qtensor_equal, host_u8, poisoned_qtensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsq():
    import block_scaled_precision_03_gb300 as b
    b.lib()
    return b


def _quantize(bsq, x, axis):
    """Quantize into 0xAB-filled outputs (a byte the kernel skips shows)."""
    R, C = x.shape
    row = poisoned_qtensor(bsq, "nvfp4", R, C) if axis in ("row", "both") else None
    col = poisoned_qtensor(bsq, "nvfp4", C, R) if axis in ("col", "both") else None
    bsq.quantize_into(dev_bf16(x), "nvfp4", axis, row, col)
    return row, col


def _check(bsq, x, axis, what):
    row, col = _quantize(bsq, x, axis)
    exp = expected(x, "nvfp4", axis)
    if row is not None:
        assert_qtensor_equal(row, exp["row"], f"{what} row")
    if col is not None:
        assert_qtensor_equal(col, exp["col"], f"{what} col")


@pytest.mark.parametrize("chunk", range(8))
def test_jit_block_scales_every_reachable_quotient(bsq, chunk):
    for t in range(chunk * 16, chunk * 16 + 16):
        _check(bsq, E.jit_scale_tensor(t), "row", f"scale tensor {t}")
    bsq.sync_status()


@pytest.mark.parametrize("chunk", range(8))
def test_jit_elements_every_reachable_quotient(bsq, chunk):
    for t in range(chunk * 16, chunk * 16 + 16):
        _check(bsq, E.jit_element_tensor(t), "row", f"element tensor {t}")
    bsq.sync_status()


@pytest.mark.parametrize("axis", ["col", "both"])
def test_jit_edges_column_kernel(bsq, axis):
    # the column-wise quantization of x^T is the row-wise one of x
    for t in range(0, 128, 21):
        _check(bsq, np.ascontiguousarray(E.jit_element_tensor(t).T), axis, f"element tensor {t}^T")
        _check(bsq, np.ascontiguousarray(E.jit_scale_tensor(t).T), axis, f"scale tensor {t}^T")
    bsq.sync_status()


def _check_delayed(bsq, x, hist, axis, what):
    import torch
    R, C = x.shape
    row = poisoned_qtensor(bsq, "nvfp4", R, C) if axis in ("row", "both") else None
    col = poisoned_qtensor(bsq, "nvfp4", C, R) if axis in ("col", "both") else None
    h = torch.from_numpy(hist.copy()).cuda()
    bsq.quantize_nvfp4_delayed_into(dev_bf16(x), axis, row, col, h)
    exp = oracle.nvfp4_delayed_quantize(x, hist, axis)
    for q, key in ((row, "row"), (col, "col")):
        if q is None:
            continue
        codes, scales = exp[key]
        got_c = host_u8(q.codes)
        exp_c = oracle.storage_codes(codes, "nvfp4").ravel()
        assert np.array_equal(got_c, exp_c), f"{what} {key}: {(got_c != exp_c).sum()} code bytes differ"
        assert np.array_equal(host_u8(q.scales), oracle.swizzle_scales(scales)), f"{what} {key}: scales differ"
        assert np.float32(q.tensor_scale.cpu().numpy()[0]) == np.float32(exp["s_t"]), what
    np.testing.assert_array_equal(h.cpu().numpy(), exp["history"])


@pytest.mark.parametrize("axis", ["row", "col", "both"])
def test_delayed_quotients_at_every_edge(bsq, axis):
    for j in E.DELAYED_J:
        hist, _ = E.delayed_history(j)
        x = E.delayed_tensor(j)
        if axis != "row":
            x = np.ascontiguousarray(x.T)
        _check_delayed(bsq, x, hist, axis, f"j={j}")
    bsq.sync_status()


@pytest.mark.parametrize("axis", ["row", "col", "both"])
def test_subnormal_tensor_scale(bsq, axis):
    x = E.subnormal_scale_tensor()
    s_t = oracle.nvfp4_tensor_scale(x)
    assert 0.0 < s_t < 2.0 ** -126                    # FP32 subnormal
    _check(bsq, x, axis, "subnormal s_t")
    # the same scale through delayed scaling
    hist = np.zeros(16, np.float32)
    hist[0] = oracle.tensor_amax(x)
    _check_delayed(bsq, x, hist, axis, "subnormal s_t, delayed")
    bsq.sync_status()
