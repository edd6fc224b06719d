"""Adversarial NVFP4 inputs for the parity tests.

The NVFP4 recipe (every step IEEE FP32, round to nearest):
    s_t = amax_t / 2688,   q_b = (amax_b / 6) / s_t,   s_b = UE4M3(RNE(q_b)),
    d = s_b * s_t,         code = E2M1(RNE(x / d)).
A code changes only where a quotient crosses a rounding boundary of its
target format: the UE4M3 midpoints for q_b, the E2M1 midpoints
{0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5} (and the saturation point 6) for
x / d.  A kernel that reaches these quotients by another route (reciprocals,
products of reciprocals) agrees with the recipe everywhere except within a
few ulps of those boundaries, so these helpers search, in numpy float32, for
BF16 tensors whose quotients land exactly on a boundary and 1, 2 or 3 FP32
ulps either side of it.

Everything here builds inputs only; expected outputs come from the oracle.
"""
import functools

import numpy as np

from block_scaled_precision_03_gb300 import inputs

F32 = np.float32
E2M1_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
E2M1_EDGES = np.concatenate([E2M1_MIDS, np.float32([6.0])])   # plus the saturation point
MAX_ULPS = 3


def ue4m3_values() -> np.ndarray:
    """Values of the UE4M3 codes 0..126 (sign 0, bias 7, 3-bit mantissa)."""
    c = np.arange(127)
    e, m = c >> 3, c & 7
    return np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * 2.0 ** (e - 7.0))


UE4M3 = ue4m3_values()
UE4M3_MIDS = ((UE4M3[:-1] + UE4M3[1:]) / 2).astype(np.float32)      # exact in FP32


def bits(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).view(np.int32).astype(np.int64)


def bf16_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def nearest_bf16(v) -> np.ndarray:
    """BF16 bit patterns nearest to the FP32 values v (ties to even)."""
    return inputs.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def tensor_scale(amax_t: float) -> np.float32:
    return F32(1.0) if amax_t == 0 else F32(F32(amax_t) / F32(2688.0))


def block_q(amax_b, s_t) -> np.ndarray:
    """(amax_b / 6) / s_t, two FP32 divisions."""
    return ((np.asarray(amax_b, np.float32) / F32(6.0)).astype(np.float32) / F32(s_t)).astype(np.float32)


def ue4m3_code(q) -> np.ndarray:
    """RNE UE4M3 code with saturation at 448 (table search, no library cast)."""
    q = np.minimum(np.asarray(q, dtype=np.float64), 448.0)
    i = np.clip(np.searchsorted(UE4M3, q, side="right") - 1, 0, 126)
    j = np.minimum(i + 1, 126)
    lo, hi = UE4M3[i], UE4M3[j]
    up = (q - lo > hi - q) | ((q - lo == hi - q) & (i % 2 == 1))
    return np.where(up & (j != i), j, i).astype(np.uint8)


def _edge_dist(q, edges):
    """Signed ulp distance of each FP32 quotient to its nearest edge, and the edge index."""
    q = np.asarray(q, dtype=np.float32)
    k = np.clip(np.searchsorted(edges, q), 1, len(edges) - 1)
    lo, hi = edges[k - 1], edges[k]
    idx = np.where(np.abs(q - lo) <= np.abs(hi - q), k - 1, k)
    return bits(q) - bits(edges[idx]), idx


# Just-in-time scaling.  amax_t is a BF16 value, so s_t = RN(amax_t / 2688)
# takes one of only 128 mantissas (one per BF16 mantissa; the binade shifts
# every quotient by a power of two and changes nothing), the block scale
# code c one of 126 values, and x is BF16.  The set of reachable quotients is
# small enough to cover completely: one tensor per amax_t mantissa, holding
# every BF16 block maximum that can give a nonzero scale (block-scale
# tensors) or, for every scale code, every BF16 element the block can hold
# (element tensors).
AMAX_T = tuple(float(F32((128 + t) * 16.0)) for t in range(128))     # [2048, 4096), every mantissa


def _rows(blocks):
    """Blocks of 16 values -> [R, 64] BF16 tensor, R a multiple of 16."""
    n = len(blocks)
    pad = (-n) % 64
    t = np.concatenate([np.stack(blocks).astype(np.float32), np.zeros((pad, 16), np.float32)])
    return nearest_bf16(t).reshape(-1, 64)


def jit_scale_tensor(t: int):
    """Every BF16 block maximum amax_b from 2^-20 amax_t up to amax_t, one
    block each (the other 15 values below it), for amax_t = AMAX_T[t]."""
    amax_t = F32(AMAX_T[t])
    lo = int(np.ravel(nearest_bf16(np.float32([amax_t * 2.0 ** -20])))[0])
    hi = int(np.ravel(nearest_bf16(np.float32([amax_t])))[0])
    rng = np.random.default_rng(100 + t)
    blocks = [np.concatenate([[amax_t], np.zeros(15)])]
    for b in range(lo, hi + 1):
        a = float(bf16_to_f32(np.uint32(b)))
        blk = rng.uniform(-1.0, 1.0, 16) * a
        blk[rng.integers(16)] = a if (b & 1) else -a
        blocks.append(blk)
    return _rows(blocks)


def jit_element_tensor(t: int):
    """For amax_t = AMAX_T[t] and every scale code c: blocks whose maximum is
    the largest BF16 value with code c and whose other values run through
    every BF16 value from d / 8 up to that maximum (d = value(c) s_t), with
    alternating signs."""
    amax_t = F32(AMAX_T[t])
    s_t = tensor_scale(amax_t)
    blocks = [np.concatenate([[amax_t], np.zeros(15)])]
    top = np.arange(0x0080, 0x7F80, dtype=np.uint32)
    topv = bf16_to_f32(top)
    topv = topv[topv <= amax_t]
    codes = ue4m3_code(block_q(topv, s_t))
    for c in range(1, 127):
        hit = np.flatnonzero(codes == c)
        if len(hit) == 0:
            continue
        amax_b = float(topv[hit[-1]])
        d = F32(F32(UE4M3[c]) * s_t)
        lo = int(np.ravel(nearest_bf16(np.float32([d / 8])))[0])
        hi = int(np.ravel(nearest_bf16(np.float32([amax_b])))[0])
        xs = bf16_to_f32(np.arange(lo, hi + 1, dtype=np.uint32))
        xs = xs[xs <= amax_b]
        xs = np.where(np.arange(len(xs)) % 2 == 1, -xs, xs)
        for i in range(0, len(xs), 15):
            blk = np.zeros(16)
            blk[0] = amax_b
            chunk = xs[i:i + 15]
            blk[1:1 + len(chunk)] = chunk
            blocks.append(blk)
    return _rows(blocks)


def quotient_coverage(x_bits: np.ndarray, scales, s_t):
    """Set of (E2M1 edge index, ulp distance) pairs, |distance| <= MAX_ULPS,
    that the element quotients |x| / d of a row-wise quantized tensor reach
    (d from the given row-major block scales; FP32 restatement)."""
    R, C = x_bits.shape
    x = np.abs(bf16_to_f32(x_bits).reshape(R, C // 16, 16))
    d = (UE4M3[np.minimum(scales, 126)].astype(np.float32) * F32(s_t)).astype(np.float32)
    live = (scales > 0) & (scales < 127)
    q = (x[live] / d[live][:, None]).astype(np.float32).ravel()
    q = q[np.isfinite(q) & (q > 0)]
    dist, idx = _edge_dist(q, E2M1_EDGES)
    near = np.abs(dist) <= MAX_ULPS
    return {(int(i), int(k)) for i, k in zip(idx[near], dist[near])}


def scale_coverage(x_bits: np.ndarray, s_t):
    """Set of (UE4M3 midpoint index, ulp distance) pairs, |distance| <=
    MAX_ULPS, that the block quotients (amax_b / 6) / s_t reach."""
    R, C = x_bits.shape
    amax = np.abs(bf16_to_f32(x_bits).reshape(R, C // 16, 16)).max(axis=2).ravel()
    q = block_q(amax[amax > 0], s_t)
    q = q[q < 500]
    dist, idx = _edge_dist(q, UE4M3_MIDS)
    near = np.abs(dist) <= MAX_ULPS
    return {(int(i), int(k)) for i, k in zip(idx[near], dist[near])}


# Delayed scaling takes s_t from an FP32 history, so quotients can be placed
# at chosen ulp offsets: with s_t = 2^-3 (1 + j 2^-24), an element x = m v 2^-3
# (exact in BF16) of a block with scale value v has x / d within a few ulps
# of the edge m, and a block maximum 0.75 w (w a UE4M3 midpoint) has
# (amax_b / 6) / s_t = w / (1 + j 2^-24).
DELAYED_J = tuple(range(-16, 17))


def delayed_history(j: int):
    """A 16-entry FP32 amax history whose maximum h gives s_t = RN(h / 2688)
    at or next to 2^-3 (1 + j 2^-24) (not every FP32 value is a reachable
    quotient); returns (history, s_t)."""
    target = 2.0 ** -3 * (1 + j * 2.0 ** -24)
    h = F32(target * 2688.0)
    s_t = F32(h / F32(2688.0))
    hist = np.zeros(16, dtype=np.float32)
    hist[5] = h
    hist[9] = h * F32(0.5)
    return hist, s_t


def delayed_tensor(j: int):
    """Blocks for every (scale code, E2M1 edge) with an exact BF16 element
    m v 2^-3, and blocks whose maximum sits on every UE4M3 midpoint."""
    _, s_t = delayed_history(j)
    blocks = []
    rng = np.random.default_rng(200 + j)
    for c in range(1, 127):
        v = UE4M3[c]
        xs = [float(m * v * 2.0 ** -3) for m in E2M1_EDGES]
        xs = [x for x in xs if float(bf16_to_f32(nearest_bf16(np.float32([x])))[0]) == x]
        if not xs:
            continue
        amax_b = _amax_for_code(c, max(xs), s_t, 1e30)
        if amax_b is None:
            continue
        vals = [v for x in xs for v in (x, -x)][:15]
        blk = np.zeros(16)
        blk[0] = amax_b
        blk[1:1 + len(vals)] = vals
        blocks.append(blk)
    for w in UE4M3_MIDS:
        a = float(F32(0.75) * w)
        blk = rng.uniform(-1, 1, 16) * a
        blk[0] = a
        blocks.append(blk)
    return _rows(blocks)


def _amax_for_code(c, x, s_t, limit):
    """Smallest BF16 amax_b >= x (and <= limit) whose block scale code is c."""
    b0 = int(np.ravel(nearest_bf16(np.float32([x])))[0])
    cand = np.arange(b0, min(b0 + 400, 0x7F80), dtype=np.uint32)
    v = bf16_to_f32(cand)
    ok = (v >= F32(x)) & (v <= F32(limit)) & (ue4m3_code(block_q(v, s_t)) == c)
    hit = np.flatnonzero(ok)
    return float(v[hit[0]]) if len(hit) else None


def subnormal_scale_tensor(seed: int = 3):
    """A tensor whose amax is far below 2688 * 2^-126: its tensor scale is an
    FP32 subnormal (and 1 / s_t overflows)."""
    x = inputs.normal_bf16((64, 128), seed)
    f = bf16_to_f32(x).astype(np.float64) * 2.0 ** -120
    return nearest_bf16(f.astype(np.float32)).reshape(64, 128)
