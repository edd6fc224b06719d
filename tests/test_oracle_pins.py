"""Pins for the CPU oracle: each test ties an oracle function to something
other than itself -- values the pages print, closed forms, an independent
library routine (torch's float8 casts), invariants and brute force.

Sources: "FP8 Training Infrastructure" (introl.com), section "O panorama da
precisao numerica" (E4M3 up to +-448; E5M2 wider range); the MoE FP4 page
("Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs"),
section 2 "Metodologia" (32-element MXFP4 blocks, power-of-two scales,
numerically equivalent FP4->FP8 conversion); OCP Microscaling v1.0 for the
element encodings.
"""
import os
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, E2M1, UE4M3
from block_scaled_precision_03_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ codecs
def test_page_constants():
    g = dict(_golden("format_constants.txt"))
    assert oracle.max_finite(E4M3) == float(g["e4m3_max"])          # 448 (FP8 page)
    assert oracle.BLOCK["mxfp4"] == int(g["mxfp4_block"])            # 32 (MoE FP4 page)
    # NVFP4 4 + 8/16 = 4.5 bit/elem vs FP8 8 bit: ~1.8x (FP8 page)
    nv_bits = 8.0 * (8192 * 4096 // 2 + oracle.scales_nbytes(8192, 4096 // 16)) / (8192 * 4096)
    assert abs(8.0 / nv_bits - float(g["nvfp4_vs_fp8_memory"])) < 0.05
    mx8_bits = 8.0 * (8192 * 4096 + oracle.scales_nbytes(8192, 4096 // 32)) / (8192 * 4096)
    assert mx8_bits == 8.25 and nv_bits == 4.5


def test_closed_form_extremes():
    assert oracle.max_finite(E5M2) == 1.75 * 2 ** 15 == 57344.0
    assert oracle.max_finite(E2M1) == 6.0
    assert oracle.decode(E4M3, 0x01) == 2.0 ** -9
    assert oracle.decode(E5M2, 0x01) == 2.0 ** -16
    assert oracle.decode(E2M1, 0x1) == 0.5
    assert oracle.decode_e8m0(127) == 1.0
    assert oracle.decode_e8m0(0) == 2.0 ** -127
    assert oracle.decode_e8m0(254) == 2.0 ** 127
    assert math.isnan(oracle.decode_e8m0(255))


def test_e2m1_value_set():
    t = oracle.decode_table(E2M1)
    assert list(t[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(t[8:]) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    assert math.copysign(1, t[8]) == -1


@pytest.mark.parametrize("fmt,dt", [(E4M3, torch.float8_e4m3fn), (E5M2, torch.float8_e5m2)])
def test_decode_matches_torch_float8(fmt, dt):
    """All 256 codes decode exactly as torch's independent float8 types do."""
    ours = oracle.decode_table(fmt)
    ref = torch.arange(256, dtype=torch.uint8).view(dt).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])
    np.testing.assert_array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


@pytest.mark.parametrize("fmt", [E4M3, E5M2, E2M1])
def test_roundtrip_and_monotonic(fmt):
    t = oracle.decode_table(fmt)
    half = len(t) // 2
    for c, v in enumerate(t):
        if math.isnan(v):
            assert oracle.encode(fmt, v) == 0x7F
        elif math.isinf(v):
            # saturating encode: Inf maps to the largest finite magnitude
            assert oracle.decode(fmt, oracle.encode(fmt, v)) == math.copysign(oracle.max_finite(fmt), v)
        else:
            assert oracle.encode(fmt, v) == c, (fmt, c, v)
    pos = t[:half]
    pos = pos[np.isfinite(pos)]
    assert np.all(np.diff(pos) > 0)


@pytest.mark.parametrize("fmt", [E4M3, E5M2, E2M1])
def test_midpoints_round_to_even(fmt):
    t = oracle.decode_table(fmt)
    n = {E4M3: 127, E5M2: 124, E2M1: 8}[fmt]
    for i in range(n - 1):
        lo, hi = t[i], t[i + 1]
        mid = (lo + hi) / 2
        even = i if i % 2 == 0 else i + 1
        assert oracle.encode(fmt, mid) == even
        assert oracle.encode(fmt, -mid) == even | (0x8 if fmt == E2M1 else 0x80)
        assert oracle.encode(fmt, np.nextafter(mid, 0)) == i
        assert oracle.encode(fmt, np.nextafter(mid, np.inf)) == i + 1
    # saturation above the largest finite value
    mx = oracle.max_finite(fmt)
    assert oracle.decode(fmt, oracle.encode(fmt, mx * 1.5)) == mx
    assert oracle.decode(fmt, oracle.encode(fmt, -mx * 100)) == -mx


def test_e2m1_golden_rounding():
    for v, code in _golden("e2m1_rounding.txt"):
        assert oracle.encode(E2M1, float(v)) == int(code, 16), v


@pytest.mark.parametrize("fmt,dt", [(E4M3, torch.float8_e4m3fn), (E5M2, torch.float8_e5m2)])
def test_encode_matches_torch_cast(fmt, dt):
    """In range, RNE encode equals torch's float32 -> float8 cast."""
    rng = np.random.default_rng(7)
    mx = oracle.max_finite(fmt)
    v = (rng.uniform(-1, 1, 4000) * np.exp2(rng.uniform(-24, math.log2(mx), 4000))).astype(np.float32)
    v = np.clip(v, -mx, mx)
    ref = torch.from_numpy(v).to(dt).view(torch.uint8).numpy()
    ours = np.array([oracle.encode(fmt, float(x)) for x in v], dtype=np.uint8)
    np.testing.assert_array_equal(ours, ref)


# ------------------------------------------------------------- block scale
def _blk(fmt, vals, n=32):
    v = np.zeros(n)
    v[:len(vals)] = vals
    return oracle.mx_block(fmt, v)


def test_block_scale_hand_cases():
    # amax exactly a power of two: e = k - emax
    c, s = _blk(E4M3, [2.0 ** 5, 1.0])
    assert s == 127 + 5 - 8 and c[0] == oracle.encode(E4M3, 2.0 ** 8)
    # amax = 448 * 2^k: top code, no saturation
    c, s = _blk(E4M3, [448.0 * 2 ** -3])
    assert s == 127 - 3 and c[0] == 0x7E
    # amax just below 2^(k+1): scaled value 510 > 448 saturates to 448
    c, s = _blk(E4M3, [1.9921875 * 2 ** 4])
    assert s == 127 + 4 - 8 and c[0] == 0x7E
    c, s = _blk(E2M1, [7.5, -1.0])
    assert s == 127 + 2 - 2 and c[0] == 0x7 and c[1] == 0xA
    c, s = _blk(E5M2, [3.0 * 2 ** -20])
    assert s == 127 - 19 - 15 and oracle.decode(E5M2, c[0]) == 1.5 * 2 ** 15  # 3*2^-20 = 1.5*2^-19
    # all-zero block
    c, s = _blk(E4M3, [])
    assert s == 0 and not c.any()
    # NaN / Inf blocks
    c, s = _blk(E4M3, [1.0, float("nan")])
    assert s == 0xFF and (c == 0x7F).all()
    c, s = _blk(E2M1, [float("inf")])
    assert s == 0xFF and not c.any()
    # single large outlier (the x50 activations): scale follows the outlier
    v = np.full(32, 0.01)
    v[3] = -50.0 * 1.3
    c, s = oracle.mx_block(E4M3, v)
    assert s == 127 + 6 - 8 and oracle.decode(E4M3, c[3]) * 2.0 ** (s - 127) == pytest.approx(-65.0, rel=2 ** -4)


def test_block_scale_exponent_range_clamps():
    c, s = _blk(E4M3, [2.0 ** -130])
    assert s == 0
    c, s = _blk(E2M1, [2.0 ** 127])
    assert s == 127 + 127 - 2


@pytest.mark.parametrize("fmt,top", [(E4M3, range(0x78, 0x7F)), (E5M2, range(0x78, 0x7C)), (E2M1, (6, 7))])
def test_quantize_dequant_identity(fmt, top):
    """Blocks whose values are code * 2^e with e the rule's exponent come back unchanged."""
    rng = np.random.default_rng(fmt)
    t = oracle.decode_table(fmt)
    finite = [c for c in range(len(t)) if np.isfinite(t[c])]
    for trial in range(200):
        codes = rng.choice(finite, 32).astype(np.uint8)
        codes[rng.integers(32)] = rng.choice(list(top)) | (0x80 if fmt != E2M1 and rng.random() < .5 else 0)
        e = int(rng.integers(-100, 100))
        vals = np.array([t[c] * 2.0 ** e for c in codes])
        c2, s2 = oracle.mx_block(fmt, vals)
        assert s2 == e + 127
        np.testing.assert_array_equal(c2, codes)


def test_mx_rows_matches_torch_pipeline():
    """Whole-tensor E4M3 MX quantize equals: rule exponent, then torch's RNE cast
    of the clamped scaled values (saturation is clamp-then-round)."""
    x = inputs.outlier_activations_bf16((64, 256), seed=3)
    codes, scales = oracle.mx_quantize_rows(x, "mxfp8_e4m3")
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64).reshape(64, 8, 32)
    amax = np.abs(xf).max(axis=2)
    e = np.floor(np.log2(amax)).astype(np.int64) - 8
    np.testing.assert_array_equal(scales, e + 127)
    scaled = np.clip(xf * np.exp2(-e)[:, :, None], -448, 448).astype(np.float32)
    ref = torch.from_numpy(scaled.reshape(64, 256)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, ref)


# ------------------------------------------------------------------- NVFP4
def test_nvfp4_tensor_amax_block():
    x = inputs.normal_bf16((32, 64), seed=5)
    xf = inputs.bf16_bits_to_f32(x)
    r, c = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
    codes, scales, s_t = oracle.nvfp4_quantize_rows(x)
    amax = float(np.abs(xf).max())
    assert s_t == float(np.float32(amax) / np.float32(2688.0))
    assert scales[r, c // 16] == 0x7E                  # 448 = 2688 / 6
    assert codes[r, c] & 0x7 == 0x7                    # magnitude 6
    # dequantized values stay within half an E2M1 step of the block scale grid
    deq = oracle.dequant_rows(codes, scales, "nvfp4", s_t)
    assert np.all(np.abs(deq - xf) <= np.abs(xf) * 0.25 + 1e-30 + np.repeat(
        oracle.decode_table(E4M3)[scales].reshape(32, 4, 1), 16, axis=2).reshape(32, 64) * s_t * 0.25)


def test_nvfp4_zero_and_tiny_blocks():
    x = np.zeros((1, 32), dtype=np.uint16)
    x[0, 0] = inputs.f32_to_bf16_bits(np.array([1000.0], np.float32))[0]
    x[0, 16] = inputs.f32_to_bf16_bits(np.array([1e-6], np.float32))[0]
    codes, scales, s_t = oracle.nvfp4_quantize_rows(x)
    assert scales[0, 0] == 0x7E and scales[0, 1] == 0 and not codes[0, 16:].any()
    z = np.zeros((2, 16), dtype=np.uint16)
    codes, scales, s_t = oracle.nvfp4_quantize_rows(z)
    assert s_t == 1.0 and not scales.any() and not codes.any()


def test_nvfp4_division_is_fp32():
    """The E2M1 code is the RNE code of the FP32-rounded quotient x / d."""
    x = inputs.normal_bf16((16, 256), seed=11)
    codes, scales, s_t = oracle.nvfp4_quantize_rows(x)
    xf = inputs.bf16_bits_to_f32(x).reshape(16, 16, 16)
    sb = oracle.decode_table(E4M3)[scales].astype(np.float32)
    d = (sb * np.float32(s_t)).astype(np.float32)
    q = (xf / d[:, :, None]).astype(np.float32)
    ref = np.array([oracle.encode(E2M1, float(v)) for v in q.ravel()]).reshape(16, 256)
    ref[np.repeat(scales == 0, 16, axis=1)] = 0
    np.testing.assert_array_equal(codes, ref)


def test_nvfp4_block_scale_two_fp32_divisions():
    """The NVFP4 block scale is UE4M3(RNE((amax_b / 6) / s_t)) with both
    divisions in FP32 (the recipe of the NVFP4 forward workload), on every
    block: checked against numpy float32 arithmetic with two independent
    encoders (a UE4M3 value-table RNE and torch's float8_e4m3fn cast), on
    seeded tensors of the workload's distributions and on tensors whose
    quotients sit on, or 1-3 ulps either side of, every UE4M3 rounding
    midpoint.  The two plausible slips, amax_b / (6 s_t) and a quotient
    rounded once from double precision, each change some of those bytes."""
    import _nvfp4_edges as E
    f32 = np.float32
    cases = [(inputs.normal_bf16((64, 256), 40), None), (inputs.normal_bf16((64, 256), 41, std=0.02), None),
             (inputs.outlier_activations_bf16((64, 256), 42), None), (inputs.loguniform_grad_bf16((64, 256), 43), None)]
    cases += [(E.jit_scale_tensor(t), None) for t in (0, 37, 101)]
    for j in (-16, -5, -1, 0, 1, 4, 9, 16):
        _, s_t = E.delayed_history(j)
        cases.append((E.delayed_tensor(j), float(s_t)))
    slip_one_division = slip_double = 0
    for x, s_t_given in cases:
        codes, scales, s_t = oracle.nvfp4_quantize_rows(x, s_t_given)
        R, C = x.shape
        amax = np.abs(E.bf16_to_f32(x).reshape(R, C // 16, 16)).max(axis=2)
        q = E.block_q(amax, s_t)
        np.testing.assert_array_equal(scales, E.ue4m3_code(q))
        via_torch = torch.from_numpy(np.minimum(q, f32(448))).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(scales, via_torch)
        slip_one_division += int((E.ue4m3_code((amax / (f32(6) * f32(s_t))).astype(f32)) != scales).sum())
        slip_double += int((E.ue4m3_code(amax.astype(np.float64) / 6.0 / np.float64(s_t)) != scales).sum())
    assert slip_one_division > 0 and slip_double > 0


def test_nvfp4_edge_inputs_reach_every_boundary():
    """The adversarial NVFP4 inputs of the GPU parity tests do what they are
    for: under delayed scaling the element quotients reach every E2M1 edge
    and the block quotients every UE4M3 midpoint at distances -3..3 ulps;
    under just-in-time scaling (BF16 inputs) every edge is hit exactly."""
    import _nvfp4_edges as E
    el, sc = set(), set()
    for j in E.DELAYED_J:
        hist, s_t = E.delayed_history(j)
        x = E.delayed_tensor(j)
        d = oracle.nvfp4_delayed_quantize(x, hist, "row")
        assert d["s_t"] == float(s_t)
        el |= E.quotient_coverage(x, d["row"][1], s_t)
        sc |= E.scale_coverage(x, s_t)
    assert el == {(e, k) for e in range(8) for k in range(-3, 4)}
    assert {k for _, k in sc} == set(range(-3, 4))
    jit = set()
    for t in (0, 64, 127):
        x = E.jit_element_tensor(t)
        _, scales, s_t = oracle.nvfp4_quantize_rows(x)
        jit |= E.quotient_coverage(x, scales, s_t)
    assert {(e, 0) for e in range(8)} <= jit


# ------------------------------------------------------------------- repack
REPACK_SCALES = [0, 1, 2, 5, 6, 7, 8, 9, 10, 60, 117, 118, 119, 120, 127, 128, 200, 254, 255]


def test_repack_preserves_values_exhaustive():
    """dequant(repack(x)) == dequant(x) exactly, for every E2M1 code next to
    every other code, over scales including the clamp edge near 2^-127."""
    rows = []
    for a in range(16):
        for b in range(16):
            blk = np.zeros(32, dtype=np.uint8)
            blk[0], blk[1] = a, b
            blk[2:] = (np.arange(30) * 7 + a) % 16
            rows.append(blk)
    codes = np.array(rows, dtype=np.uint8)
    for s in REPACK_SCALES:
        scales = np.full((codes.shape[0], 1), s, dtype=np.uint8)
        c8, s8 = oracle.mxfp4_to_mxfp8_rows(codes, scales)
        d4 = oracle.dequant_rows(codes, scales, "mxfp4")
        d8 = oracle.dequant_rows(c8, s8, "mxfp8_e4m3")
        if s == 255:
            assert np.isnan(d8).all() and (s8 == 255).all()
            continue
        np.testing.assert_array_equal(d8, d4)
        np.testing.assert_array_equal(np.signbit(d8), np.signbit(d4))


def test_repack_integer_rule():
    """For scales away from the E8M0 floor, the new scale is e + e_c - 8 where
    e_c = floor(log2(max |code value|)), and each code is shifted exactly."""
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 16, (500, 32)).astype(np.uint8)
    scales = rng.integers(12, 250, (500, 1)).astype(np.uint8)
    c8, s8 = oracle.mxfp4_to_mxfp8_rows(codes, scales)
    t4 = oracle.decode_table(E2M1)
    for r in range(500):
        m = np.abs(t4[codes[r]]).max()
        if m == 0:
            assert s8[r, 0] == 0 and all(c in (0, 0x80) for c in c8[r])
            continue
        e_c = int(math.floor(math.log2(m)))
        assert s8[r, 0] == scales[r, 0] + e_c - 8
        for k in range(32):
            assert oracle.decode(E4M3, c8[r, k]) == t4[codes[r, k]] * 2.0 ** (8 - e_c)


# --------------------------------------------------------------------- GEMM
def test_gemm_brute_force_integers():
    """Hand-chosen codes whose values are small integers: the result must be
    the exact integer dot product times 2^(eA + eB)."""
    rng = np.random.default_rng(0)
    int_codes = {v: oracle.encode(E4M3, v) for v in range(-16, 17)}
    for M, N, K in [(1, 1, 32), (3, 5, 64), (8, 8, 32), (7, 2, 96)]:
        Ai = rng.integers(-16, 17, (M, K))
        Bi = rng.integers(-16, 17, (N, K))
        Ac = np.vectorize(int_codes.get)(Ai).astype(np.uint8)
        Bc = np.vectorize(int_codes.get)(Bi).astype(np.uint8)
        eA = rng.integers(120, 135, (M, K // 32)).astype(np.uint8)
        eB = rng.integers(120, 135, (N, K // 32)).astype(np.uint8)
        A = oracle.dequant_rows(Ac, eA, "mxfp8_e4m3")
        B = oracle.dequant_rows(Bc, eB, "mxfp8_e4m3")
        ref, mag = oracle.gemm_full(A, B)
        for m in range(M):
            for n in range(N):
                exact = sum(int(Ai[m, k]) * int(Bi[n, k]) * 2.0 ** (int(eA[m, k // 32]) + int(eB[n, k // 32]) - 254)
                            for k in range(K))
                absum = sum(abs(int(Ai[m, k]) * int(Bi[n, k])) * 2.0 ** (int(eA[m, k // 32]) + int(eB[n, k // 32]) - 254)
                            for k in range(K))
                assert ref[m, n] == exact and mag[m, n] == absum
        ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        r2, g2 = oracle.gemm_pairs(A, B, ms.ravel(), ns.ravel())
        np.testing.assert_array_equal(r2, ref.ravel())
        np.testing.assert_array_equal(g2, mag.ravel())


def test_gemm_single_block_is_integer_dot():
    a = np.zeros((1, 32), np.uint8)
    b = np.zeros((1, 32), np.uint8)
    a[0, :4] = [oracle.encode(E4M3, v) for v in (1, 2, -3, 0.5)]
    b[0, :4] = [oracle.encode(E4M3, v) for v in (4, -1, 2, 8)]
    A = oracle.dequant_rows(a, np.array([[130]], np.uint8), "mxfp8_e4m3")
    B = oracle.dequant_rows(b, np.array([[120]], np.uint8), "mxfp8_e4m3")
    ref, mag = oracle.gemm_full(A, B)
    assert ref[0, 0] == (4 - 2 - 6 + 4) * 2.0 ** (3 - 7)
    assert mag[0, 0] == (4 + 2 + 6 + 4) * 2.0 ** (3 - 7)


# ------------------------------------------------------------- scale layout
def test_scale_layout_positions():
    # hand-computed offsets: (r, c) in a [200, 9] scale matrix (S padded to 12)
    assert oracle.scale_tile_offset(0, 0, 9) == 0
    assert oracle.scale_tile_offset(1, 0, 9) == 16
    assert oracle.scale_tile_offset(32, 0, 9) == 4
    assert oracle.scale_tile_offset(33, 5, 9) == 512 + 16 + 4 + 1
    assert oracle.scale_tile_offset(127, 3, 9) == 31 * 16 + 3 * 4 + 3
    assert oracle.scale_tile_offset(128, 0, 9) == 3 * 512
    assert oracle.scale_tile_offset(199, 8, 9) == (3 + 2) * 512 + (199 % 32) * 16 + (71 // 32) * 4


def test_scale_layout_bijection_and_padding():
    rng = np.random.default_rng(2)
    for R, S in [(1, 1), (130, 9), (256, 128), (77, 4)]:
        s = rng.integers(1, 255, (R, S)).astype(np.uint8)
        buf = oracle.swizzle_scales(s)
        assert buf.size == oracle.scales_nbytes(R, S) == ((R + 127) // 128 * 128) * ((S + 3) // 4 * 4)
        np.testing.assert_array_equal(oracle.unswizzle_scales(buf, R, S), s)
        pad = oracle.scale_pad_mask(R, S)
        assert pad.sum() == buf.size - R * S and not buf[pad].any()


def test_fp4_packing():
    c = np.array([[1, 2, 3, 4, 0xF, 0x8]], np.uint8)
    p = oracle.pack_fp4(c)
    np.testing.assert_array_equal(p, [[0x21, 0x43, 0x8F]])
    np.testing.assert_array_equal(oracle.unpack_fp4(p), c)


def test_column_wise_is_transpose():
    x = inputs.normal_bf16((64, 96), seed=4)
    c1, s1, _ = oracle.quantize_cols(x, "mxfp8_e5m2")
    c2, s2 = oracle.mx_quantize_rows(np.ascontiguousarray(x.T), "mxfp8_e5m2")
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(s1, s2)
    assert c1.shape == (96, 64)


# ------------------------------------------------------------ delayed scaling
def _abs_max_numpy(x_bits):
    """max |x| of finite BF16 values, by numpy on the FP32 widening."""
    f = (np.asarray(x_bits, np.uint32) << 16).view(np.float32)
    f = np.abs(f[np.isfinite(f)])
    return float(f.max()) if f.size else 0.0


def test_delayed_equals_just_in_time_when_history_holds_the_amax():
    # a history whose max is this tensor's own amax reproduces the
    # just-in-time recipe exactly (tensor scale, block scales, codes)
    x = inputs.outlier_activations_bf16((96, 256), 5)
    amax = _abs_max_numpy(x)
    hist = np.float32([amax / 4, amax, 0.0, amax / 2] + [0.0] * 12)
    d = oracle.nvfp4_delayed_quantize(x, hist, "both")
    for key, src in (("row", x), ("col", np.ascontiguousarray(x.T))):
        c, s, st = oracle.nvfp4_quantize_rows(src)
        np.testing.assert_array_equal(d[key][0], c)
        np.testing.assert_array_equal(d[key][1], s)
        assert d["s_t"] == st


def test_delayed_history_update():
    x = inputs.normal_bf16((32, 64), 6)
    hist = np.float32(np.arange(1, 17))
    d = oracle.nvfp4_delayed_quantize(x, hist)
    assert d["history"].dtype == np.float32 and d["history"].shape == (16,)
    assert d["history"][0] == np.float32(_abs_max_numpy(x))
    np.testing.assert_array_equal(d["history"][1:], hist[:-1])
    assert d["s_t"] == float(np.float32(16.0) / np.float32(2688.0))


def test_delayed_saturates_beyond_the_history():
    # history max = amax / 64: the block holding the amax takes the largest
    # UE4M3 scale (448) and its largest element the largest E2M1 code (6), so
    # it dequantizes to 6 * 448 * s_t = max(history) exactly; nothing is larger
    x = inputs.normal_bf16((16, 128), 7)
    amax = _abs_max_numpy(x)
    h = np.float32([amax / 64.0] + [0.0] * 15)
    d = oracle.nvfp4_delayed_quantize(x, h)
    c, s = d["row"]
    v = oracle.dequant_rows(c, s, "nvfp4", d["s_t"])
    assert np.abs(v).max() == 6.0 * 448.0 * d["s_t"]
    r, k = np.unravel_index(np.argmax(np.abs((np.asarray(x, np.uint32) << 16).view(np.float32))), x.shape)
    assert s[r, k // 16] == 0x7E and abs(v[r, k]) == 6.0 * 448.0 * d["s_t"]


def test_delayed_empty_history_uses_unit_scale():
    x = inputs.normal_bf16((16, 64), 8)
    d = oracle.nvfp4_delayed_quantize(x, np.zeros(16, np.float32))
    assert d["s_t"] == 1.0
    c, s, _ = oracle.nvfp4_quantize_rows(x, 1.0)
    np.testing.assert_array_equal(d["row"][0], c)
    np.testing.assert_array_equal(d["row"][1], s)


# ------------------------------------------------------------ FP4RowToFP8Col
def _bf16_bits_of_exact(v):
    """Exact doubles that BF16 represents -> BF16 bit patterns (asserts exactness)."""
    f = np.asarray(v, np.float64).astype(np.float32)
    assert np.array_equal(f.astype(np.float64), v)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(((bits.astype(np.uint32) << 16).view(np.float32)).astype(np.float64), v)
    return bits


def test_fp4_row_to_fp8_col_equals_column_quantize_of_dequant():
    # MXFP4 made from BF16 data dequantizes to values BF16 holds exactly, so the
    # fused step must equal the (separately pinned) column-wise E4M3 quantize of
    # those values
    for seed, shape in ((40, (64, 96)), (41, (128, 64)), (42, (96, 256))):
        x = inputs.outlier_activations_bf16(shape, seed)
        c4, s4 = oracle.mx_quantize_rows(x, "mxfp4")
        v = oracle.dequant_rows(c4, s4, "mxfp4")
        cc, sc, _ = oracle.quantize_cols(_bf16_bits_of_exact(v), "mxfp8_e4m3")
        c8, s8 = oracle.mxfp4_row_to_mxfp8_col(c4, s4)
        np.testing.assert_array_equal(c8, cc)
        np.testing.assert_array_equal(s8, sc)


def test_fp4_row_to_fp8_col_lossless_with_uniform_row_scales():
    # one E8M0 scale for every row of a column block: every value is an E2M1
    # value times that scale, which E4M3 holds exactly after the re-scale
    rng = np.random.default_rng(43)
    R, C = 64, 64
    c4 = rng.integers(0, 16, (R, C)).astype(np.uint8)
    s4 = np.full((R, C // 32), 120, np.uint8)
    c8, s8 = oracle.mxfp4_row_to_mxfp8_col(c4, s4)
    v4 = oracle.dequant_rows(c4, s4, "mxfp4")
    v8 = oracle.dequant_rows(c8, s8, "mxfp8_e4m3")
    np.testing.assert_array_equal(v8, v4.T)


def test_fp4_row_to_fp8_col_nan_scale_and_zero_block():
    c4 = np.zeros((64, 32), np.uint8)
    c4[40, 5] = 0x7                       # 6.0 in the second row block
    s4 = np.full((64, 1), 127, np.uint8)
    s4[3, 0] = 0xFF                       # NaN scale on row 3: first row block of every column
    c8, s8 = oracle.mxfp4_row_to_mxfp8_col(c4, s4)
    assert (s8[:, 0] == 0xFF).all() and (c8[:, :32] == 0x7F).all()
    assert (s8[:, 1][np.arange(32) != 5] == 0).all()      # all-zero blocks: scale 2^-127
    assert s8[5, 1] == 127 + 2 - 8 and c8[5, 40] == oracle.encode(E4M3, 6.0 * 2.0 ** 6)


# ------------------------------------------------ per-expert padded scales
def test_grouped_scale_layout_reduces_to_plain():
    rng = np.random.default_rng(70)
    s = rng.integers(1, 255, (300, 9)).astype(np.uint8)
    # one expert, or experts whose sizes are multiples of 128: the plain layout
    np.testing.assert_array_equal(oracle.swizzle_scales_grouped(s, [0, 300]), oracle.swizzle_scales(s))
    s2 = rng.integers(1, 255, (384, 5)).astype(np.uint8)
    np.testing.assert_array_equal(oracle.swizzle_scales_grouped(s2, [0, 128, 128, 384]), oracle.swizzle_scales(s2))


def test_grouped_scale_layout_rows_and_padding():
    # each expert's rows start on a 128-row tile boundary of the padded
    # matrix; read back through the plain (independently pinned) layout
    rng = np.random.default_rng(71)
    counts = np.array([100, 0, 300, 1, 129, 70])
    off = np.concatenate([[0], np.cumsum(counts)])
    R, S = int(off[-1]), 7
    s = rng.integers(1, 255, (R, S)).astype(np.uint8)
    P, total = oracle.grouped_scale_starts(off)
    assert list(P) == [0, 128, 128, 512, 640, 896] and total == 1024
    buf = oracle.swizzle_scales_grouped(s, off, capacity_rows=1152)
    m = oracle.unswizzle_scales(buf, 1152, S)
    used = np.zeros(1152, bool)
    for g in range(len(counts)):
        np.testing.assert_array_equal(m[P[g]:P[g] + counts[g]], s[off[g]:off[g + 1]])
        used[P[g]:P[g] + counts[g]] = True
        assert P[g] % 128 == 0
    assert not m[~used].any()
    assert buf.size == 1152 * 8 and not buf[oracle.scale_pad_mask(1152, S)].any()


# ------------------------------------------------- MXFP4 -> FP8 1x128 blocks
# E4M3 bytes of the eight E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, worked
# out by hand from E4M3's fields (bias 7, 3 mantissa bits): 0.5 = 2^-1 ->
# exponent field 6 -> 0x30; 1.5 = 1.5 * 2^0 -> field 7, mantissa 4 -> 0x3C;
# 6 = 1.5 * 2^2 -> field 9, mantissa 4 -> 0x4C; the sign is bit 7.
E4M3_OF_E2M1 = [0x00, 0x30, 0x38, 0x3C, 0x40, 0x44, 0x48, 0x4C]


def test_1x128_equal_scales_maps_each_code():
    # four equal block scales: the 128-block keeps that scale and every E2M1
    # code becomes the E4M3 code of the same value
    codes = (np.arange(2 * 256) % 16).astype(np.uint8).reshape(2, 256)
    scales = np.array([[90] * 8, [200] * 8], np.uint8)
    c8, s8 = oracle.mxfp4_to_fp8_1x128(codes, scales)
    assert s8.tolist() == [[90, 90], [200, 200]]
    want = [E4M3_OF_E2M1[n & 7] | (0x80 if n & 8 else 0) for n in range(16)]
    assert c8.tolist() == [[want[n] for n in row] for row in codes.tolist()]


def test_1x128_scale_is_the_largest_of_four_and_ragged_tail():
    # C = 160: one full 128-block and a 32-element tail block of its own
    codes = np.zeros((3, 160), np.uint8)
    scales = np.array([[10, 13, 12, 11, 7],
                       [0, 0, 0, 0, 0],
                       [254, 1, 2, 3, 255]], np.uint8)
    _, s8 = oracle.mxfp4_to_fp8_1x128(codes, scales)
    assert s8.tolist() == [[13, 7], [0, 0], [254, 255]]


def test_1x128_exact_within_five_binades():
    # a block whose scale is d <= 5 binades below the largest keeps every value
    # (0.5 * 2^-5 = 2^-6 is E4M3's smallest normal): dequantizing the output
    # over the 128-block scale gives back the MXFP4 values
    rng = np.random.default_rng(60)
    R, C = 16, 256
    codes = rng.integers(0, 16, (R, C)).astype(np.uint8)
    top = rng.integers(20, 230, (R, C // 128))
    d = rng.integers(0, 6, (R, C // 32))
    d[:, ::4] = 0                                        # each group holds its largest scale
    scales = (np.repeat(top, 4, axis=1) - d).astype(np.uint8)
    c8, s8 = oracle.mxfp4_to_fp8_1x128(codes, scales)
    v4 = oracle.dequant_rows(codes, scales, "mxfp4")
    e4m3 = oracle.decode_table(E4M3)
    v8 = e4m3[c8] * np.repeat(np.exp2(s8.astype(np.float64) - 127.0), 128, axis=1)
    np.testing.assert_array_equal(v8, v4)


def test_1x128_rounding_worked_examples():
    # one group: block 0 holds the largest scale 140, block 1 sits d binades
    # below it; each value is code * 2^-d rounded once to E4M3 (subnormal step
    # 2^-9), the cases below worked by hand
    cases = [  # (E2M1 code, d, expected E4M3 byte)
        (0x7, 8, 0x0C),    # 6 * 2^-8 = 1.5 * 2^-6: smallest normal binade, mantissa 4
        (0x7, 9, 0x06),    # 6 * 2^-9: subnormal 6
        (0x5, 10, 0x02),   # 3 * 2^-10 = 1.5 * 2^-9: tie between 1 and 2, even -> 2
        (0x3, 9, 0x02),    # 1.5 * 2^-9: tie -> 2
        (0x1, 9, 0x00),    # 0.5 * 2^-9 = 2^-10: tie between 0 and 1, even -> 0
        (0x6, 12, 0x00),   # 4 * 2^-12 = 2^-10: tie -> 0
        (0x6, 11, 0x01),   # 4 * 2^-11 = 2^-9: the smallest subnormal
        (0xD, 10, 0x82),   # -3 * 2^-10: tie -> -2 subnormals
        (0xF, 30, 0x80),   # -6 * 2^-30 rounds to -0
    ]
    for code, d, want in cases:
        codes = np.zeros((1, 128), np.uint8)
        codes[0, 32] = code
        scales = np.array([[140, 140 - d, 140, 140]], np.uint8)
        c8, s8 = oracle.mxfp4_to_fp8_1x128(codes, scales)
        assert s8[0, 0] == 140 and c8[0, 32] == want, (code, d, hex(c8[0, 32]), hex(want))


def test_1x128_nan_scale_poisons_its_block_only():
    codes = np.full((2, 256), 0x2, np.uint8)           # 1.0 everywhere
    scales = np.full((2, 8), 127, np.uint8)
    scales[0, 5] = 0xFF                                # second 128-block of row 0
    c8, s8 = oracle.mxfp4_to_fp8_1x128(codes, scales)
    assert s8.tolist() == [[127, 255], [127, 127]]
    assert (c8[0, 128:] == 0x7F).all() and (c8[0, :128] == 0x38).all() and (c8[1] == 0x38).all()
