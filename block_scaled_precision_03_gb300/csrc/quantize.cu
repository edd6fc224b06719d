// Quantize kernels: BF16 -> MXFP8 (E4M3 / E5M2), MXFP4, NVFP4.
//
// Row-wise MX ("FP8 Training Infrastructure", section "Estrategias de
// escalonamento": per-block scale factors; "Practical FP4 Training for
// Large-Scale MoE Models on Hopper GPUs", section 2, kernel BF16ToFP4Row:
// quantize and pack).  The row kernel streams the input once with 16-byte
// loads; four lanes own one 32-element block and find its amax with two
// shuffles.
//
// Column-wise / both (MoE FP4 page, section 2: the transposed operand of
// FP4RowToFP8Col; the backward needs column blocks of activations, weights
// and gradients).  The tile kernel loads a 128 x 64 BF16 tile into
// registers (an 8 x 8 sub-tile per thread) and emits the transposed
// column-wise tensor and, in BOTH mode, the row-wise tensor from the same
// read.
//
// NVFP4 (FP8 page, section "MXFP8 e NVFP4 do Blackwell"): a tensor amax
// pass, then per 16-block UE4M3 scales against the FP32 tensor scale
// amax / (448 * 6), each step an IEEE FP32 operation.  Just in time, the
// amax pass runs first and the quantize kernel (row pass or tile kernel)
// follows as its programmatic dependent.
#include "common.cuh"
#include "internal.h"

namespace bsq {

// ---------------------------------------------------------------------------
// Division of 32-bit unsigned integers by an invariant divisor d (1 <= d <
// 2^31), after Granlund and Montgomery, "Division by invariant integers
// using multiplication" (PLDI 1994), the round-up method: with l = ceil(log2
// d) and m = floor(2^32 (2^l - d) / d) + 1, n / d = (t + ((n - t) >> 1)) >>
// (l - 1) where t = umulhi(m, n), for every 32-bit n; d = 1 is n itself.
// ---------------------------------------------------------------------------
struct DivU32 {
    uint32_t m, l;
};
static DivU32 make_div_u32(uint32_t d) {
    uint32_t l = 0;
    while (l < 32 && (1ull << l) < d) l++;
    const uint64_t m = ((((1ull << l) - d) << 32) / d) + 1;
    return DivU32{(uint32_t)m, l};
}
__device__ __forceinline__ uint32_t div_u32(uint32_t n, DivU32 q) {
    if (q.l == 0) return n;
    const uint32_t t = __umulhi(q.m, n);
    return (t + ((n - t) >> 1)) >> (q.l - 1);
}

// ---------------------------------------------------------------------------
// Block encoders working on registers.
// ---------------------------------------------------------------------------

// Packed FP32 pairs (Blackwell f32x2 arithmetic, each half IEEE RN).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// MX: encode n values (n multiple of 8) given the block's scale byte.
// FP8 output: n bytes; FP4 output: n/2 bytes.  Writes to `out` words.
template <int FMT, int N>
__device__ __forceinline__ void mx_encode(const float* x, uint32_t sbyte, uint32_t* out) {
    if (sbyte == 0xFF) {
        // NaN/Inf in the block: NaN scale, NaN codes (E2M1 has no NaN: 0)
#pragma unroll
        for (int i = 0; i < (is_fp4(FMT) ? N / 8 : N / 4); i++) out[i] = is_fp4(FMT) ? 0u : 0x7F7F7F7Fu;
        return;
    }
    // times 2^-e, two values per packed multiply (exact: a power of two)
    const float inv = mx_inv_scale(sbyte);
    const uint64_t inv2 = f2(inv, inv);
    float v[N];
#pragma unroll
    for (int i = 0; i < N; i += 2) f2split(mul2(f2(x[i], x[i + 1]), inv2), v[i], v[i + 1]);
    if (is_fp4(FMT)) {
#pragma unroll
        for (int i = 0; i < N / 8; i++) out[i] = pack8_fp4(v + 8 * i);
    } else {
#pragma unroll
        for (int i = 0; i < N / 8; i++) {
            uint2 p = pack8_fp8<FMT>(v + 8 * i);
            out[2 * i] = p.x;
            out[2 * i + 1] = p.y;
        }
    }
}

// Correctly rounded a / b from r = RN(1 / b) (Markstein's theorem): q0 =
// RN(a r) lies within one ulp of a / b, the residual q0 b - a is exact in
// one FMA, and one correction with r rounds to RN(a / b).  Holds while b, r
// and the quotient are normal and nothing overflows; the callers keep to
// that range and divide exactly outside it.  The residual is formed as q0 b
// - a and subtracted, so a zero a keeps its sign.
__device__ __forceinline__ float div_from_rcp(float a, float b, float r) {
    const float q0 = __fmul_rn(a, r);
    const float e = __fmaf_rn(q0, b, -a);
    return __fmaf_rn(-e, r, q0);
}

// The exact IEEE divisions of the recipe, out of line so that the compiler
// branches around them instead of issuing them predicated on every lane.
__device__ __noinline__ float nv_exact_block_q(float amax_b, float s_t) {
    return __fdiv_rn(__fdiv_rn(amax_b, 6.0f), s_t);
}
__device__ __noinline__ float nv_exact_div(float x, float d) { return __fdiv_rn(x, d); }

// Per-tensor constants of the NVFP4 block step: s_t, RN(1 / s_t), and
// whether the reciprocal route applies (s_t and 1 / s_t normal).
struct NvT {
    float s_t, rst;
    bool fast;
};
__device__ __forceinline__ NvT nv_tensor_consts(float s_t) {
    NvT t;
    t.s_t = s_t;
    t.rst = __frcp_rn(s_t);
    t.fast = s_t >= 1.17549435e-38f && t.rst < 1.0e38f;
    return t;
}

// NVFP4 per-block scale byte from the block amax (BF16 bits, sign cleared):
// UE4M3(RNE((amax_b / 6) / s_t)), both divisions IEEE FP32 (through
// div_from_rcp; amax_b below 2^-100 or a subnormal s_t divide exactly).
// `sat`: the quotient lies beyond the UE4M3 range (>= 464), so the block's
// element quotients are unbounded.  A block holding NaN/Inf gets 0x7F.
__device__ __forceinline__ uint32_t nv_scale_byte(uint32_t amax_bits, const NvT& t, bool& sat) {
    sat = false;
    if (amax_bits >= 0x7F80u) return 0x7Fu;
    const float amax_b = __uint_as_float(amax_bits << 16);
    float q;
    if (t.fast && amax_bits >= 0x0D80u) {
        const float a6 = div_from_rcp(amax_b, 6.0f, 1.0f / 6.0f);
        const float q0 = __fmul_rn(a6, t.rst);
        if (q0 > 470.0f) {              // beyond 464 + one ulp: saturates to 448
            sat = true;
            return 0x7Eu;
        }
        q = __fmaf_rn(-__fmaf_rn(q0, t.s_t, -a6), t.rst, q0);
    } else {
        q = nv_exact_block_q(amax_b, t.s_t);
    }
    sat = q >= 464.0f;
    return cvt_e4m3x2(q, 0.0f) & 0xFFu;
}

// Eight values -> eight E2M1 nibbles (element i in nibble i), RNE with
// saturation, four cvt and one byte pack.
__device__ __forceinline__ uint32_t pack8_e2m1(const float* v) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r) : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// NVFP4: encode n values (multiple of 8) of one block with scale byte sb:
// code = E2M1(RNE(x / d)), d = RN(s_b s_t), x / d correctly rounded.  Within
// the scale's range |x / d| <= 9 and the reciprocal route applies while d
// and 1 / d are normal; saturated blocks and subnormal d divide exactly.
template <int N>
__device__ __forceinline__ void nv_encode(const float* x, uint32_t sb, bool sat, float s_t, uint32_t* out) {
    if (sb == 0 || sb == 0x7F) {
#pragma unroll
        for (int i = 0; i < N / 8; i++) out[i] = 0u;
        return;
    }
    const float d = __fmul_rn(e4m3_to_float(sb), s_t);
    const float r = __frcp_rn(d);
    float v[N];
    if (!sat && d >= 1.17549435e-38f && r < 1.0e38f) {
#pragma unroll
        for (int i = 0; i < N; i++) v[i] = div_from_rcp(x[i], d, r);
    } else {
#pragma unroll
        for (int i = 0; i < N; i++) v[i] = nv_exact_div(x[i], d);
    }
#pragma unroll
    for (int i = 0; i < N / 8; i++) out[i] = pack8_e2m1(v + 8 * i);
}

// Just in time, the amax pass leaves max over CTAs of RN(amax_cta / 2688)
// in the tensor-scale slot.  Division by a positive constant is monotone, so
// that max is RN(amax / 2688) of the tensor amax; a slot still at 0 means
// the tensor has no nonzero finite value, and s_t = 1.
__device__ __forceinline__ float nv_tensor_scale(const unsigned* ts_bits) {
    unsigned b;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(b) : "l"(ts_bits) : "memory");
    return b == 0u ? 1.0f : __uint_as_float(b);
}

// Where a kernel takes the NVFP4 tensor scale from: the amax of this tensor
// (just in time, after the amax pass) or, with delayed scaling ("FP8 Training
// Infrastructure", "Estrategias de escalonamento": scale factors from the
// amax of previous iterations, history length 16, algorithm max), the
// largest positive finite entry of the amax history; then this tensor's
// amax is accumulated in the same pass for the history update.
struct NvScale {
    unsigned* ts_bits;             // just in time: the tensor-scale slot the amax pass filled
    float* ts_other;               // just in time: a second tensor-scale output (both axes), or nullptr
    const float* history;          // delayed: amax history (nullptr: just in time)
    int32_t hist_len;
    unsigned* amax_acc;            // delayed: this tensor's amax accumulates here (FP32 bits)
};

__device__ __forceinline__ float nv_history_scale(const float* h, int n) {
    float m = 0.0f;
    for (int i = 0; i < n; i++) {
        const float v = h[i];
        if (isfinite(v) && v > m) m = v;
    }
    return m == 0.0f ? 1.0f : __fdiv_rn(m, 2688.0f);
}

__device__ __forceinline__ float nv_scale_of(const NvScale& ns) {
    return ns.history ? nv_history_scale(ns.history, ns.hist_len) : nv_tensor_scale(ns.ts_bits);
}

// Just in time, one thread of the quantize grid completes the tensor-scale
// outputs: an all-zero tensor's slot becomes 1.0 (threads still reading it
// see 0 or 1.0, both meaning s_t = 1), and a second output gets a copy.
__device__ __forceinline__ void nv_publish_scale(const NvScale& ns, float s_t) {
    if (ns.history) return;
    atomicCAS(ns.ts_bits, 0u, __float_as_uint(1.0f));
    if (ns.ts_other) *ns.ts_other = s_t;
}

// Programmatic dependent launch: a quantize kernel launched with programmatic
// stream serialization may start while the amax pass before it still runs;
// it waits here before its first read of the tensor scale.  Under an
// ordinary launch both instructions do nothing.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Running max of finite |x| (BF16 bit patterns without sign): `am` is the
// max over a group of values given as packed words `w`; a group holding a
// non-finite value is rescanned for its finite ones.
__device__ __forceinline__ void nv_acc_group(uint32_t& acc, uint32_t am, const uint32_t* w, int nw) {
    if (am < 0x7F80u) {
        acc = max(acc, am);
        return;
    }
    for (int q = 0; q < nw; q++) {
        const uint32_t lo = w[q] & 0x7FFFu, hi = (w[q] >> 16) & 0x7FFFu;
        if (lo < 0x7F80u) acc = max(acc, lo);
        if (hi < 0x7F80u) acc = max(acc, hi);
    }
}

// Warp-wide max of `acc`, one atomic per warp (all lanes of the warp call it).
__device__ __forceinline__ void nv_acc_flush(const NvScale& ns, uint32_t acc) {
#pragma unroll
    for (int o = 16; o; o >>= 1) acc = max(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
    if ((threadIdx.x & 31) == 0 && acc) atomicMax(ns.amax_acc, acc << 16);
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ void unpack8(const uint4& w, float* f) {
    f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

// Per half, the BF16 value of larger magnitude (sign the XOR of the signs,
// NaN if either is NaN): the magnitudes of max.NaN.xorsign.abs are exact,
// subnormals included, so |result| & 0x7FFF is the larger |x| bit pattern.
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// largest |x| bit pattern of 8 bf16 values (packed 16-bit max on the
// sign-cleared halves; for non-negative finite values and NaN/Inf the
// integer order is the order the block scale needs)
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b);
// largest |x| bit pattern of 8 BF16 values; NaN anywhere gives a NaN
// pattern (above 0x7F80), like an Inf
__device__ __forceinline__ uint32_t absmax8(const uint4& w) {
    const uint32_t m = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
    return bmax2(m, __byte_perm(m, 0, 0x1032)) & 0x7FFFu;
}

// ---------------------------------------------------------------------------
// Row-wise kernel: one thread = 8 elements; BLK/8 lanes = one block.
// ---------------------------------------------------------------------------
constexpr int kRowThreads = 256;
constexpr int kRowUnroll = 4;

template <int FMT>
__global__ void __launch_bounds__(kRowThreads)
quantize_rows_kernel(const uint4* __restrict__ src, int64_t nchunks, uint32_t blocks_per_row,
                     int64_t s_tiles, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                     const NvScale nv) {
    constexpr int BLK = block_of(FMT);
    constexpr int LPB = BLK / 8;            // lanes per block: 4 (MX) or 2 (NV)
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kRowThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kRowThreads) >> 5;
    const bool vec_sf = (blocks_per_row & 3u) == 0;
    NvT nt{1.0f, 1.0f, true};
    if (FMT == kNVFP4) nt = nv_tensor_consts(nv_scale_of(nv));

    // software pipeline: the loads of the next iteration are in flight while
    // the current chunks are encoded
    const int64_t step = nwarps * 32 * kRowUnroll;
    uint4 w[kRowUnroll];
    int64_t base = warp * 32 * kRowUnroll;
#pragma unroll
    for (int u = 0; u < kRowUnroll; u++) {
        const int64_t c = base + u * 32 + lane;
        w[u] = c < nchunks ? ld_stream(src + c) : make_uint4(0, 0, 0, 0);
    }
    // row and block column of this lane's block at u = 0, advanced without a
    // division: by 32 / LPB blocks per u and by step / LPB per iteration
    const int64_t blk_first = base / LPB + lane / LPB;
    uint32_t rb = (uint32_t)(blk_first / blocks_per_row);
    uint32_t jb = (uint32_t)(blk_first - (int64_t)rb * blocks_per_row);
    const uint32_t uq = (uint32_t)(32 / LPB) / blocks_per_row, ur = (uint32_t)(32 / LPB) % blocks_per_row;
    const uint32_t dq = (uint32_t)((step / LPB) / blocks_per_row), dr = (uint32_t)((step / LPB) % blocks_per_row);
    for (; base < nchunks; base += step) {
        uint32_t r = rb, j = jb;
        uint4 wn[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; u++) {
            const int64_t c = base + step + u * 32 + lane;
            wn[u] = c < nchunks ? ld_stream(src + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kRowUnroll; u++) {
            const int64_t c = base + u * 32 + lane;
            uint32_t am = absmax8(w[u]);
            am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
            if (LPB == 4) am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
            bool sat = false;
            uint32_t sb = FMT == kNVFP4 ? nv_scale_byte(am, nt, sat) : mx_scale_byte<FMT>(am);
            float f[8];
            unpack8(w[u], f);
            uint32_t out[2];
            if (FMT == kNVFP4) nv_encode<8>(f, sb, sat, nt.s_t, out);
            else mx_encode<FMT, 8>(f, sb, out);
            if (c < nchunks) {
                if (is_fp4(FMT)) reinterpret_cast<uint32_t*>(codes)[c] = out[0];
                else reinterpret_cast<uint2*>(codes)[c] = make_uint2(out[0], out[1]);
            }
            // scale bytes: gather 4 consecutive blocks into one 32-bit store
            // when a row holds a multiple of 4 blocks, else one byte each.
            if (vec_sf) {
                uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sb, LPB);
                uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sb, 2 * LPB);
                uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sb, 3 * LPB);
                if ((lane % (4 * LPB)) == 0 && c < nchunks)
                    *reinterpret_cast<uint32_t*>(scales + sf_offset(r, j, s_tiles)) =
                        sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
            } else if ((lane % LPB) == 0 && c < nchunks) {
                scales[sf_offset(r, j, s_tiles)] = (uint8_t)sb;
            }
            j += ur;
            r += uq;
            if (j >= blocks_per_row) { j -= blocks_per_row; ++r; }
        }
#pragma unroll
        for (int u = 0; u < kRowUnroll; u++) w[u] = wn[u];
        jb += dr;
        rb += dq;
        if (jb >= blocks_per_row) { jb -= blocks_per_row; ++rb; }
    }
}

// ---------------------------------------------------------------------------
// Row-wise MX kernel for 32-byte aligned source and codes: one thread = one
// 32-element block, read with two 32-byte loads (a warp instruction covers
// 32 whole sectors) and written with one 32-byte (FP8) or 16-byte (FP4)
// store; the block amax needs no shuffle and the scale byte is computed once
// per block.  Two blocks per thread per iteration, the next iteration's
// loads in flight while these encode.
// ---------------------------------------------------------------------------
constexpr int kWideUnroll = 2;

__device__ __forceinline__ void ld_v8(const void* p, uint32_t* r) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "l"(p));
}
__device__ __forceinline__ void st_v8(void* p, const uint32_t* r) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
// four FP32 values -> four FP8 codes in one word (first value in the low byte)
template <int FMT>
__device__ __forceinline__ uint32_t pack4_fp8(float a, float b, float c, float d) {
    uint32_t r;
    if (FMT == kE4M3)
        asm("{\n\t.reg .b16 h0, h1;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 h0, %2, %1;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 h1, %4, %3;\n\t"
            "mov.b32 %0, {h0, h1};\n\t}"
            : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
    else
        asm("{\n\t.reg .b16 h0, h1;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 h0, %2, %1;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 h1, %4, %3;\n\t"
            "mov.b32 %0, {h0, h1};\n\t}"
            : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

template <int FMT>
__global__ void __launch_bounds__(kRowThreads)
quantize_rows_wide_kernel(const uint8_t* __restrict__ src, int64_t nblocks, uint32_t blocks_per_row, int64_t s_tiles,
                          uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    static_assert(FMT != kNVFP4, "MX formats only");
    constexpr int U = kWideUnroll;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kRowThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kRowThreads) >> 5;
    const bool vec_sf = (blocks_per_row & 3u) == 0;
    // a warp takes U x 32 consecutive blocks per iteration (lane-consecutive
    // within each u, so the four blocks of one scale word sit in four lanes)
    const int64_t step = nwarps * 32 * U;
    int64_t base = warp * 32 * U;
    uint32_t w[U][16];
#pragma unroll
    for (int u = 0; u < U; u++) {
        const int64_t b = base + u * 32 + lane;
        if (b < nblocks) {
            ld_v8(src + b * 64, w[u]);
            ld_v8(src + b * 64 + 32, w[u] + 8);
        } else {
#pragma unroll
            for (int k = 0; k < 16; k++) w[u][k] = 0;
        }
    }
    const int64_t b0 = base + lane;
    uint32_t rb = (uint32_t)(b0 / blocks_per_row);
    uint32_t jb = (uint32_t)(b0 - (int64_t)rb * blocks_per_row);
    const uint32_t uq = 32u / blocks_per_row, ur = 32u % blocks_per_row;
    const uint32_t dq = (uint32_t)(step / blocks_per_row), dr = (uint32_t)(step % blocks_per_row);
    for (; base < nblocks; base += step) {
        uint32_t wn[U][16];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t b = base + step + u * 32 + lane;
            if (b < nblocks) {
                ld_v8(src + b * 64, wn[u]);
                ld_v8(src + b * 64 + 32, wn[u] + 8);
            } else {
#pragma unroll
                for (int k = 0; k < 16; k++) wn[u][k] = 0;
            }
        }
        uint32_t r = rb, j = jb;
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t b = base + u * 32 + lane;
            uint32_t m8[8];
#pragma unroll
            for (int k = 0; k < 8; k++) m8[k] = bmax2(w[u][2 * k], w[u][2 * k + 1]);
            uint32_t m = bmax2(bmax2(bmax2(m8[0], m8[1]), bmax2(m8[2], m8[3])),
                               bmax2(bmax2(m8[4], m8[5]), bmax2(m8[6], m8[7])));
            m = bmax2(m, __byte_perm(m, 0, 0x1032)) & 0x7FFFu;
            const uint32_t sb = mx_scale_byte<FMT>(m);
            uint32_t out[8];
            if (sb == 0xFFu) {
                // NaN/Inf in the block: NaN scale, NaN codes (E2M1 has no NaN: 0)
#pragma unroll
                for (int k = 0; k < 8; k++) out[k] = is_fp4(FMT) ? 0u : 0x7F7F7F7Fu;
            } else {
                const float inv = mx_inv_scale(sb);
                if (is_fp4(FMT)) {
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            f[2 * e] = bf16lo(w[u][4 * k + e]) * inv;
                            f[2 * e + 1] = bf16hi(w[u][4 * k + e]) * inv;
                        }
                        out[k] = pack8_e2m1(f);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 8; k++)
                        out[k] = pack4_fp8<FMT>(bf16lo(w[u][2 * k]) * inv, bf16hi(w[u][2 * k]) * inv,
                                                bf16lo(w[u][2 * k + 1]) * inv, bf16hi(w[u][2 * k + 1]) * inv);
                }
            }
            if (b < nblocks) {
                if (is_fp4(FMT)) *reinterpret_cast<uint4*>(codes + b * 16) = make_uint4(out[0], out[1], out[2], out[3]);
                else st_v8(codes + b * 32, out);
            }
            // scale bytes: 4 consecutive blocks -> one 32-bit store when a row
            // holds a multiple of 4 blocks, else one byte each
            if (vec_sf) {
                const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sb, 1);
                const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
                const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sb, 3);
                if ((lane & 3) == 0 && b < nblocks)
                    *reinterpret_cast<uint32_t*>(scales + sf_offset(r, j, s_tiles)) =
                        sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
            } else if (b < nblocks) {
                scales[sf_offset(r, j, s_tiles)] = (uint8_t)sb;
            }
            j += ur;
            r += uq;
            if (j >= blocks_per_row) { j -= blocks_per_row; ++r; }
        }
#pragma unroll
        for (int u = 0; u < U; u++)
#pragma unroll
            for (int k = 0; k < 16; k++) w[u][k] = wn[u][k];
        jb += dr;
        rb += dq;
        if (jb >= blocks_per_row) { jb -= blocks_per_row; ++rb; }
    }
}

// ---------------------------------------------------------------------------
// NVFP4 row-wise encode: a lane takes two consecutive 16-element blocks per
// item (two 32-byte loads, or four 16-byte loads when the input is only
// 16-byte aligned) and loads the next two before encoding these.  Each
// block's scale work is done once, by its lane; d and -RN(1 / d) for the
// 126 finite scale codes come from a table each CTA builds once, and the
// element quotients run two at a time on the packed FP32 pipe.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_cached(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// blocks b and b + 1 (zeros past the end) into w[0..7] and w[8..15]
template <bool V8>
__device__ __forceinline__ void ld_nv_pair(const uint8_t* src, int64_t b, int64_t nblocks, uint32_t* w) {
#pragma unroll
    for (int u = 0; u < 2; u++) {
        uint32_t* o = w + 8 * u;
        if (b + u < nblocks) {
            if (V8) {
                ld_v8(src + (b + u) * 32, o);
            } else {
                const uint4 lo = ld_cached(reinterpret_cast<const uint4*>(src + (b + u) * 32));
                const uint4 hi = ld_cached(reinterpret_cast<const uint4*>(src + (b + u) * 32 + 16));
                o[0] = lo.x; o[1] = lo.y; o[2] = lo.z; o[3] = lo.w;
                o[4] = hi.x; o[5] = hi.y; o[6] = hi.z; o[7] = hi.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; k++) o[k] = 0;
        }
    }
}

// -(x / d), correctly rounded, for both halves of x: div_from_rcp run with
// -r in place of r.  Round to nearest is odd-symmetric, so every step yields
// the exact negation of the corresponding div_from_rcp step, signed zeros
// included: q0' = RN(x (-r)) = -q0, e' = RN(q0' d + x) = -e, and RN(e' (-r) +
// q0') = -q.
__device__ __forceinline__ uint64_t neg_div2(uint64_t x, uint64_t d2, uint64_t nr2) {
    const uint64_t q0 = mul2(x, nr2);
    const uint64_t e = fma2(q0, d2, x);
    return fma2(e, nr2, q0);
}

// (d, -RN(1 / d)) of scale code c against s_t, the second 0 where the
// reciprocal route does not apply (d or 1 / d outside the normal range);
// codes 0 and 0x7F never reach it.
__device__ __forceinline__ float2 nv_scale_entry(uint32_t c, float s_t) {
    if (c == 0 || c >= 0x7F) return make_float2(0.0f, 0.0f);
    const float d = __fmul_rn(e4m3_to_float(c), s_t);
    const float r = __frcp_rn(d);
    return make_float2(d, (d >= 1.17549435e-38f && r < 1.0e38f) ? -r : 0.0f);
}

// E2M1 codes of one block (8 BF16 pairs) with scale entry t into out[0..1]:
// code(x / d) = code(-(x / d)) with the sign bit of every nibble flipped
// (E2M1 is sign-magnitude and its rounding symmetric).
__device__ __forceinline__ void nv_encode_pairs(const uint32_t* w, float2 t, bool fast, uint32_t* out) {
    if (fast) {
        const uint64_t d2 = f2(t.x, t.x), nr2 = f2(t.y, t.y);
#pragma unroll
        for (int h = 0; h < 2; h++) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 4; k++)
                f2split(neg_div2(f2(bf16lo(w[4 * h + k]), bf16hi(w[4 * h + k])), d2, nr2), v[2 * k], v[2 * k + 1]);
            out[h] = pack8_e2m1(v) ^ 0x88888888u;
        }
    } else {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                v[2 * k] = nv_exact_div(bf16lo(w[4 * h + k]), t.x);
                v[2 * k + 1] = nv_exact_div(bf16hi(w[4 * h + k]), t.x);
            }
            out[h] = pack8_e2m1(v);
        }
    }
}

// largest |x| bit pattern of one block (8 BF16 pairs); NaN anywhere gives a
// NaN pattern (above 0x7F80), like an Inf
__device__ __forceinline__ uint32_t block_absmax(const uint32_t* w) {
    const uint32_t m = bmax2(bmax2(bmax2(w[0], w[1]), bmax2(w[2], w[3])), bmax2(bmax2(w[4], w[5]), bmax2(w[6], w[7])));
    return bmax2(m, __byte_perm(m, 0, 0x1032)) & 0x7FFFu;
}

// scale byte (returned) and the two code words of one block
__device__ __forceinline__ uint32_t nv_quantize_block(const uint32_t* w, uint32_t am, const NvT& nt,
                                                      const float2* tab, uint32_t* out) {
    bool sat;
    const uint32_t sb = nv_scale_byte(am, nt, sat);
    if (sb == 0 || sb == 0x7F) {
        out[0] = out[1] = 0u;
    } else {
        const float2 t = tab[sb];
        nv_encode_pairs(w, t, !sat && t.y != 0.0f, out);
    }
    return sb;
}

// ---------------------------------------------------------------------------
// Tile kernel for column-wise and both.  A CTA covers a 128 x TC BF16 tile
// (TC = 64: 128 threads; twice as many CTAs as 128-column tiles, a shorter
// last wave and more warps per SM, measured 2-4% faster on every tensor of
// the step); each thread loads an 8 x 8 sub-tile straight into registers
// (eight 16-byte row loads) and encodes it in both directions without shared
// memory: the 32 (NVFP4: 16) rows of a column block are the four (two) lanes
// of a warp that differ in lane bits 0-1, the columns of a row block the
// lanes that differ in bits 2-3, so block maxima are warp shuffles.  Warp w
// covers rows 32 (w & 3).. and columns 64 (w >> 2)..; lane (q = lane & 3,
// g = lane >> 2) rows 8 q.. and columns 8 g.. of it.  A column's 8 codes
// leave as one 8-byte (FP4: 4-byte) store, four lanes filling 32 contiguous
// bytes; only the scale bytes go through shared memory, to leave as 32-bit
// (two 32-element blocks of a 64-column tile row: 16-bit) words.
// ---------------------------------------------------------------------------
constexpr int kTile = 128;          // tile rows
constexpr int kTileCols = 64;       // tile columns
// Resident CTAs per SM the register budget must allow: 9 (56 registers) for
// the MX formats (10, at 48 registers with a few spills, measured slower),
// 8 for NVFP4 column-wise, 4 (128 registers) for NVFP4 both ways, whose two
// encodes of each element keep more values live.


template <int FMT, bool ROW, bool COL, int TC>
__global__ void __launch_bounds__(2 * TC, FMT == kNVFP4 ? (ROW ? 4 : 8) : 9)
quantize_tile_kernel(const uint16_t* __restrict__ src, int64_t R, int64_t C,
                     uint8_t* __restrict__ codes_r, uint8_t* __restrict__ scales_r, int64_t s_tiles_r,
                     uint8_t* __restrict__ codes_c, uint8_t* __restrict__ scales_c, int64_t s_tiles_c,
                     const NvScale nv) {
    constexpr int BLK = block_of(FMT);
    constexpr int NB = kTile / BLK;                 // blocks per tile edge: 4 or 8
    constexpr int LB = BLK / 8;                     // lanes per block along either axis: 4 or 2
    constexpr int NBC = TC / BLK;                   // column blocks per tile row: 2, 4 or 8
    constexpr int NT = 2 * TC;                      // threads: four warps per 64 columns
    __shared__ __align__(16) uint8_t sf_col[TC * NB];      // [column][row-block]
    __shared__ __align__(16) uint8_t sf_row[kTile * NBC];  // [row][col-block]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q = lane & 3, g = lane >> 2;
    const int tr = (warp & 3) * 32 + q * 8;         // sub-tile origin within the tile
    const int tc = (warp >> 2) * 64 + g * 8;
    const int64_t gr0 = (int64_t)blockIdx.y * kTile + tr;
    const int64_t gc0 = (int64_t)blockIdx.x * TC + tc;
    const bool col_in = gc0 < C, row_in = gr0 < R;  // R % BLK == 0 and C % 8 == 0: chunks are whole
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; i++)
        w[i] = (row_in && col_in) ? ld_stream(reinterpret_cast<const uint4*>(src + (gr0 + i) * C + gc0))
                                  : make_uint4(0, 0, 0, 0);
    NvT nt{1.0f, 1.0f, true};
    if (FMT == kNVFP4) {
        // just in time, the tensor scale comes from the amax pass this grid may
        // overlap; delayed, the history update after this grid may be scheduled now
        if (!nv.history) pdl_wait();
        else pdl_launch_dependents();
        const float s_t = nv_scale_of(nv);
        if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) nv_publish_scale(nv, s_t);
        nt = nv_tensor_consts(s_t);
    }

    if (COL) {
        // column maxima of the 8 rows (packed |bf16| pairs, NaN-propagating,
        // the sign bits masked off at the end), then across the block's lanes
        uint32_t cm[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
#pragma unroll
        for (int i = 1; i < 8; i++) {
            cm[0] = bmax2(cm[0], w[i].x);
            cm[1] = bmax2(cm[1], w[i].y);
            cm[2] = bmax2(cm[2], w[i].z);
            cm[3] = bmax2(cm[3], w[i].w);
        }
        if (FMT == kNVFP4 && nv.amax_acc) {
            // delayed scaling: this tensor's finite amax (zero padding adds nothing)
            uint32_t acc = 0;
            const uint32_t m = bmax2(bmax2(cm[0], cm[1]), bmax2(cm[2], cm[3])) & 0x7FFF7FFFu;
            if (((m & 0xFFFFu) >= 0x7F80u) || ((m >> 16) >= 0x7F80u)) {
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
                    nv_acc_group(acc, 0x7F80u, ws, 4);
                }
            } else {
                acc = max(m & 0xFFFFu, m >> 16);
            }
            nv_acc_flush(nv, acc);
        }
#pragma unroll
        for (int k = 0; k < 4; k++) {
            cm[k] = bmax2(cm[k], __shfl_xor_sync(0xFFFFFFFFu, cm[k], 1));
            if (LB == 4) cm[k] = bmax2(cm[k], __shfl_xor_sync(0xFFFFFFFFu, cm[k], 2));
            cm[k] &= 0x7FFF7FFFu;
        }
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const uint32_t am = (j & 1) ? (cm[j >> 1] >> 16) : (cm[j >> 1] & 0xFFFFu);
            bool sat = false;
            const uint32_t sb = FMT == kNVFP4 ? nv_scale_byte(am, nt, sat) : mx_scale_byte<FMT>(am);
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint32_t word = (j >> 1) == 0 ? w[i].x : ((j >> 1) == 1 ? w[i].y : ((j >> 1) == 2 ? w[i].z : w[i].w));
                f[i] = (j & 1) ? bf16hi(word) : bf16lo(word);
            }
            uint32_t out[2];
            if (FMT == kNVFP4) nv_encode<8>(f, sb, sat, nt.s_t, out);
            else mx_encode<FMT, 8>(f, sb, out);
            if (row_in && col_in) {
                const int64_t gc = gc0 + j;
                if (is_fp4(FMT)) *reinterpret_cast<uint32_t*>(codes_c + gc * (R / 2) + gr0 / 2) = out[0];
                else *reinterpret_cast<uint2*>(codes_c + gc * R + gr0) = make_uint2(out[0], out[1]);
            }
            if ((q % LB) == 0) sf_col[(tc + j) * NB + tr / BLK] = (uint8_t)sb;
        }
    }
    if (ROW) {
#pragma unroll
        for (int i = 0; i < 8; i++) {
            uint32_t am = absmax8(w[i]);
            am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 4));
            if (LB == 4) am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 8));
            bool sat = false;
            const uint32_t sb = FMT == kNVFP4 ? nv_scale_byte(am, nt, sat) : mx_scale_byte<FMT>(am);
            float f[8];
            unpack8(w[i], f);
            uint32_t out[2];
            if (FMT == kNVFP4) nv_encode<8>(f, sb, sat, nt.s_t, out);
            else mx_encode<FMT, 8>(f, sb, out);
            if (row_in && col_in) {
                const int64_t gr = gr0 + i;
                if (is_fp4(FMT)) *reinterpret_cast<uint32_t*>(codes_r + gr * (C / 2) + gc0 / 2) = out[0];
                else *reinterpret_cast<uint2*>(codes_r + gr * C + gc0) = make_uint2(out[0], out[1]);
            }
            if ((g % LB) == 0) sf_row[(tr + i) * NBC + tc / BLK] = (uint8_t)sb;
        }
    }
    __syncthreads();
    // scale stores: groups of 4 consecutive blocks -> one 32-bit word
    const int64_t r0 = (int64_t)blockIdx.y * kTile, c0 = (int64_t)blockIdx.x * TC;
    constexpr int G = NB / 4;
    if (COL) {
        const int64_t S = R / BLK;                       // scale columns of the [C, R] output
        for (int id = tid; id < TC * G; id += NT) {
            const int cl = id / G, gg = id % G;
            const int64_t gc = c0 + cl, sc = r0 / BLK + 4 * gg;
            if (gc < C && sc < S)
                *reinterpret_cast<uint32_t*>(scales_c + sf_offset(gc, sc, s_tiles_c)) =
                    *reinterpret_cast<const uint32_t*>(&sf_col[cl * NB + 4 * gg]);
        }
    }
    if (ROW) {
        const int64_t S = C / BLK;
        if constexpr (NBC >= 4) {
            constexpr int GR = NBC / 4;
            for (int id = tid; id < kTile * GR; id += NT) {
                const int rr = id / GR, gg = id % GR;
                const int64_t gr = r0 + rr, sc = c0 / BLK + 4 * gg;
                if (gr < R && sc < S)
                    *reinterpret_cast<uint32_t*>(scales_r + sf_offset(gr, sc, s_tiles_r)) =
                        *reinterpret_cast<const uint32_t*>(&sf_row[rr * NBC + 4 * gg]);
            }
        } else {
            // a 64-column tile of 32-element blocks: two scale bytes per row, one
            // 16-bit store (the tile's first block column is even)
            for (int rr = tid; rr < kTile; rr += NT) {
                const int64_t gr = r0 + rr, sc = c0 / BLK;
                if (gr < R && sc < S)
                    *reinterpret_cast<uint16_t*>(scales_r + sf_offset(gr, sc, s_tiles_r)) =
                        *reinterpret_cast<const uint16_t*>(&sf_row[rr * NBC]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// NVFP4 tensor amax, just in time: max over finite |x|.  Each CTA reduces its
// share and folds RN(amax_cta / 2688) into the tensor-scale slot with one
// atomicMax on the FP32 bit pattern (for non-negative floats the integer
// order is the float order).  A persistent grid sweeps the tensor from its
// end to its start in NW-word chunks (8 words: one 32-byte load), so that
// the quantize pass, which runs forward, first meets the part read last and
// still held in L2.
// ---------------------------------------------------------------------------
constexpr int kAmaxThreads = 256;
constexpr int kAmaxUnroll = 4;

template <int NW>
__device__ __forceinline__ void ld_chunk(const uint32_t* p, uint32_t* w) {
    if (NW == 8) {
        ld_v8(p, w);
    } else {
        const uint4 v = ld_stream(reinterpret_cast<const uint4*>(p));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
}

// running max of the finite |x| of one chunk (a chunk holding a non-finite
// value can still hold finite ones)
template <int NW>
__device__ __forceinline__ void amax_chunk(uint32_t& am, const uint32_t* w) {
    uint32_t m;
    if (NW == 8)
        m = bmax2(bmax2(bmax2(w[0], w[1]), bmax2(w[2], w[3])), bmax2(bmax2(w[4], w[5]), bmax2(w[6], w[7])));
    else
        m = bmax2(bmax2(w[0], w[1]), bmax2(w[2], w[3]));
    m = bmax2(m, __byte_perm(m, 0, 0x1032)) & 0x7FFFu;
    if (m < 0x7F80u) {
        am = max(am, m);
        return;
    }
#pragma unroll
    for (int k = 0; k < NW; k++) {
        const uint32_t lo = w[k] & 0x7FFFu, hi = (w[k] >> 16) & 0x7FFFu;
        if (lo < 0x7F80u) am = max(am, lo);
        if (hi < 0x7F80u) am = max(am, hi);
    }
}

template <int NW>
__global__ void __launch_bounds__(kAmaxThreads)
amax_kernel(const uint32_t* __restrict__ src, int64_t nchunks, unsigned* __restrict__ ts_bits) {
    // the quantize grid may be scheduled now; it waits for this grid's end
    pdl_launch_dependents();
    uint32_t am = 0;
    const int64_t stride = (int64_t)gridDim.x * kAmaxThreads;
    const uint32_t* last = src + (nchunks - 1) * NW;         // chunk i is read at last - i NW
    int64_t i = (int64_t)blockIdx.x * kAmaxThreads + threadIdx.x;
    for (; i + (kAmaxUnroll - 1) * stride < nchunks; i += kAmaxUnroll * stride) {
        uint32_t w[kAmaxUnroll][NW];
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; u++) ld_chunk<NW>(last - (i + u * stride) * NW, w[u]);
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; u++) amax_chunk<NW>(am, w[u]);
    }
    for (; i < nchunks; i += stride) {
        uint32_t w[NW];
        ld_chunk<NW>(last - i * NW, w);
        amax_chunk<NW>(am, w);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
    __shared__ uint32_t red[kAmaxThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = am;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < kAmaxThreads / 32; k++) m = max(m, red[k]);
        if (m) atomicMax(ts_bits, __float_as_uint(__fdiv_rn(__uint_as_float(m << 16), 2688.0f)));
    }
}

// ---------------------------------------------------------------------------
// Row-wise NVFP4 pass: just in time as the programmatic dependent of the
// amax pass (it waits before it reads the tensor scale), or with delayed
// scaling.  One 768-thread CTA per SM owns a contiguous share of the blocks;
// its warps take 64-block items (two blocks per lane) from a shared-memory
// counter, so that warps the scheduler favours do more of the work instead
// of idling the SM at the end (clock traces of a static split showed CTAs
// on one SM finishing up to 10 us apart).
// ---------------------------------------------------------------------------
constexpr int kNvPassThreads = 768;
constexpr int kNvPassWarps = kNvPassThreads / 32;

// the next item of this CTA's share for the calling warp (lane 0 takes it)
__device__ __forceinline__ unsigned take_item(unsigned* counter) {
    unsigned v = 0;
    if ((threadIdx.x & 31) == 0) v = atomicAdd(counter, 1u);
    return __shfl_sync(0xFFFFFFFFu, v, 0);
}

template <bool DELAYED, bool V8, typename IDX>
__global__ void __launch_bounds__(kNvPassThreads, 1)
quantize_rows_nv_pass_kernel(const uint8_t* __restrict__ src, int64_t nblocks, uint32_t blocks_per_row,
                             DivU32 div_bpr, int64_t s_tiles, uint8_t* __restrict__ codes,
                             uint8_t* __restrict__ scales, const NvScale nv) {
    __shared__ float2 tab[128];
    __shared__ unsigned counter;
    const unsigned G = gridDim.x, cta = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (DELAYED) pdl_launch_dependents();       // the history update may be scheduled now
    if (tid == 0) counter = kNvPassWarps;           // warp w starts on item w
    const IDX nb = (IDX)nblocks;
    const IDX n_items = (IDX)((nblocks + 63) / 64);
    const IDX i0 = (IDX)((int64_t)n_items * cta / G), i1 = (IDX)((int64_t)n_items * (cta + 1) / G);
    IDX it = i0 + warp;
    uint32_t w[16];
    // the input is not written by the amax pass: its first load may precede the wait
    if (it < i1) ld_nv_pair<V8>(src, (int64_t)(it * 64 + 2 * lane), nblocks, w);
    if (!DELAYED) pdl_wait();
    const float s_t = nv_scale_of(nv);
    if (!DELAYED && cta == 0 && tid == 0) nv_publish_scale(nv, s_t);
    const NvT nt = nv_tensor_consts(s_t);
    if (tid < 128) tab[tid] = nv_scale_entry(tid, s_t);
    __syncthreads();
    const bool vec_sf = (blocks_per_row & 3u) == 0;
    uint32_t acc = 0;                 // delayed scaling: running amax of this tensor
    while (it < i1) {
        const IDX nx = i0 + take_item(&counter);
        uint32_t wn[16];
        if (nx < i1) ld_nv_pair<V8>(src, (int64_t)(nx * 64 + 2 * lane), nblocks, wn);
        const IDX b = it * 64 + 2 * lane;
        uint32_t sb[2], out[4];
#pragma unroll
        for (int u = 0; u < 2; u++) {
            const uint32_t am = block_absmax(w + 8 * u);
            if (DELAYED && b + u < nb) nv_acc_group(acc, am, w + 8 * u, 8);
            sb[u] = nv_quantize_block(w + 8 * u, am, nt, tab, out + 2 * u);
        }
        if (b + 1 < nb)
            *reinterpret_cast<uint4*>(codes + (size_t)b * 8) = make_uint4(out[0], out[1], out[2], out[3]);
        else if (b < nb)
            *reinterpret_cast<uint2*>(codes + (size_t)b * 8) = make_uint2(out[0], out[1]);
        uint32_t r, j;
        if (sizeof(IDX) == 4) {
            r = div_u32((uint32_t)b, div_bpr);
            j = (uint32_t)b - r * blocks_per_row;
        } else {
            r = (uint32_t)(b / blocks_per_row);
            j = (uint32_t)(b - (IDX)r * blocks_per_row);
        }
        const uint32_t pair = sb[0] | (sb[1] << 8);
        const uint32_t next = __shfl_down_sync(0xFFFFFFFFu, pair, 1);
        if (vec_sf) {
            if ((lane & 1) == 0 && b < nb)
                *reinterpret_cast<uint32_t*>(scales + sf_offset(r, j, s_tiles)) = pair | (next << 16);
        } else {
            if (b < nb) scales[sf_offset(r, j, s_tiles)] = (uint8_t)sb[0];
            if (b + 1 < nb) {
                const bool wrap = j + 1 == blocks_per_row;
                scales[sf_offset(wrap ? r + 1 : r, wrap ? 0 : j + 1, s_tiles)] = (uint8_t)sb[1];
            }
        }
#pragma unroll
        for (int k = 0; k < 16; k++) w[k] = wn[k];
        it = nx;
    }
    if (DELAYED) nv_acc_flush(nv, acc);
}

// Delayed scaling, after the quantize pass: the outputs get the tensor scale
// the pass used (from the history as it stood), and the history takes this
// tensor's amax at the front, dropping its oldest entry.  Launched as the
// pass's programmatic dependent: it may be resident while the pass runs and
// waits here for the pass's end.
__global__ void nv_delayed_finalize_kernel(float* hist, int n, float* ts0, float* ts1) {
    pdl_wait();
    const float s = nv_history_scale(hist, n);
    const float amax = __uint_as_float(*reinterpret_cast<const unsigned*>(ts0));
    for (int i = n - 1; i > 0; i--) hist[i] = hist[i - 1];
    hist[0] = amax;
    *ts0 = s;
    if (ts1) *ts1 = s;
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
// Launches kernel k; with `dependent` as a programmatic dependent of the
// kernel before it on the stream (the amax pass before a quantize kernel, the
// quantize pass before the history update): k may be scheduled while that
// kernel still runs and waits for its end in pdl_wait.
template <typename... P, typename... A>
static cudaError_t launch_k(bool dependent, void (*k)(P...), dim3 grid, unsigned threads, cudaStream_t st,
                            A... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

// CTAs of k (256 threads) resident on one SM, asked once per kernel
template <typename K>
static int resident_ctas(K k, int fallback) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kRowThreads, 0) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = fallback;
    }
    return n;
}
template <int FMT>
static cudaError_t launch_rows(const void* src, int64_t R, int64_t C, uint8_t* codes, uint8_t* scales,
                               const NvScale& nv, cudaStream_t st, int num_sms) {
    const bool wide = ((reinterpret_cast<uintptr_t>(src) & 31) == 0) &&
                      (is_fp4(FMT) || (reinterpret_cast<uintptr_t>(codes) & 31) == 0);
    if (FMT != kNVFP4 && wide) {
        // persistent grid: as many CTAs as fit on the SMs at once
        static int resident = 0;
        if (resident == 0 &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, quantize_rows_wide_kernel<FMT == kNVFP4 ? kE4M3 : FMT>,
                                                          kRowThreads, 0) != cudaSuccess)
            resident = 4;
        if (resident < 1) resident = 1;
        const int64_t nblocks = R * C / 32;
        const int64_t per_cta = (int64_t)kRowThreads * kWideUnroll;
        int64_t grid = (nblocks + per_cta - 1) / per_cta;
        if (grid > (int64_t)num_sms * resident) grid = (int64_t)num_sms * resident;
        if (grid < 1) grid = 1;
        const int64_t S = C / 32;
        quantize_rows_wide_kernel<FMT == kNVFP4 ? kE4M3 : FMT><<<(unsigned)grid, kRowThreads, 0, st>>>(
            reinterpret_cast<const uint8_t*>(src), nblocks, (uint32_t)S, (S + 3) / 4, codes, scales);
        return cudaGetLastError();
    }
    const int64_t nchunks = R * C / 8;
    const int64_t per_cta = (int64_t)kRowThreads * kRowUnroll;
    int64_t grid = (nchunks + per_cta - 1) / per_cta;
    grid = grid < (int64_t)num_sms * 8 ? grid : (int64_t)num_sms * 8;
    if (grid < 1) grid = 1;
    const int64_t S = C / block_of(FMT);
    quantize_rows_kernel<FMT><<<(unsigned)grid, kRowThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(src), nchunks, (uint32_t)S, (S + 3) / 4, codes, scales, nv);
    return cudaGetLastError();
}

template <int FMT>
static cudaError_t launch_tile(const void* src, int64_t R, int64_t C, int axis,
                               uint8_t* cr, uint8_t* sr, uint8_t* cc, uint8_t* sc,
                               const NvScale& nv, cudaStream_t st) {
    const int BLK = block_of(FMT);
    const int64_t str = (C / BLK + 3) / 4, stc = (R / BLK + 3) / 4;
    const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
    const bool after_amax = FMT == kNVFP4 && !nv.history;
    dim3 grid((unsigned)((C + kTileCols - 1) / kTileCols), (unsigned)((R + kTile - 1) / kTile));
    if (axis == 3)
        return launch_k(after_amax, quantize_tile_kernel<FMT, true, true, kTileCols>, grid, 2 * kTileCols, st,
                        s, R, C, cr, sr, str, cc, sc, stc, nv);
    return launch_k(after_amax, quantize_tile_kernel<FMT, false, true, kTileCols>, grid, 2 * kTileCols, st,
                    s, R, C, cr, sr, str, cc, sc, stc, nv);
}

cudaError_t run_quantize(const QuantizeArgs& a, cudaStream_t st) {
    cudaError_t e;
    const int64_t R = a.rows, C = a.cols;
    // zero the padding of the tiled scale buffers when there is any
    if (a.row_scales && a.row_scales_pad) {
        if ((e = cudaMemsetAsync(a.row_scales, 0, a.row_scales_bytes, st)) != cudaSuccess) return e;
    }
    if (a.col_scales && a.col_scales_pad) {
        if ((e = cudaMemsetAsync(a.col_scales, 0, a.col_scales_bytes, st)) != cudaSuccess) return e;
    }
    unsigned* slot = nullptr;
    NvScale nv{};
    if (a.fmt == kNVFP4) {
        // just in time the slot collects the tensor scale, delayed the tensor amax
        slot = reinterpret_cast<unsigned*>(a.axis & 1 ? a.row_ts : a.col_ts);
        if ((e = cudaMemsetAsync(slot, 0, sizeof(float), st)) != cudaSuccess) return e;
    }
    const bool src32 = (reinterpret_cast<uintptr_t>(a.src) & 31) == 0;
    if (a.fmt == kNVFP4 && a.history) {
        // delayed scaling: no amax pass; the quantize pass accumulates the amax
        nv.history = a.history;
        nv.hist_len = a.hist_len;
        nv.amax_acc = slot;
    } else if (a.fmt == kNVFP4) {
        nv.ts_bits = slot;
        nv.ts_other = a.axis == 3 ? a.col_ts : nullptr;
        // persistent grid, as many CTAs as fit on the SMs at once
        static const int res8 = resident_ctas(amax_kernel<8>, 4), res4 = resident_ctas(amax_kernel<4>, 4);
        const int NW = src32 ? 8 : 4;
        const int64_t nchunks = R * C * 2 / (NW * 4);
        int64_t grid = (nchunks + kAmaxThreads * kAmaxUnroll - 1) / (kAmaxThreads * kAmaxUnroll);
        const int64_t cap = (int64_t)a.num_sms * (src32 ? res8 : res4);
        if (grid > cap) grid = cap;
        if (grid < 1) grid = 1;
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(a.src);
        if (src32)
            amax_kernel<8><<<(unsigned)grid, kAmaxThreads, 0, st>>>(s32, nchunks, slot);
        else
            amax_kernel<4><<<(unsigned)grid, kAmaxThreads, 0, st>>>(s32, nchunks, slot);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.axis == 1) {
        switch (a.fmt) {
        case kE4M3: e = launch_rows<kE4M3>(a.src, R, C, a.row_codes, a.row_scales, nv, st, a.num_sms); break;
        case kE5M2: e = launch_rows<kE5M2>(a.src, R, C, a.row_codes, a.row_scales, nv, st, a.num_sms); break;
        case kMXFP4: e = launch_rows<kMXFP4>(a.src, R, C, a.row_codes, a.row_scales, nv, st, a.num_sms); break;
        default: {
            const int64_t nblocks = R * C / 16;
            const int64_t S = C / 16;
            const uint8_t* s8 = reinterpret_cast<const uint8_t*>(a.src);
            const DivU32 dv = make_div_u32((uint32_t)S);
            const bool small = nblocks < (1ll << 32) - 64 * (int64_t)a.num_sms;   // item indices stay in 32 bits
            // one CTA per SM; just in time as the programmatic dependent of the amax pass
            int64_t g = a.num_sms;
            const int64_t items = (nblocks + 63) / 64;
            if (g > items) g = items;
            if (g < 1) g = 1;
            const bool jit = !nv.history;
            auto k = jit ? (src32 ? (small ? quantize_rows_nv_pass_kernel<false, true, uint32_t>
                                           : quantize_rows_nv_pass_kernel<false, true, int64_t>)
                                  : (small ? quantize_rows_nv_pass_kernel<false, false, uint32_t>
                                           : quantize_rows_nv_pass_kernel<false, false, int64_t>))
                         : (src32 ? (small ? quantize_rows_nv_pass_kernel<true, true, uint32_t>
                                           : quantize_rows_nv_pass_kernel<true, true, int64_t>)
                                  : (small ? quantize_rows_nv_pass_kernel<true, false, uint32_t>
                                           : quantize_rows_nv_pass_kernel<true, false, int64_t>));
            e = launch_k(jit, k, dim3((unsigned)g), kNvPassThreads, st, s8, nblocks, (uint32_t)S, dv, (S + 3) / 4,
                         a.row_codes, a.row_scales, nv);
            break;
        }
        }
    } else {
        switch (a.fmt) {
        case kE4M3: e = launch_tile<kE4M3>(a.src, R, C, a.axis, a.row_codes, a.row_scales, a.col_codes, a.col_scales, nv, st); break;
        case kE5M2: e = launch_tile<kE5M2>(a.src, R, C, a.axis, a.row_codes, a.row_scales, a.col_codes, a.col_scales, nv, st); break;
        case kMXFP4: e = launch_tile<kMXFP4>(a.src, R, C, a.axis, a.row_codes, a.row_scales, a.col_codes, a.col_scales, nv, st); break;
        default: e = launch_tile<kNVFP4>(a.src, R, C, a.axis, a.row_codes, a.row_scales, a.col_codes, a.col_scales, nv, st); break;
        }
    }
    if (e != cudaSuccess) return e;
    if (a.fmt == kNVFP4 && a.history) {
        float* other = (a.axis == 3) ? a.col_ts : nullptr;
        if ((e = launch_k(true, nv_delayed_finalize_kernel, dim3(1), 1, st, a.history, (int)a.hist_len,
                          reinterpret_cast<float*>(slot), other)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace bsq
