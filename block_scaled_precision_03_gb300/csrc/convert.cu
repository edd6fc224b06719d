// MXFP4 re-encodes and exact dequantization:
//   repack_kernel        MXFP4 -> MXFP8 E4M3 rows, plain or with per-expert
//                        padded scales for the grouped GEMM
//   repack_1x128_kernel  MXFP4 -> FP8 E4M3 with 1 x 128 blocks
//   repack_col_kernel    FP4RowToFP8Col: MXFP4 rows -> MXFP8 E4M3 columns
//   dequant_kernel       any format -> FP32 / BF16, rounded once
//
// Re-encode ("Practical FP4 Training for Large-Scale MoE Models on Hopper
// GPUs", section 2, "Algoritmo de Conversao Direta" and kernel
// FP4RowToFP8Row): the conversion stays in the integer domain.  For a
// 32-block with scale byte s and largest code magnitude exponent e_c the
// new scale byte is s + e_c - 8 (floored at 0, the E8M0 minimum); each E2M1
// nibble keeps its sign and mantissa bit and its exponent moves by the
// shift between the two scales, so every value is carried over exactly.
// There is no BF16 or FP32 intermediate.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace bsq {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// 8 E2M1 nibbles of w -> 8 E4M3 bytes given the magnitude table (lut_lo =
// bytes for magnitudes 0..3, lut_hi = 4..7).  The magnitudes index the table
// directly (a byte permute reads its 4 selector nibbles from the low 16
// bits); the sign bits are moved to bit 7 of their bytes in place (odd
// nibbles' signs already sit at bit 7 of a byte, even nibbles' after a
// 4-bit shift) and interleaved with two more byte permutes.
__device__ __forceinline__ uint2 remap8(uint32_t w, uint32_t lut_lo, uint32_t lut_hi) {
    const uint32_t m = w & 0x77777777u;
    const uint32_t s_even = (w << 4) & 0x80808080u;      // nibbles 0, 2, 4, 6
    const uint32_t s_odd = w & 0x80808080u;              // nibbles 1, 3, 5, 7
    const uint32_t lo = prmt(lut_lo, lut_hi, m) | prmt(s_even, s_odd, 0x5140u);
    const uint32_t hi = prmt(lut_lo, lut_hi, m >> 16) | prmt(s_even, s_odd, 0x7362u);
    return make_uint2(lo, hi);
}

// Expert offsets for the per-expert padded scale layout of the output: expert
// g's scale rows start at P_g = sum over earlier experts of their row counts
// rounded up to 128 (clamped offsets, as in the grouped GEMM).
struct ExpertRows {
    const int64_t* offsets;        // device, num_groups + 1 (nullptr: plain layout)
    int32_t num_groups;
};
constexpr int kMaxExperts = kMaxGroups;

// One 32-block: 16 code bytes in, 32 code bytes and the new scale byte out.
__device__ __forceinline__ void repack_block(const uint4 w, const uint32_t s, uint4& o0, uint4& o1, uint32_t& ns) {
    if (s == 0xFF) {
        ns = 0xFF;
        o0 = o1 = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        return;
    }
    // exponent of the largest magnitude index m (0.5 -> -1, 1|1.5 -> 0, 2|3 -> 1,
    // 4|6 -> 2) is (m >> 1) - 1, and m >> 1 is 3 if some nibble has bits 1 and
    // 2 set, else 2 if some nibble has bit 2, else 1 if some has bit 1, else 0:
    // two OR reductions instead of a byte-wise maximum
    const uint32_t any = w.x | w.y | w.z | w.w;
    const uint32_t both = (w.x & (w.x >> 1)) | (w.y & (w.y >> 1)) | (w.z & (w.z >> 1)) | (w.w & (w.w >> 1));
    uint32_t lut_lo = 0, lut_hi = 0;
    if ((any & 0x77777777u) == 0) {
        ns = 0;                                  // all-zero block: e = -127
    } else {
        const int lvl = (both & 0x22222222u) ? 3 : (any & 0x44444444u) ? 2 : (any & 0x22222222u) ? 1 : 0;
        const int e_c = lvl - 1;
        int nb = (int)s + e_c - 8;
        if (nb < 0) nb = 0;
        ns = (uint32_t)nb;
        const uint32_t E = (uint32_t)((int)s - nb + 7);   // biased E4M3 exponent of magnitude 1.0
        // E4M3 bytes of magnitudes 0, 0.5, 1, 1.5 | 2, 3, 4, 6 scaled by 2^(s - nb)
        lut_lo = ((E - 1) << 11) | ((E << 3) << 16) | (((E << 3) | 4u) << 24);
        lut_hi = ((E + 1) << 3) | ((((E + 1) << 3) | 4u) << 8) | (((E + 2) << 3) << 16) |
                 ((((E + 2) << 3) | 4u) << 24);
    }
    const uint2 a = remap8(w.x, lut_lo, lut_hi), bb = remap8(w.y, lut_lo, lut_hi);
    const uint2 c = remap8(w.z, lut_lo, lut_hi), d = remap8(w.w, lut_lo, lut_hi);
    o0 = make_uint4(a.x, a.y, bb.x, bb.y);
    o1 = make_uint4(c.x, c.y, d.x, d.y);
}

// One 32-byte store (both halves of a converted block): a warp then writes
// 1 KB of whole sectors per instruction instead of two half-filled passes.
// The address must be 32-byte aligned.
__device__ __forceinline__ void st_global_32B(uint4* p, const uint4 a, const uint4 b) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
                 "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

constexpr int kRepackThreads = 256;
constexpr int kRepackUnroll = 2;     // 32-blocks in flight per thread

// Each CTA converts one contiguous range of 32-blocks (row-major order), a
// thread taking every 256th block, two per iteration so that two 16-byte
// loads are in flight (the kernel is bound by memory latency times the loads
// in flight per SM; one, four or eight per thread, with their register
// counts and resident CTAs, measured slower).  Rows grow along a thread's walk, so in the grouped
// form its expert only moves forward (o_s / p_s: expert row starts and
// padded scale row starts, built per CTA from the clamped offsets).  The
// grouped form also writes every other byte of the scale buffer (cap_bytes)
// as zero, each byte by exactly one thread: the pad columns of live rows,
// the rows between an expert's last row and its next 128-row boundary, and
// the whole tiles past the last expert.  Rows past the last offset belong to
// no expert: their codes are converted, their scales have no slot.  WIDE:
// the output codes are 32-byte aligned and each block is one 32-byte store.
template <bool GROUPED, bool WIDE>
__global__ void __launch_bounds__(kRepackThreads)
repack_kernel(const uint4* __restrict__ in, const uint8_t* __restrict__ sin, uint4* __restrict__ out,
              uint8_t* __restrict__ sout, int64_t nblocks, int64_t per_cta, uint32_t bpr, int64_t s_tiles, int64_t R,
              const ExpertRows er, int64_t cap_bytes) {
    __shared__ int32_t o_s[kMaxExperts + 1], p_s[kMaxExperts + 1];
    const int64_t b_lo = (int64_t)blockIdx.x * per_cta;
    const int64_t b_hi = min(nblocks, b_lo + per_cta);
    int g = 0;
    if (GROUPED) {
        if (threadIdx.x < 32) {
            int carry = 0, prev = 0;
            for (int g0 = 0; g0 <= er.num_groups; g0 += 32) {
                const int gi = g0 + (int)threadIdx.x;
                int o = 0;
                if (gi <= er.num_groups) o = gi == 0 ? 0 : clamp_rows(er.offsets[gi], 0, R);
                // offsets are non-decreasing after a running max
                int om = o;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int u = __shfl_up_sync(0xffffffffu, om, d);
                    if ((int)threadIdx.x >= d) om = max(om, u);
                }
                om = max(om, prev);
                const int lo = __shfl_up_sync(0xffffffffu, om, 1);
                const int lo_g = threadIdx.x == 0 ? prev : lo;          // start of expert gi - 1
                int padded = (gi >= 1 && gi <= er.num_groups) ? (om - lo_g + 127) / 128 * 128 : 0;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int u = __shfl_up_sync(0xffffffffu, padded, d);
                    if ((int)threadIdx.x >= d) padded += u;
                }
                if (gi <= er.num_groups) { o_s[gi] = om; p_s[gi] = carry + padded; }
                carry += __shfl_sync(0xffffffffu, padded, 31);
                prev = __shfl_sync(0xffffffffu, om, 31);
            }
        }
        __syncthreads();
        // expert of this CTA's first row: the last g < num_groups with o_s[g] <= row
        // (rows at or past o_s[num_groups] stay with the last expert)
        const int r0 = (int)(b_lo / bpr);
        int lo = 0, hi = er.num_groups;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (o_s[mid] <= r0) lo = mid;
            else hi = mid;
        }
        g = lo;
    }
    const int o_end = GROUPED ? o_s[er.num_groups] : 0;
    // expert cursor: first row of the next expert, scale row shift of this one
    int next_row = 0, shift = 0;
    if (GROUPED) {
        next_row = g + 1 < er.num_groups ? o_s[g + 1] : INT_MAX;
        shift = p_s[g] - o_s[g];
    }
    // block coordinates (row r, block column j) advance by kRepackThreads
    // blocks per step without a division
    const int64_t b_first = b_lo + threadIdx.x;
    uint32_t r = (uint32_t)(b_first / bpr);
    uint32_t j = (uint32_t)(b_first - (int64_t)r * bpr);
    const uint32_t dq = (uint32_t)kRepackThreads / bpr, dr = (uint32_t)kRepackThreads % bpr;
    for (int64_t b0 = b_first; b0 < b_hi; b0 += kRepackUnroll * kRepackThreads) {
        uint4 w[kRepackUnroll];
        uint32_t s[kRepackUnroll], rr[kRepackUnroll], jj[kRepackUnroll];
#pragma unroll
        for (int u = 0; u < kRepackUnroll; ++u) {
            const int64_t b = b0 + u * kRepackThreads;
            rr[u] = r;
            jj[u] = j;
            if (b < b_hi) {
                w[u] = in[b];
                s[u] = sin[sf_offset(r, j, s_tiles)];
            }
            j += dr;
            r += dq;
            if (j >= bpr) { j -= bpr; ++r; }
        }
#pragma unroll
        for (int u = 0; u < kRepackUnroll; ++u) {
            const int64_t b = b0 + u * kRepackThreads;
            if (b >= b_hi) break;
            uint4 o0, o1;
            uint32_t ns;
            repack_block(w[u], s[u], o0, o1, ns);
            if (WIDE) {
                st_global_32B(out + 2 * b, o0, o1);
            } else {
                out[2 * b] = o0;
                out[2 * b + 1] = o1;
            }
            if (GROUPED) {
                while ((int)rr[u] >= next_row) {
                    ++g;
                    next_row = g + 1 < er.num_groups ? o_s[g + 1] : INT_MAX;
                    shift = p_s[g] - o_s[g];
                }
                if ((int)rr[u] < o_end) {
                    const int64_t off_out = sf_offset((int64_t)rr[u] + shift, jj[u], s_tiles);
                    sout[off_out] = (uint8_t)ns;
                    if (jj[u] == bpr - 1)      // pad columns of the row's last 4-column group
                        for (int c = 1; c < (int)(4 * s_tiles - bpr) + 1; ++c) sout[off_out + c] = 0;
                }
            } else {
                sout[sf_offset(rr[u], jj[u], s_tiles)] = (uint8_t)ns;
            }
        }
    }
    if (GROUPED) {
        // rows from an expert's last row up to its next 128-row boundary
        for (int gg = (int)blockIdx.x; gg < er.num_groups; gg += (int)gridDim.x) {
            const int first = p_s[gg] + (o_s[gg + 1] - o_s[gg]);
            const int units = (p_s[gg + 1] - first) * (int)s_tiles;
            for (int t = (int)threadIdx.x; t < units; t += kRepackThreads) {
                const int row = first + t / (int)s_tiles, cg = t % (int)s_tiles;
                *reinterpret_cast<uint32_t*>(sout + sf_offset(row, 4 * cg, s_tiles)) = 0u;
            }
        }
        // whole tiles past the last expert (p_s[num_groups] is a multiple of 128)
        const int64_t tail_lo = (int64_t)(p_s[er.num_groups] >> 7) * s_tiles * 512;
        const int64_t n16 = (cap_bytes - tail_lo) / 16;
        uint4* tail = reinterpret_cast<uint4*>(sout + tail_lo);
        for (int64_t i = (int64_t)blockIdx.x * kRepackThreads + threadIdx.x; i < n16;
             i += (int64_t)gridDim.x * kRepackThreads)
            tail[i] = make_uint4(0u, 0u, 0u, 0u);
    }
}

cudaError_t run_repack(const RepackArgs& a, cudaStream_t st) {
    cudaError_t e;
    if (a.scales_pad && (e = cudaMemsetAsync(a.out_scales, 0, a.scales_bytes, st)) != cudaSuccess) return e;
    const int64_t nblocks = a.rows * (a.cols / 32);
    // one wave: as many CTAs as are resident on the SMs at once, each a
    // contiguous range of whole warps' worth of blocks
    const bool wide = (reinterpret_cast<uintptr_t>(a.out_codes) & 31) == 0;
    const int variant = (a.num_groups > 0 ? 2 : 0) + (wide ? 1 : 0);
    static int resident[4] = {0, 0, 0, 0};
    int& res = resident[variant];
    if (res == 0) {
        cudaError_t oe;
        switch (variant) {
            case 0: oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&res, repack_kernel<false, false>, kRepackThreads, 0); break;
            case 1: oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&res, repack_kernel<false, true>, kRepackThreads, 0); break;
            case 2: oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&res, repack_kernel<true, false>, kRepackThreads, 0); break;
            default: oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&res, repack_kernel<true, true>, kRepackThreads, 0); break;
        }
        if (oe != cudaSuccess || res < 1) res = 1;
    }
    int64_t grid = (int64_t)a.num_sms * res;
    const int64_t per_min = kRepackThreads;
    if (grid * per_min > nblocks) grid = (nblocks + per_min - 1) / per_min;
    if (grid < 1) grid = 1;
    int64_t per_cta = (nblocks + grid - 1) / grid;
    per_cta = (per_cta + 31) / 32 * 32;
    const uint32_t bpr = (uint32_t)(a.cols / 32);
    const ExpertRows er{a.offsets, a.num_groups};
    const uint4* in = reinterpret_cast<const uint4*>(a.in_codes);
    uint4* out = reinterpret_cast<uint4*>(a.out_codes);
    const int64_t st_ = (bpr + 3) / 4, cap = (int64_t)a.scales_bytes;
    const dim3 g((unsigned)grid), b(kRepackThreads);
    switch (variant) {
        case 0: repack_kernel<false, false><<<g, b, 0, st>>>(in, a.in_scales, out, a.out_scales, nblocks, per_cta, bpr, st_, a.rows, er, 0); break;
        case 1: repack_kernel<false, true><<<g, b, 0, st>>>(in, a.in_scales, out, a.out_scales, nblocks, per_cta, bpr, st_, a.rows, er, 0); break;
        case 2: repack_kernel<true, false><<<g, b, 0, st>>>(in, a.in_scales, out, a.out_scales, nblocks, per_cta, bpr, st_, a.rows, er, cap); break;
        default: repack_kernel<true, true><<<g, b, 0, st>>>(in, a.in_scales, out, a.out_scales, nblocks, per_cta, bpr, st_, a.rows, er, cap); break;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// MXFP4 -> FP8 E4M3 with 1 x 128 blocks (same page and section: the Hopper
// FP8 block holds 128 elements; the conversion takes the largest of the four
// FP4 block scales and moves each element's exponent to it).  A thread
// converts one 32-block.  The four scale bytes of its 128-group are one
// 32-bit word of the tiled layout (scale columns 4g .. 4g + 3 of a row sit
// side by side); S is their largest byte, s the block's own.  Each value is
// code * 2^(s - S), formed as an exact half product (E2M1 -> f16x2 times
// 2^(s - S), a normal half for s - S >= -14; below that every value of the
// block is under half of E4M3's smallest subnormal, so the power is taken
// as 0) and rounded once by the f16x2 -> E4M3x2 conversion.  A NaN scale
// (0xFF, the largest byte) makes the whole group NaN.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void h2_of_e2m1x8(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2, uint32_t& h3) {
    asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\tmov.b32 {t0, t1, t2, t3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, t0;\n\tcvt.rn.f16x2.e2m1x2 %1, t1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, t2;\n\tcvt.rn.f16x2.e2m1x2 %3, t3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2_rn(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// f16x2 -> two E4M3 bytes (low half in the low byte), one rounding (RNE).
__device__ __forceinline__ uint32_t e4m3x2_of_h2(uint32_t h) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
    return r;
}
// 8 E2M1 codes (element k in nibble k) times the f16x2 power P2 -> 8 E4M3 bytes
__device__ __forceinline__ uint2 e4m3x8_of_e2m1x8(uint32_t w, uint32_t P2) {
    uint32_t h0, h1, h2, h3;
    h2_of_e2m1x8(w, h0, h1, h2, h3);
    const uint32_t e0 = e4m3x2_of_h2(hmul2_rn(h0, P2)), e1 = e4m3x2_of_h2(hmul2_rn(h1, P2));
    const uint32_t e2 = e4m3x2_of_h2(hmul2_rn(h2, P2)), e3 = e4m3x2_of_h2(hmul2_rn(h3, P2));
    return make_uint2(prmt(e0, e1, 0x5410u), prmt(e2, e3, 0x5410u));
}

template <bool WIDE>
__global__ void __launch_bounds__(kRepackThreads)
repack_1x128_kernel(const uint4* __restrict__ in, const uint8_t* __restrict__ sin, uint4* __restrict__ out,
                    uint8_t* __restrict__ sout, int64_t nblocks, int64_t per_cta, uint32_t bpr, int64_t s_tiles,
                    uint32_t groups) {
    const int64_t b_lo = (int64_t)blockIdx.x * per_cta;
    const int64_t b_hi = min(nblocks, b_lo + per_cta);
    const int64_t b_first = b_lo + threadIdx.x;
    uint32_t r = (uint32_t)(b_first / bpr);
    uint32_t j = (uint32_t)(b_first - (int64_t)r * bpr);
    const uint32_t dq = (uint32_t)kRepackThreads / bpr, dr = (uint32_t)kRepackThreads % bpr;
    for (int64_t b = b_first; b < b_hi; b += kRepackThreads) {
        const uint4 w = in[b];
        const uint32_t g = j >> 2;
        uint32_t word = *reinterpret_cast<const uint32_t*>(sin + sf_offset(r, 4 * g, s_tiles));
        const uint32_t nin = bpr - 4 * g;                  // blocks of this group in the row
        if (nin < 4) word &= (1u << (8 * nin)) - 1u;
        const uint32_t m4 = __vmaxu4(word, word >> 16);
        const uint32_t S = max(m4 & 0xFFu, (m4 >> 8) & 0xFFu);
        const uint32_t s = (word >> (8 * (j & 3))) & 0xFFu;
        uint4 o0, o1;
        if (S == 0xFFu) {
            o0 = o1 = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        } else {
            const int d = (int)s - (int)S;
            const uint32_t P = d >= -14 ? (uint32_t)(d + 15) << 10 : 0u;
            const uint32_t P2 = P | (P << 16);
            const uint2 a = e4m3x8_of_e2m1x8(w.x, P2), bb = e4m3x8_of_e2m1x8(w.y, P2);
            const uint2 c = e4m3x8_of_e2m1x8(w.z, P2), dd = e4m3x8_of_e2m1x8(w.w, P2);
            o0 = make_uint4(a.x, a.y, bb.x, bb.y);
            o1 = make_uint4(c.x, c.y, dd.x, dd.y);
        }
        if (WIDE) {
            st_global_32B(out + 2 * b, o0, o1);
        } else {
            out[2 * b] = o0;
            out[2 * b + 1] = o1;
        }
        if ((j & 3) == 0) sout[(int64_t)r * groups + g] = (uint8_t)S;
        j += dr;
        r += dq;
        if (j >= bpr) { j -= bpr; ++r; }
    }
}

cudaError_t run_repack_1x128(const RepackArgs& a, cudaStream_t st) {
    const int64_t nblocks = a.rows * (a.cols / 32);
    const bool wide = (reinterpret_cast<uintptr_t>(a.out_codes) & 31) == 0;
    static int resident[2] = {0, 0};
    int& res = resident[wide ? 1 : 0];
    if (res == 0) {
        const cudaError_t oe =
            wide ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&res, repack_1x128_kernel<true>, kRepackThreads, 0)
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&res, repack_1x128_kernel<false>, kRepackThreads, 0);
        if (oe != cudaSuccess || res < 1) res = 1;
    }
    int64_t grid = (int64_t)a.num_sms * res;
    if (grid * kRepackThreads > nblocks) grid = (nblocks + kRepackThreads - 1) / kRepackThreads;
    if (grid < 1) grid = 1;
    int64_t per_cta = (nblocks + grid - 1) / grid;
    per_cta = (per_cta + 31) / 32 * 32;
    const uint32_t bpr = (uint32_t)(a.cols / 32);
    const uint32_t groups = (bpr + 3) / 4;
    const uint4* in = reinterpret_cast<const uint4*>(a.in_codes);
    uint4* out = reinterpret_cast<uint4*>(a.out_codes);
    if (wide)
        repack_1x128_kernel<true><<<(unsigned)grid, kRepackThreads, 0, st>>>(in, a.in_scales, out, a.out_scales, nblocks,
                                                                             per_cta, bpr, (bpr + 3) / 4, groups);
    else
        repack_1x128_kernel<false><<<(unsigned)grid, kRepackThreads, 0, st>>>(in, a.in_scales, out, a.out_scales, nblocks,
                                                                              per_cta, bpr, (bpr + 3) / 4, groups);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// FP4RowToFP8Col (same page and section, kernel FP4RowToFP8Col): dequantize,
// transpose and re-quantize column-wise to MXFP8 E4M3 in one pass, without a
// BF16 intermediate.  An E2M1 magnitude index m = 1..7 is a * 2^b with
// (a, b) = (1,-1) (1,0) (3,-1) (1,1) (3,0) (1,2) (3,1); under the row scale
// byte s its value is a * 2^(b + s - 127), whose floor(log2) is
// b + [a == 3] + s - 127.  A 32-row block of one column takes the E8M0
// exponent e = clamp(max floor(log2) - 8, -127, 127) (the MX rule with
// E4M3's largest exponent 8; -127 for an all-zero block), and each element
// a * 2^(b + s - 127 - e) is formed exactly and rounded once by the
// hardware E4M3 conversion; a NaN row scale (0xFF) in the block makes the
// block NaN.  Tiles of 256 input rows x 128 input columns: the codes
// (16 KB) and the two 512-byte scale tiles that cover them are staged in
// shared memory.
// ---------------------------------------------------------------------------
constexpr int kColRows = 256;       // tile: 256 input rows x 128 input columns
constexpr int kColCols = 128;
constexpr int kColThreads = 256;    // one thread = 8 columns x 16 rows

// b + 1 of the E2M1 magnitudes, 4 bits each (index m), for the exact path
constexpr uint32_t kBexp = 0x23120100u;     // m 1..7 -> 0,1,0,2,1,3,2 (m = 0 unused)

// Exact FP32 value a * 2^t of magnitude index m (sign from the nibble) with
// t = b + s_minus_e; values below 2^-126 become 0 (E4M3 rounds them to 0).
__device__ __forceinline__ float e2m1_scaled(uint32_t n, int s_minus_e) {
    const uint32_t m = n & 7u;
    float v = 0.0f;
    if (m) {
        const int t = (int)((kBexp >> (4 * m)) & 0xFu) - 1 + s_minus_e;
        const bool three = (m & 1u) && m > 1;                              // a = 3: 1.5 * 2^(t+1)
        const int ex = three ? t + 1 : t;
        if (ex >= -126) v = __uint_as_float(((uint32_t)(ex + 127) << 23) | (three ? 0x400000u : 0u));
    }
    return (n & 8u) ? -v : v;
}

// E4M3 byte of nibble n with row scale byte sr in a block of scale byte sb.
// For m = 1..7, floor(log2 |value|) + 1 = (m >> 1) + sr - 127, so the E4M3
// exponent field is key - sb + 6 with key = (m >> 1) + sr, and the mantissa
// field is 4 for m = 3, 5, 7 (a = 3) and 0 otherwise; a field below 1 means
// E4M3's subnormal range, which the exact conversion handles.
// the rare subnormal case, out of line to keep the unrolled loops small
__device__ __noinline__ uint32_t fp8_of_nibble_exact(uint32_t n, int s_minus_e) {
    return cvt_e4m3x2(e2m1_scaled(n, s_minus_e), 0.0f) & 0xFFu;
}
__device__ __forceinline__ uint32_t fp8_of_nibble(uint32_t n, uint32_t sr, uint32_t sb) {
    const uint32_t m = n & 7u, sign = (n & 8u) << 4;
    const int E = (int)(m >> 1) + (int)sr - (int)sb + 6;
    const uint32_t normal = sign | ((uint32_t)E << 3) | (((m & 1u) && m > 1) ? 4u : 0u);
    if (m == 0) return sign;
    if (E >= 1) return normal;
    return fp8_of_nibble_exact(n, (int)sr - (int)sb);
}

// Per-nibble tables for the column maximum, indexed by the magnitude m
// through a byte permute: lev1 = (m >> 1) + 1 (0 for m = 0), and a high byte
// 0xFC for m = 0 so that a zero code becomes the 16-bit lane -1024, which
// no row scale lifts above 0.
constexpr uint32_t kLev1Lo = 0x02020100u;   // m 0..3 -> 0, 1, 2, 2
constexpr uint32_t kLev1Hi = 0x04040303u;   // m 4..7 -> 3, 3, 4, 4
constexpr uint32_t kZeroLo = 0x000000FCu;   // m 0 -> 0xFC, 1..3 -> 0
constexpr uint32_t kZeroHi = 0x00000000u;

// max(|a|, |b|) per half (the sign bit of the result is sign(a) ^ sign(b))
__device__ __forceinline__ uint32_t habsmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Layout: a thread owns one code word (8 columns) of 16 rows, half of a
// 32-row block; the two threads of a block are neighbouring lanes and
// combine their column maxima with shuffles.  The 16 code words stay in
// registers, and the row scales are staged by column block ([column
// block][row]), so a thread's 16 row scales are one 16-byte load.
//
// Blocks without a NaN row scale whose row scales lie within 14 binades
// (nearly all) take the half path: each element is formed exactly as
// code * 2^(sr - smax) in FP16 (E2M1 -> f16x2 is exact, and the factor's
// exponent field sr - smax + 15 lies in [1, 15], so the product is an exact
// half, a subnormal at worst); the column's largest |product| gives its
// largest exponent directly (floor(log2 amax) = exponent(max) + smax - 127),
// and the encode multiplies the same product by 2^(smax - sb), which makes
// the exact value code * 2^(sr - sb) whenever that factor's exponent field
// smax - sb + 15 lies in [1, 30], then rounds once (f16x2 -> E4M3).  Other
// blocks take the column maximum in the integer domain and the scalar
// encode.
__global__ void __launch_bounds__(kColThreads, 4)
repack_col_kernel(const uint8_t* __restrict__ in, const uint8_t* __restrict__ sin, int64_t R, int64_t C,
                  int64_t s_tiles_in, uint8_t* __restrict__ out, uint8_t* __restrict__ sout, int64_t s_tiles_out) {
    // codes: 256 rows x 64 bytes; row r sits at r ^ 1 where bit 4 of r is set,
    // so that a block's two threads (rows 16 apart) read opposite bank halves
    __shared__ __align__(16) uint32_t codes[kColRows * 16];
    __shared__ __align__(16) uint8_t sfr[4 * kColRows];       // row scales: [column block][row]
    const int tid = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.y * kColRows, c0 = (int64_t)blockIdx.x * kColCols;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const int idx = tid + k * kColThreads, rr = idx >> 2, ch = idx & 3;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r0 + rr < R && c0 + 32 * ch < C)
            v = *reinterpret_cast<const uint4*>(in + (r0 + rr) * (C / 2) + c0 / 2 + 16 * ch);
        *reinterpret_cast<uint4*>(&codes[(rr ^ ((rr >> 4) & 1)) * 16 + ch * 4]) = v;
    }
    // row tid's four scale bytes (the tile's column blocks 0-3) from its 128x4
    // scale tile; warp k stages rows 32 k .. 32 k + 31, the 32-row block it
    // encodes, so it also takes each column block's largest and smallest
    // row scale (a NaN scale is the largest byte), byte cb of smax4 / smin4
    uint32_t smax4, smin4;
    {
        const int band = tid >> 7;
        uint32_t v = 0;
        if (r0 + 128 * band < R)
            v = *reinterpret_cast<const uint32_t*>(sin + ((r0 / 128 + band) * s_tiles_in + c0 / 128) * 512 +
                                                   (tid & 31) * 16 + ((tid >> 5) & 3) * 4);
#pragma unroll
        for (int cb = 0; cb < 4; cb++) sfr[cb * kColRows + tid] = (uint8_t)(v >> (8 * cb));
        smax4 = smin4 = 0;
#pragma unroll
        for (int cb = 0; cb < 4; cb++) {
            const uint32_t b = (v >> (8 * cb)) & 0xFFu;
            smax4 |= __reduce_max_sync(0xFFFFFFFFu, b) << (8 * cb);
            smin4 |= __reduce_min_sync(0xFFFFFFFFu, b) << (8 * cb);
        }
    }
    __syncthreads();
    const int lane = tid & 31, rb = tid >> 5, w = lane >> 1, h = lane & 1;
    const int c = 8 * w, cb = w >> 2;                  // columns c .. c + 7, rows 32 rb + 16 h .. + 15
    if (c0 + c >= C || r0 + 32 * rb >= R) return;
    const unsigned pair = 3u << (lane & 30);
    uint32_t nb[16];
#pragma unroll
    for (int i = 0; i < 16; i++) nb[i] = codes[((32 * rb + 16 * h + i) ^ h) * 16 + w];
    const uint4 s4 = *reinterpret_cast<const uint4*>(&sfr[cb * kColRows + 32 * rb + 16 * h]);
    const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};   // row i's scale: byte i & 3 of word i >> 2
    const uint32_t smax = (smax4 >> (8 * cb)) & 0xFFu, smin = (smin4 >> (8 * cb)) & 0xFFu;
    const bool nan = smax == 0xFFu;
    const uint32_t kr = (15u - smax) * 0x04000400u;    // row factor 2^(sr - smax): sr * 0x04000400 + kr
    uint32_t SB[4];                                      // scale bytes, columns (0,1) (2,3) (4,5) (6,7)
    uint32_t Fc[4];                                      // half path: column factors 2^(smax - sb)
    bool fast = !nan && smax - smin <= 14u;
    if (fast) {
        uint32_t M[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            uint32_t fr[4];
#pragma unroll
            for (int j = 0; j < 4; j++) fr[j] = prmt(sw[q], 0u, 0x4440u | (uint32_t)j) * 0x04000400u + kr;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                uint32_t h0, h1, h2, h3;
                h2_of_e2m1x8(nb[4 * q + j], h0, h1, h2, h3);
                M[0] = habsmax2(M[0], hmul2_rn(h0, fr[j]));
                M[1] = habsmax2(M[1], hmul2_rn(h1, fr[j]));
                M[2] = habsmax2(M[2], hmul2_rn(h2, fr[j]));
                M[3] = habsmax2(M[3], hmul2_rn(h3, fr[j]));
            }
        }
        // per two columns in 16-bit lanes: scale byte = floor(log2 amax) - 8 + 127
        // = exponent field - 23 + smax (at least 0; it cannot pass 254 here); the
        // column factor's exponent field smax + 15 - sb, which must not pass 30
        // (it is at least 15: 21 unless the scale byte was raised to 0, where every
        // product stays below 2^8); an all-zero column gets scale byte 0 and the
        // field 30 (any finite factor keeps its zeros)
        const uint32_t k23 = ((smax - 23u) & 0xFFFFu) * 0x00010001u, k15 = (smax + 15u) * 0x00010001u;
        uint32_t fmax = 0;
#pragma unroll
        for (int p2 = 0; p2 < 4; p2++) {
            const uint32_t Mp = habsmax2(M[p2], __shfl_xor_sync(pair, M[p2], 1)) & 0x7FFF7FFFu;
            const uint32_t sbv = __viaddmax_s16x2((Mp >> 10) & 0x001F001Fu, k23, 0u);
            const uint32_t nz = prmt(Mp + 0x7FFF7FFFu, 0u, 0xBB99u);     // 0xFFFF per nonzero column
            SB[p2] = sbv & nz;
            const uint32_t F = ((k15 - sbv) & nz) | (0x001E001Eu & ~nz);
            fmax = __viaddmax_u16x2(F, 0u, fmax);
            Fc[p2] = F << 10;
        }
        fast = (fmax & 0xFFFFu) <= 30u && (fmax >> 16) <= 30u;
    } else {
        // column maximum in the integer domain: per column the largest
        // key + 1 = (m >> 1) + 1 + sr over nonzero codes (0 if none), in
        // 16-bit lanes for two columns at a time
        uint32_t acc[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const uint32_t j = (uint32_t)(i & 3);
            const uint32_t sr2 = prmt(sw[i >> 2], 0u, 0x4040u | j | (j << 8));
            // the byte permutes read only the low 16 bits of their selector
            const uint32_t sel_lo = nb[i] & 0x77777777u, sel_hi = sel_lo >> 16;
            const uint32_t lev_lo = prmt(kLev1Lo, kLev1Hi, sel_lo), z_lo = prmt(kZeroLo, kZeroHi, sel_lo);
            const uint32_t lev_hi = prmt(kLev1Lo, kLev1Hi, sel_hi), z_hi = prmt(kZeroLo, kZeroHi, sel_hi);
            acc[0] = __viaddmax_s16x2(prmt(lev_lo, z_lo, 0x5140u), sr2, acc[0]);
            acc[1] = __viaddmax_s16x2(prmt(lev_lo, z_lo, 0x7362u), sr2, acc[1]);
            acc[2] = __viaddmax_s16x2(prmt(lev_hi, z_hi, 0x5140u), sr2, acc[2]);
            acc[3] = __viaddmax_s16x2(prmt(lev_hi, z_hi, 0x7362u), sr2, acc[3]);
        }
#pragma unroll
        for (int k = 0; k < 4; k++) acc[k] = __viaddmax_s16x2(__shfl_xor_sync(pair, acc[k], 1), 0u, acc[k]);
        // scale bytes: floor(log2 amax) = key - 128, e = that - 8 clamped to [-127, 127]
#pragma unroll
        for (int p2 = 0; p2 < 4; p2++) {
            const int k0 = (int)(acc[p2] & 0xFFFFu), k1 = (int)(acc[p2] >> 16);
            SB[p2] = nan ? 0x00FF00FFu
                         : (uint32_t)min(max(k0 - 10, 0), 254) | ((uint32_t)min(max(k1 - 10, 0), 254) << 16);
            Fc[p2] = 0;
        }
    }
    uint8_t* dst0 = out + (c0 + c) * R + r0 + 32 * rb + 16 * h;
    if (fast) {
        uint32_t ow[8][4];            // column k, rows 4 q .. 4 q + 3 in word q
#pragma unroll
        for (int q = 0; q < 4; q++) {
            uint32_t fr[4];
#pragma unroll
            for (int j = 0; j < 4; j++) fr[j] = prmt(sw[q], 0u, 0x4440u | (uint32_t)j) * 0x04000400u + kr;
            uint32_t e[4][4];         // row 4 q + j, columns (2 p, 2 p + 1): two E4M3 bytes
#pragma unroll
            for (int j = 0; j < 4; j++) {
                uint32_t hh[4];
                h2_of_e2m1x8(nb[4 * q + j], hh[0], hh[1], hh[2], hh[3]);
#pragma unroll
                for (int p2 = 0; p2 < 4; p2++) e[j][p2] = e4m3x2_of_h2(hmul2_rn(hmul2_rn(hh[p2], fr[j]), Fc[p2]));
            }
            // 4 x 4 byte transposes straight from the byte pairs: rows -> columns
#pragma unroll
            for (int p2 = 0; p2 < 4; p2 += 2) {
                const uint32_t t0 = prmt(e[0][p2], e[1][p2], 0x5140u), t1 = prmt(e[0][p2 + 1], e[1][p2 + 1], 0x5140u);
                const uint32_t t2 = prmt(e[2][p2], e[3][p2], 0x5140u), t3 = prmt(e[2][p2 + 1], e[3][p2 + 1], 0x5140u);
                ow[2 * p2 + 0][q] = prmt(t0, t2, 0x5410u);
                ow[2 * p2 + 1][q] = prmt(t0, t2, 0x7632u);
                ow[2 * p2 + 2][q] = prmt(t1, t3, 0x5410u);
                ow[2 * p2 + 3][q] = prmt(t1, t3, 0x7632u);
            }
        }
        // a column's 16 rows leave as one 16-byte store; with the neighbouring
        // lane's 16 they fill a whole 32-byte sector
#pragma unroll
        for (int k = 0; k < 8; k++)
            *reinterpret_cast<uint4*>(dst0 + (int64_t)k * R) = make_uint4(ow[k][0], ow[k][1], ow[k][2], ow[k][3]);
    } else {
        // scalar path: the E4M3 byte of each code in the integer domain, four
        // rows at a time (codes and row scales read again from shared memory)
#pragma unroll 1
        for (int q = 0; q < 4; q++) {
            uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int i = 4 * q + j;
                const uint32_t n8 = codes[((32 * rb + 16 * h + i) ^ h) * 16 + w];
                const uint32_t sr = sfr[cb * kColRows + 32 * rb + 16 * h + i];
#pragma unroll
                for (int k = 0; k < 8; k++)
                    o[k] |= fp8_of_nibble((n8 >> (4 * k)) & 0xFu, sr, (SB[k >> 1] >> (16 * (k & 1))) & 0xFFu) << (8 * j);
            }
#pragma unroll
            for (int k = 0; k < 8; k++)
                *reinterpret_cast<uint32_t*>(dst0 + (int64_t)k * R + 4 * q) = nan ? 0x7F7F7F7Fu : o[k];
        }
    }
    // the four output rows c0 + c + 4 h + k (k = 0..3) sit 16 bytes apart in their 128x4 tile
    uint8_t* s_dst = sout + sf_offset(c0 + c + 4 * h, r0 / 32 + rb, s_tiles_out);
    const uint32_t sa = h ? SB[2] : SB[0], sbb = h ? SB[3] : SB[1];
    s_dst[0] = (uint8_t)sa;
    s_dst[16] = (uint8_t)(sa >> 16);
    s_dst[32] = (uint8_t)sbb;
    s_dst[48] = (uint8_t)(sbb >> 16);
}

cudaError_t run_repack_col(const RepackArgs& a, cudaStream_t st) {
    cudaError_t e;
    if (a.scales_pad && (e = cudaMemsetAsync(a.out_scales, 0, a.scales_bytes, st)) != cudaSuccess) return e;
    const int64_t R = a.rows, C = a.cols;
    dim3 grid((unsigned)((C + kColCols - 1) / kColCols), (unsigned)((R + kColRows - 1) / kColRows));
    repack_col_kernel<<<grid, kColThreads, 0, st>>>(a.in_codes, a.in_scales, R, C, (C / 32 + 3) / 4, a.out_codes,
                                                   a.out_scales, (R / 32 + 3) / 4);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Dequantize: value = code * scale (* tensor scale), rounded once.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float e5m2_to_float(uint32_t b) {
    // an E5M2 byte is the high byte of the binary16 with the same value
    return __half2float(__ushort_as_half((uint16_t)((b & 0xFF) << 8)));
}
__device__ __forceinline__ float e2m1_to_float(uint32_t n) {
    const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    const float v = mag[n & 7];
    return (n & 8) ? -v : v;
}
__device__ __forceinline__ float e8m0_to_float(uint32_t s) {
    if (s == 0xFF) return __uint_as_float(0x7FC00000u);
    if (s == 0) return __uint_as_float(0x00400000u);    // 2^-127 (subnormal)
    return __uint_as_float(s << 23);
}

// Round the exact product p*q (FP32 inputs) once to BF16, nearest-even:
// hi = RN(p*q), lo = p*q - hi exactly (FMA two-product, Ogita-Rump-Oishi
// 2005); when hi sits exactly on a BF16 midpoint the residual decides.
__device__ __forceinline__ uint16_t mul_round_bf16(float p, float q) {
    const float hi = __fmul_rn(p, q);
    const float lo = __fmaf_rn(p, q, -hi);
    uint32_t u = __float_as_uint(hi);
    if ((u & 0x7F800000u) == 0x7F800000u) return __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    if ((u & 0xFFFFu) == 0x8000u && lo != 0.0f) {
        // exact value is above or below the midpoint in magnitude
        const bool away = (lo > 0.0f) == (hi > 0.0f);
        return (uint16_t)((u >> 16) + (away ? 1u : 0u));
    }
    return __bfloat16_as_ushort(__float2bfloat16_rn(hi));
}

template <int FMT>
__global__ void __launch_bounds__(256)
dequant_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, const float* __restrict__ ts,
               int64_t nchunks, uint32_t cols, int64_t s_tiles, void* __restrict__ dst, int out_bf16) {
    constexpr int BLK = block_of(FMT);
    const float s_t = FMT == kNVFP4 ? *ts : 1.0f;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < nchunks; c += stride) {
        const int64_t e0 = c * 8;
        const uint32_t r = (uint32_t)(e0 / cols), k = (uint32_t)(e0 - (int64_t)r * cols);
        const uint32_t sb = scales[sf_offset(r, k / BLK, s_tiles)];
        float v[8];
        if (is_fp4(FMT)) {
            const uint32_t w = reinterpret_cast<const uint32_t*>(codes)[c];
#pragma unroll
            for (int i = 0; i < 8; i++) v[i] = e2m1_to_float(w >> (4 * i));
        } else {
            const uint2 w = reinterpret_cast<const uint2*>(codes)[c];
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint32_t b = ((i < 4 ? w.x : w.y) >> (8 * (i & 3))) & 0xFF;
                v[i] = FMT == kE4M3 ? e4m3_to_float(b) : e5m2_to_float(b);
            }
        }
        if (FMT == kNVFP4) {
            const float sv = sb == 0x7F ? __uint_as_float(0x7FC00000u) : e4m3_to_float(sb);
#pragma unroll
            for (int i = 0; i < 8; i++) v[i] = __fmul_rn(v[i], sv);     // exact: <= 6 significant bits
            if (out_bf16) {
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; i++)
                    o[i] = (uint32_t)mul_round_bf16(v[2 * i], s_t) | ((uint32_t)mul_round_bf16(v[2 * i + 1], s_t) << 16);
                reinterpret_cast<uint4*>(dst)[c] = make_uint4(o[0], o[1], o[2], o[3]);
                continue;
            }
#pragma unroll
            for (int i = 0; i < 8; i++) v[i] = __fmul_rn(v[i], s_t);
        } else {
            const float f = e8m0_to_float(sb);
#pragma unroll
            for (int i = 0; i < 8; i++) v[i] = __fmul_rn(v[i], f);     // exact (power of two)
        }
        if (out_bf16) {
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; i++)
                o[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i])) |
                       ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1])) << 16);
            reinterpret_cast<uint4*>(dst)[c] = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            float4* d = reinterpret_cast<float4*>(dst) + 2 * c;
            d[0] = make_float4(v[0], v[1], v[2], v[3]);
            d[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
    }
}

cudaError_t run_dequant(const DequantArgs& a, cudaStream_t st) {
    const int64_t nchunks = a.rows * a.cols / 8;
    int64_t grid = (nchunks + 255) / 256;
    if (grid > (int64_t)a.num_sms * 16) grid = (int64_t)a.num_sms * 16;
    if (grid < 1) grid = 1;
    const int64_t S = a.cols / block_of(a.fmt);
    const int64_t st_ = (S + 3) / 4;
    const uint32_t cols = (uint32_t)a.cols;
    switch (a.fmt) {
    case kE4M3: dequant_kernel<kE4M3><<<(unsigned)grid, 256, 0, st>>>(a.codes, a.scales, a.ts, nchunks, cols, st_, a.dst, a.out_bf16); break;
    case kE5M2: dequant_kernel<kE5M2><<<(unsigned)grid, 256, 0, st>>>(a.codes, a.scales, a.ts, nchunks, cols, st_, a.dst, a.out_bf16); break;
    case kMXFP4: dequant_kernel<kMXFP4><<<(unsigned)grid, 256, 0, st>>>(a.codes, a.scales, a.ts, nchunks, cols, st_, a.dst, a.out_bf16); break;
    default: dequant_kernel<kNVFP4><<<(unsigned)grid, 256, 0, st>>>(a.codes, a.scales, a.ts, nchunks, cols, st_, a.dst, a.out_bf16); break;
    }
    return cudaGetLastError();
}

}  // namespace bsq
