// GEMM epilogue: one thread owns one output row segment of 128 FP32
// accumulator values (already moved from TMEM to registers), scales them by
// alpha, then by beta (the two NVFP4 tensor scales, one multiply each, so
// their product, which can underflow, is never formed), and stores them as
// BF16 or FP32, either
// directly (store_row128) or, for whole 32-row boxes, through a warp's
// 64-byte-swizzled shared staging buffer and one TMA tile store per chunk
// (store_tile_tma).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include "tcgen05.cuh"

namespace bsq {

__device__ __forceinline__ void store_row128(const uint32_t (&r)[4][32], void* C, int64_t ldc, int row, int col0,
                                             int N, int out_bf16, int vec_ok, float alpha, float beta) {
    if (out_bf16) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(C) + (int64_t)row * ldc + col0;
        if (vec_ok && col0 + 128 <= N) {
#pragma unroll
            for (int j = 0; j < 16; j++) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float x0 = __uint_as_float(r[j >> 2][(j & 3) * 8 + 2 * e]) * alpha * beta;
                    const float x1 = __uint_as_float(r[j >> 2][(j & 3) * 8 + 2 * e + 1]) * alpha * beta;
                    w[e] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x0)) |
                           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x1)) << 16);
                }
                *reinterpret_cast<uint4*>(out + 8 * j) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 128; j++)
                if (col0 + j < N) out[j] = __float2bfloat16_rn(__uint_as_float(r[j >> 5][j & 31]) * alpha * beta);
        }
    } else {
        float* out = reinterpret_cast<float*>(C) + (int64_t)row * ldc + col0;
        if (vec_ok && col0 + 128 <= N) {
#pragma unroll
            for (int j = 0; j < 32; j++) {
                float4 v;
                v.x = __uint_as_float(r[j >> 3][(j & 7) * 4 + 0]) * alpha * beta;
                v.y = __uint_as_float(r[j >> 3][(j & 7) * 4 + 1]) * alpha * beta;
                v.z = __uint_as_float(r[j >> 3][(j & 7) * 4 + 2]) * alpha * beta;
                v.w = __uint_as_float(r[j >> 3][(j & 7) * 4 + 3]) * alpha * beta;
                *reinterpret_cast<float4*>(out + 4 * j) = v;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 128; j++)
                if (col0 + j < N) out[j] = __uint_as_float(r[j >> 5][j & 31]) * alpha * beta;
        }
    }
}

// Staged epilogue for TMA stores.  A warp owns 32 output rows (one per lane)
// x 128 columns held in registers; it writes them in 64-byte column chunks
// (32 BF16 or 16 FP32 values per row) into a 2 KB shared buffer laid out as
// 32 rows x 64 bytes with the 64-byte swizzle (16-byte unit u of row r at
// unit u ^ ((r >> 1) & 3)), so that a warp's 16-byte writes fall in distinct
// banks, and lane 0 stores each chunk with one TMA tile store.
// `buf` is the buffer's shared address (512-byte aligned); (col0, row0) the
// output coordinates of the warp's first element.
template <bool BF16>
__device__ __forceinline__ void store_tile_tma(const uint32_t (&r)[4][32], uint32_t buf, const void* tmap, int col0,
                                               int row0, float alpha, float beta, int lane) {
    constexpr int PER = BF16 ? 32 : 16;                // values per row per chunk
    const uint32_t row_base = buf + (uint32_t)lane * 64u;
    const uint32_t sw = (uint32_t)((lane >> 1) & 3);
#pragma unroll
    for (int ch = 0; ch < 128 / PER; ch++) {
        if (lane == 0) tc::bulk_wait_read();         // previous chunk has left the buffer
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 4; u++) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                if (BF16) {
                    const int c = ch * 32 + u * 8 + 2 * e;
                    const float x0 = __uint_as_float(r[c >> 5][c & 31]) * alpha * beta;
                    const float x1 = __uint_as_float(r[(c + 1) >> 5][(c + 1) & 31]) * alpha * beta;
                    w[e] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x0)) |
                           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x1)) << 16);
                } else {
                    const int c = ch * 16 + u * 4 + e;
                    w[e] = __float_as_uint(__uint_as_float(r[c >> 5][c & 31]) * alpha * beta);
                }
            }
            const uint32_t a = row_base + ((u ^ sw) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(a), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                         : "memory");
        }
        tc::fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            tc::tma_store_2d(tmap, col0 + ch * PER, row0, buf);
            tc::bulk_commit();
        }
    }
}

// tcgen05 instruction descriptor of the block-scaled kinds, without the
// scale-factor ids: bits 7-9 A type, 10-12 B type, 17-22 N>>3, 23 scale
// type (1 = UE8M0, 0 = UE4M3), 24-28 M>>4; K-major A and B, dense.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t atype, uint32_t btype, bool ue8m0, int M, int N) {
    return (atype << 7) | (btype << 10) | ((uint32_t)(N >> 3) << 17) | ((ue8m0 ? 1u : 0u) << 23) |
           ((uint32_t)(M >> 4) << 24);
}

}  // namespace bsq
