// GEMM epilogue: one thread owns one output row segment of 128 FP32
// accumulator values (already moved from TMEM to registers), scales them by
// alpha (NVFP4 tensor scales) and stores them as BF16 or FP32.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace bsq {

__device__ __forceinline__ void store_row128(const uint32_t (&r)[4][32], void* C, int64_t ldc, int row, int col0,
                                             int N, int out_bf16, int vec_ok, float alpha) {
    if (out_bf16) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(C) + (int64_t)row * ldc + col0;
        if (vec_ok && col0 + 128 <= N) {
#pragma unroll
            for (int j = 0; j < 16; j++) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float x0 = __uint_as_float(r[j >> 2][(j & 3) * 8 + 2 * e]) * alpha;
                    const float x1 = __uint_as_float(r[j >> 2][(j & 3) * 8 + 2 * e + 1]) * alpha;
                    w[e] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x0)) |
                           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x1)) << 16);
                }
                *reinterpret_cast<uint4*>(out + 8 * j) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 128; j++)
                if (col0 + j < N) out[j] = __float2bfloat16_rn(__uint_as_float(r[j >> 5][j & 31]) * alpha);
        }
    } else {
        float* out = reinterpret_cast<float*>(C) + (int64_t)row * ldc + col0;
        if (vec_ok && col0 + 128 <= N) {
#pragma unroll
            for (int j = 0; j < 32; j++) {
                float4 v;
                v.x = __uint_as_float(r[j >> 3][(j & 7) * 4 + 0]) * alpha;
                v.y = __uint_as_float(r[j >> 3][(j & 7) * 4 + 1]) * alpha;
                v.z = __uint_as_float(r[j >> 3][(j & 7) * 4 + 2]) * alpha;
                v.w = __uint_as_float(r[j >> 3][(j & 7) * 4 + 3]) * alpha;
                *reinterpret_cast<float4*>(out + 4 * j) = v;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 128; j++)
                if (col0 + j < N) out[j] = __uint_as_float(r[j >> 5][j & 31]) * alpha;
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
