// Device helpers shared by the quantize, convert and GEMM kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace bsq {

// Status bits recorded in the device status word.
constexpr unsigned kStatusTimeout = 1u;

// Format ids (mirror bsq_format).
constexpr int kE4M3 = 0, kE5M2 = 1, kMXFP4 = 2, kNVFP4 = 3;

__host__ __device__ constexpr int block_of(int fmt) { return fmt == kNVFP4 ? 16 : 32; }
__host__ __device__ constexpr bool is_fp4(int fmt) { return fmt >= kMXFP4; }
// floor(log2(largest finite element value))
__host__ __device__ constexpr int emax_of(int fmt) { return fmt == kE4M3 ? 8 : (fmt == kE5M2 ? 15 : 2); }

// Byte offset of scale (r, c) in the 128x4-tiled scale layout of a scale
// matrix with `s_tiles` = ceil(S/4) tiles per 128-row band.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t s_tiles) {
    return ((r >> 7) * s_tiles + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// |x| bits of two packed bf16 values, NaN/Inf-aware max helpers work on
// these integer magnitudes (for non-negative finite floats integer order
// equals value order).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
    uint32_t lo = w & 0x7FFFu, hi = (w >> 16) & 0x7FFFu;
    return max(acc, max(lo, hi));
}

// --- conversions through the hardware cvt instructions (RNE, satfinite) ---
// Two FP32 values -> two E4M3 bytes, `lo` in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t cvt_e5m2x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// Two FP32 values -> one byte of two E2M1 nibbles, `lo` in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// E4M3 byte -> its exact value (through the f16x2 widening cvt).
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
    uint32_t h2;
    uint16_t in = (uint16_t)(b & 0xFF);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFF)));
}

// 8 FP32 values -> 8 FP8 codes packed little-endian into a uint2.
template <int FMT>
__device__ __forceinline__ uint2 pack8_fp8(const float* v) {
    uint32_t a, b, c, d;
    if (FMT == kE4M3) {
        a = cvt_e4m3x2(v[0], v[1]); b = cvt_e4m3x2(v[2], v[3]);
        c = cvt_e4m3x2(v[4], v[5]); d = cvt_e4m3x2(v[6], v[7]);
    } else {
        a = cvt_e5m2x2(v[0], v[1]); b = cvt_e5m2x2(v[2], v[3]);
        c = cvt_e5m2x2(v[4], v[5]); d = cvt_e5m2x2(v[6], v[7]);
    }
    return make_uint2(a | (b << 16), c | (d << 16));
}
// 8 FP32 values -> 8 E2M1 nibbles in a uint32 (element i in nibble i).
__device__ __forceinline__ uint32_t pack8_fp4(const float* v) {
    return cvt_e2m1x2(v[0], v[1]) | (cvt_e2m1x2(v[2], v[3]) << 8) |
           (cvt_e2m1x2(v[4], v[5]) << 16) | (cvt_e2m1x2(v[6], v[7]) << 24);
}

// MX shared-scale byte from the block's |amax| bf16 bits (7FFF-masked).
// e = floor(log2 amax) - emax clamped to [-127, 127]; a zero or subnormal
// amax lands on the clamp (byte 0); a non-finite amax gives 0xFF.
template <int FMT>
__device__ __forceinline__ uint32_t mx_scale_byte(uint32_t amax_bits) {
    uint32_t ef = amax_bits >> 7;             // bf16 exponent field
    if (ef == 0xFF) return 0xFF;
    int b = (int)ef - emax_of(FMT);           // = e + 127 for normal amax
    return (uint32_t)max(b, 0);
}
// 2^-e for a scale byte b = e + 127 in [0, 254]; always a normal float.
__device__ __forceinline__ float mx_inv_scale(uint32_t b) {
    return __uint_as_float((254u - b) << 23);
}

// Status word update (only on the failure path).
__device__ __forceinline__ void record_status(unsigned* status, unsigned bits) {
    if (status) atomicOr(status, bits);
}

// v clamped to [lo, hi] (row offsets read from device memory)
__device__ __forceinline__ int clamp_rows(int64_t v, int64_t lo, int64_t hi) {
    return (int)(v < lo ? lo : (v > hi ? hi : v));
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

}  // namespace bsq
