// Internal host-side interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace bsq {

struct QuantizeArgs {
    const void* src;
    int64_t rows, cols;
    int fmt, axis;
    uint8_t *row_codes, *row_scales, *col_codes, *col_scales;
    float *row_ts, *col_ts;
    size_t row_scales_bytes, col_scales_bytes;
    bool row_scales_pad, col_scales_pad;     // buffer has padding to zero
    int num_sms;
    float* history;                // NVFP4 delayed scaling: amax history (nullptr: just in time)
    int hist_len;
};
cudaError_t run_quantize(const QuantizeArgs& a, cudaStream_t st);

struct RepackArgs {
    const uint8_t* in_codes;
    const uint8_t* in_scales;
    uint8_t* out_codes;
    uint8_t* out_scales;
    int64_t rows, cols;
    size_t scales_bytes;
    bool scales_pad;
    int num_sms;
    // per-expert padded scale layout of the output (num_groups = 0: plain)
    const int64_t* offsets;
    int num_groups;
};
cudaError_t run_repack(const RepackArgs& a, cudaStream_t st);
// FP4RowToFP8Col: rows, cols = the MXFP4 input's; the output is [cols, rows]
cudaError_t run_repack_col(const RepackArgs& a, cudaStream_t st);
// MXFP4 -> FP8 E4M3 with 1 x 128 blocks: out_codes [rows, cols], out_scales
// [rows, ceil(cols / 128)] E8M0 bytes, both row-major
cudaError_t run_repack_1x128(const RepackArgs& a, cudaStream_t st);

struct DequantArgs {
    int fmt;
    const uint8_t* codes;
    const uint8_t* scales;
    const float* ts;
    int64_t rows, cols;
    void* dst;
    int out_bf16;
    int num_sms;
};
cudaError_t run_dequant(const DequantArgs& a, cudaStream_t st);

constexpr int kMaxGroups = 256;

struct GemmArgs {
    int fmt_a, fmt_b;              // bsq_format of A and B
    const uint8_t* a_codes;
    const uint8_t* a_scales;
    const uint8_t* b_codes;        // grouped: group 0, groups consecutive
    const uint8_t* b_scales;       // dense only
    const float* ts_a;             // NVFP4 tensor scales
    const float* ts_b;
    int64_t M, N, K;               // grouped: M = total rows, N = per-group rows of B
    void* C;
    int out_bf16;
    // grouped
    int num_groups;                // 0 = dense
    const int64_t* offsets;        // device
    const uint8_t* const* b_group_scales;   // host array [num_groups]
    bool a_grouped_sf;             // grouped: A's scales in the per-expert padded layout
    int num_sms;
    unsigned* status;
    uint64_t timeout_ns;
    bool single_cta;               // use the 1-CTA kernel instead of the CTA pair
    bool grouped_pair;             // grouped: CTA pairs whatever the expert sizes
};
cudaError_t run_gemm(const GemmArgs& a, cudaStream_t st);
cudaError_t run_gemm_pair(const GemmArgs& a, cudaStream_t st);
bool gemm_pair_grouped_ok(const GemmArgs& a);

cudaError_t run_timeout_probe(unsigned* status, uint64_t limit_ns, cudaStream_t st);

}  // namespace bsq
