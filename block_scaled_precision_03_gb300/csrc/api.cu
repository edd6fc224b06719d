// C ABI of libbsq.so: argument checks, status word and dispatch to kernels.
// Every check runs on the host before anything is launched; a rejected call
// launches nothing and writes nothing.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include "../../include/bsq.h"
#include "common.cuh"
#include "internal.h"

namespace {

// Device status word: kernels OR failure bits into it; bsq_sync_status takes
// and clears it in one atomic exchange on the device.  Lives in static device
// memory, no allocation.
__device__ unsigned g_status_word;
__device__ unsigned g_status_taken;     // the value the last exchange returned

__global__ void status_take_kernel() { g_status_taken = atomicExch(&g_status_word, 0u); }

int g_num_sms[64];

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (g_num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_num_sms[dev] = n;
    }
    return g_num_sms[dev];
}

unsigned* status_ptr() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    return static_cast<unsigned*>(p);
}

bool valid_fmt(int32_t f) { return f >= BSQ_MXFP8_E4M3 && f <= BSQ_NVFP4_E2M1; }
int blk(int32_t f) { return f == BSQ_NVFP4_E2M1 ? 16 : 32; }
bool fp4(int32_t f) { return f == BSQ_MXFP4_E2M1 || f == BSQ_NVFP4_E2M1; }
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t codes_bytes(int32_t f, int64_t r, int64_t c) { return fp4(f) ? (size_t)(r * c / 2) : (size_t)(r * c); }
size_t scales_bytes(int32_t f, int64_t r, int64_t c) {
    const int64_t S = c / blk(f);
    return (size_t)(((r + 127) / 128 * 128) * ((S + 3) / 4 * 4));
}
bool scales_padded(int32_t f, int64_t r, int64_t c) { return (r % 128) != 0 || ((c / blk(f)) % 4) != 0; }

// a tensor descriptor is usable as a quantized operand
bsq_status check_tensor(const bsq_tensor* t, bool need_ts) {
    if (!t || !valid_fmt(t->fmt) || t->reserved != 0) return BSQ_ERR_INVALID_ARG;
    if (t->rows < 1 || t->cols < 1 || (t->cols % blk(t->fmt)) != 0) return BSQ_ERR_INVALID_ARG;
    if (!t->codes || !t->scales) return BSQ_ERR_INVALID_ARG;
    if (need_ts && t->fmt == BSQ_NVFP4_E2M1 && !t->tensor_scale) return BSQ_ERR_INVALID_ARG;
    if (!al16(t->codes) || !al16(t->scales)) return BSQ_ERR_ALIGNMENT;
    return BSQ_OK;
}

bsq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA; }

// BSQ_GEMM_1CTA=1 routes dense GEMMs to the single-CTA kernel (the grouped
// GEMM's kernel) instead of the CTA-pair kernel; used by the test suite to
// check both tile shapes.
bool env_single_cta() {
    const char* v = std::getenv("BSQ_GEMM_1CTA");
    return v && v[0] == '1';
}

// BSQ_GEMM_GROUPED_PAIR=1 sends grouped GEMMs to the CTA-pair kernel whatever
// the expert sizes (when their layout allows it); used by the test suite.
bool env_grouped_pair() {
    const char* v = std::getenv("BSQ_GEMM_GROUPED_PAIR");
    return v && v[0] == '1';
}

const uint64_t kDefaultTimeoutNs = 4000000000ull;   // 4 s per wait



// bsq_quantize and bsq_quantize_nvfp4_delayed: argument checks and launch;
// `history` (NVFP4 only) selects delayed scaling.
bsq_status quantize_common(const void* src_bf16, int64_t rows, int64_t cols, int32_t fmt, int32_t axis,
                           bsq_tensor* out_row, bsq_tensor* out_col, float* history, int32_t hist_len,
                           void* stream) {
    if (!src_bf16 || !valid_fmt(fmt) || axis < BSQ_ROWWISE || axis > BSQ_BOTH) return BSQ_ERR_INVALID_ARG;
    if (rows < 1 || cols < 1) return BSQ_ERR_INVALID_ARG;
    if (!al16(src_bf16) || (cols % 8) != 0) return BSQ_ERR_ALIGNMENT;
    const bool want_row = axis & BSQ_ROWWISE, want_col = axis & BSQ_COLWISE;
    if (want_row) {
        if (cols % blk(fmt)) return BSQ_ERR_INVALID_ARG;
        bsq_status s = check_tensor(out_row, true);
        if (s != BSQ_OK) return s;
        if (out_row->fmt != fmt || out_row->rows != rows || out_row->cols != cols) return BSQ_ERR_INVALID_ARG;
    }
    if (want_col) {
        if (rows % blk(fmt)) return BSQ_ERR_INVALID_ARG;
        bsq_status s = check_tensor(out_col, true);
        if (s != BSQ_OK) return s;
        if (out_col->fmt != fmt || out_col->rows != cols || out_col->cols != rows) return BSQ_ERR_INVALID_ARG;
        // transposed FP4 rows of R/2 bytes must keep 8-byte (NVFP4) / 16-byte (MXFP4) stores aligned
        if (fp4(fmt) && ((rows / 2) % (fmt == BSQ_NVFP4_E2M1 ? 8 : 16))) return BSQ_ERR_ALIGNMENT;
    }
    if (want_row && fp4(fmt) && ((cols / 2) % (fmt == BSQ_NVFP4_E2M1 ? 8 : 16)) && axis == BSQ_BOTH)
        return BSQ_ERR_ALIGNMENT;
    bsq::QuantizeArgs a{};
    a.src = src_bf16;
    a.rows = rows;
    a.cols = cols;
    a.fmt = fmt;
    a.axis = axis;
    if (want_row) {
        a.row_codes = static_cast<uint8_t*>(out_row->codes);
        a.row_scales = out_row->scales;
        a.row_ts = out_row->tensor_scale;
        a.row_scales_bytes = scales_bytes(fmt, rows, cols);
        a.row_scales_pad = scales_padded(fmt, rows, cols);
    }
    if (want_col) {
        a.col_codes = static_cast<uint8_t*>(out_col->codes);
        a.col_scales = out_col->scales;
        a.col_ts = out_col->tensor_scale;
        a.col_scales_bytes = scales_bytes(fmt, cols, rows);
        a.col_scales_pad = scales_padded(fmt, cols, rows);
    }
    a.num_sms = num_sms();
    a.history = history;
    a.hist_len = hist_len;
    return from_cuda(bsq::run_quantize(a, static_cast<cudaStream_t>(stream)));
}


}  // namespace

extern "C" {

size_t bsq_codes_bytes(int32_t fmt, int64_t rows, int64_t cols) {
    if (!valid_fmt(fmt) || rows < 0 || cols < 0) return 0;
    if (fp4(fmt) && (cols % 2)) return 0;
    return codes_bytes(fmt, rows, cols);
}

size_t bsq_scales_bytes(int32_t fmt, int64_t rows, int64_t cols) {
    if (!valid_fmt(fmt) || rows < 0 || cols < 0 || (cols % blk(fmt)) != 0) return 0;
    return scales_bytes(fmt, rows, cols);
}

bsq_status bsq_quantize(const void* src_bf16, int64_t rows, int64_t cols, int32_t fmt, int32_t axis,
                        bsq_tensor* out_row, bsq_tensor* out_col, void* stream) {
    return quantize_common(src_bf16, rows, cols, fmt, axis, out_row, out_col, nullptr, 0, stream);
}

bsq_status bsq_quantize_nvfp4_delayed(const void* src_bf16, int64_t rows, int64_t cols, int32_t axis,
                                      bsq_tensor* out_row, bsq_tensor* out_col, float* amax_history,
                                      int32_t history_len, void* stream) {
    if (!amax_history || history_len < 1 || history_len > 4096) return BSQ_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(amax_history) & 3) return BSQ_ERR_ALIGNMENT;
    // same argument rules as bsq_quantize with NVFP4; the scale then comes from the history
    return quantize_common(src_bf16, rows, cols, BSQ_NVFP4_E2M1, axis, out_row, out_col, amax_history, history_len,
                           stream);
}

bsq_status bsq_dequantize(const bsq_tensor* in, void* dst, int32_t dst_type, void* stream) {
    bsq_status s = check_tensor(in, true);
    if (s != BSQ_OK) return s;
    if (!dst || (dst_type != BSQ_OUT_F32 && dst_type != BSQ_OUT_BF16)) return BSQ_ERR_INVALID_ARG;
    if (!al16(dst)) return BSQ_ERR_ALIGNMENT;
    bsq::DequantArgs a{};
    a.fmt = in->fmt;
    a.codes = static_cast<const uint8_t*>(in->codes);
    a.scales = in->scales;
    a.ts = in->tensor_scale;
    a.rows = in->rows;
    a.cols = in->cols;
    a.dst = dst;
    a.out_bf16 = dst_type == BSQ_OUT_BF16;
    a.num_sms = num_sms();
    return from_cuda(bsq::run_dequant(a, static_cast<cudaStream_t>(stream)));
}

static bsq_status check_gemm_pair(const bsq_tensor* A, const bsq_tensor* B) {
    bsq_status s = check_tensor(A, true);
    if (s != BSQ_OK) return s;
    if ((s = check_tensor(B, true)) != BSQ_OK) return s;
    if (A->cols != B->cols) return BSQ_ERR_INVALID_ARG;
    if (A->cols % 32) return BSQ_ERR_INVALID_ARG;
    const bool a8 = A->fmt == BSQ_MXFP8_E4M3 || A->fmt == BSQ_MXFP8_E5M2;
    const bool b8 = B->fmt == BSQ_MXFP8_E4M3 || B->fmt == BSQ_MXFP8_E5M2;
    if (a8 && b8) return BSQ_OK;
    if (A->fmt == BSQ_NVFP4_E2M1 && B->fmt == BSQ_NVFP4_E2M1) return BSQ_OK;
    if (A->fmt == BSQ_MXFP4_E2M1 && B->fmt == BSQ_MXFP4_E2M1) return BSQ_OK;
    return BSQ_ERR_UNSUPPORTED;
}

// bsq_gemm and bsq_debug_gemm_timeout: checks and launch with a given wait
// limit; `force_single` selects the 1-CTA kernel.
static bsq_status gemm_common(const bsq_tensor* A, const bsq_tensor* B, void* C, int32_t out_type, uint64_t timeout_ns,
                              bool force_single, void* stream) {
    bsq_status s = check_gemm_pair(A, B);
    if (s != BSQ_OK) return s;
    if (!C || (out_type != BSQ_OUT_F32 && out_type != BSQ_OUT_BF16)) return BSQ_ERR_INVALID_ARG;
    if (A->rows > 0x7FFFFF00LL || B->rows > 0x7FFFFF00LL) return BSQ_ERR_UNSUPPORTED;
    if (!al16(C)) return BSQ_ERR_ALIGNMENT;
    // MXFP4 runs on the CTA-pair kernel only
    if (force_single && A->fmt == BSQ_MXFP4_E2M1) return BSQ_ERR_UNSUPPORTED;
    unsigned* st = status_ptr();
    if (!st) return BSQ_ERR_CUDA;
    bsq::GemmArgs a{};
    a.fmt_a = A->fmt;
    a.fmt_b = B->fmt;
    a.a_codes = static_cast<const uint8_t*>(A->codes);
    a.a_scales = A->scales;
    a.b_codes = static_cast<const uint8_t*>(B->codes);
    a.b_scales = B->scales;
    a.ts_a = A->tensor_scale;
    a.ts_b = B->tensor_scale;
    a.M = A->rows;
    a.N = B->rows;
    a.K = A->cols;
    a.C = C;
    a.out_bf16 = out_type == BSQ_OUT_BF16;
    a.num_groups = 0;
    a.single_cta = force_single || env_single_cta();
    a.num_sms = num_sms();
    a.status = st;
    a.timeout_ns = timeout_ns;
    return from_cuda(bsq::run_gemm(a, static_cast<cudaStream_t>(stream)));
}

bsq_status bsq_gemm(const bsq_tensor* A, const bsq_tensor* B, void* C, int32_t out_type, void* stream) {
    return gemm_common(A, B, C, out_type, kDefaultTimeoutNs, false, stream);
}

bsq_status bsq_debug_gemm_timeout(const bsq_tensor* A, const bsq_tensor* B, void* C, int32_t out_type,
                                  uint64_t timeout_ns, int32_t kernel, void* stream) {
    if (timeout_ns == 0 || timeout_ns > kDefaultTimeoutNs || kernel < 0 || kernel > 1) return BSQ_ERR_INVALID_ARG;
    return gemm_common(A, B, C, out_type, timeout_ns, kernel == 1, stream);
}

// bsq_grouped_gemm and bsq_grouped_gemm_padded: checks and launch; `padded`
// says A's scales are in the per-expert padded layout.
static bsq_status grouped_gemm_common(const bsq_tensor* A, const int64_t* group_offsets_dev, int32_t num_groups,
                               const bsq_tensor* B_groups, void* C, int32_t out_type, bool padded, void* stream) {
    if (!B_groups || !group_offsets_dev || num_groups < 1) return BSQ_ERR_INVALID_ARG;
    if (num_groups > bsq::kMaxGroups) return BSQ_ERR_UNSUPPORTED;
    bsq_status s = check_gemm_pair(A, &B_groups[0]);
    if (s != BSQ_OK) return s;
    if (A->fmt == BSQ_NVFP4_E2M1) return BSQ_ERR_UNSUPPORTED;
    if (!C || (out_type != BSQ_OUT_F32 && out_type != BSQ_OUT_BF16)) return BSQ_ERR_INVALID_ARG;
    if (!al16(C)) return BSQ_ERR_ALIGNMENT;
    const bsq_tensor& b0 = B_groups[0];
    const size_t gbytes = codes_bytes(b0.fmt, b0.rows, b0.cols);
    const uint8_t* sf[bsq::kMaxGroups];
    for (int g = 0; g < num_groups; g++) {
        const bsq_tensor& bg = B_groups[g];
        if ((s = check_tensor(&bg, false)) != BSQ_OK) return s;
        if (bg.fmt != b0.fmt || bg.rows != b0.rows || bg.cols != b0.cols) return BSQ_ERR_INVALID_ARG;
        if (static_cast<const uint8_t*>(bg.codes) != static_cast<const uint8_t*>(b0.codes) + g * gbytes)
            return BSQ_ERR_UNSUPPORTED;
        sf[g] = bg.scales;
    }
    if (A->rows > 0x7FFFFF00LL || (int64_t)num_groups * b0.rows > 0x7FFFFF00LL) return BSQ_ERR_UNSUPPORTED;
    unsigned* st = status_ptr();
    if (!st) return BSQ_ERR_CUDA;
    bsq::GemmArgs a{};
    a.fmt_a = A->fmt;
    a.fmt_b = b0.fmt;
    a.a_codes = static_cast<const uint8_t*>(A->codes);
    a.a_scales = A->scales;
    a.b_codes = static_cast<const uint8_t*>(b0.codes);
    a.b_scales = b0.scales;
    a.M = A->rows;
    a.N = b0.rows;
    a.K = A->cols;
    a.C = C;
    a.out_bf16 = out_type == BSQ_OUT_BF16;
    a.num_groups = num_groups;
    a.offsets = group_offsets_dev;
    a.b_group_scales = sf;
    a.a_grouped_sf = padded;
    a.single_cta = env_single_cta();
    a.grouped_pair = env_grouped_pair();
    a.num_sms = num_sms();
    a.status = st;
    a.timeout_ns = kDefaultTimeoutNs;
    // MXFP4 runs on the CTA-pair kernel only, which spans the experts' scales
    // with one tensor map: they must be evenly spaced (as group views are)
    if (A->fmt == BSQ_MXFP4_E2M1 && !bsq::gemm_pair_grouped_ok(a)) return BSQ_ERR_UNSUPPORTED;
    return from_cuda(bsq::run_gemm(a, static_cast<cudaStream_t>(stream)));
}

bsq_status bsq_grouped_gemm(const bsq_tensor* A, const int64_t* group_offsets_dev, int32_t num_groups,
                            const bsq_tensor* B_groups, void* C, int32_t out_type, void* stream) {
    return grouped_gemm_common(A, group_offsets_dev, num_groups, B_groups, C, out_type, false, stream);
}

bsq_status bsq_grouped_gemm_padded(const bsq_tensor* A, const int64_t* group_offsets_dev, int32_t num_groups,
                                   const bsq_tensor* B_groups, void* C, int32_t out_type, void* stream) {
    return grouped_gemm_common(A, group_offsets_dev, num_groups, B_groups, C, out_type, true, stream);
}

size_t bsq_grouped_scales_bytes(int32_t fmt, int64_t rows, int64_t cols, int32_t num_groups) {
    if (num_groups < 1 || num_groups > bsq::kMaxGroups) return 0;
    if (!valid_fmt(fmt) || rows < 0 || cols < 0 || (cols % blk(fmt)) != 0) return 0;
    const int64_t s_pad = (cols / blk(fmt) + 3) / 4 * 4;
    return (size_t)(((rows + 127) / 128 * 128) + 128 * (int64_t)num_groups) * (size_t)s_pad;
}

bsq_status bsq_mxfp4_to_mxfp8_grouped(const bsq_tensor* in, bsq_tensor* out, const int64_t* group_offsets_dev,
                                      int32_t num_groups, void* stream) {
    if (!group_offsets_dev || num_groups < 1) return BSQ_ERR_INVALID_ARG;
    if (num_groups > bsq::kMaxGroups) return BSQ_ERR_UNSUPPORTED;
    bsq_status s = check_tensor(in, false);
    if (s != BSQ_OK) return s;
    if ((s = check_tensor(out, false)) != BSQ_OK) return s;
    if (in->fmt != BSQ_MXFP4_E2M1 || out->fmt != BSQ_MXFP8_E4M3) return BSQ_ERR_UNSUPPORTED;
    if (in->rows != out->rows || in->cols != out->cols) return BSQ_ERR_INVALID_ARG;
    if (in->rows > 0x7FFFFF00LL) return BSQ_ERR_UNSUPPORTED;
    bsq::RepackArgs a{};
    a.in_codes = static_cast<const uint8_t*>(in->codes);
    a.in_scales = in->scales;
    a.out_codes = static_cast<uint8_t*>(out->codes);
    a.out_scales = out->scales;
    a.rows = in->rows;
    a.cols = in->cols;
    a.scales_bytes = bsq_grouped_scales_bytes(BSQ_MXFP8_E4M3, in->rows, in->cols, num_groups);
    a.scales_pad = false;              // the kernel writes every byte of the capacity
    a.num_sms = num_sms();
    a.offsets = group_offsets_dev;
    a.num_groups = num_groups;
    return from_cuda(bsq::run_repack(a, static_cast<cudaStream_t>(stream)));
}

bsq_status bsq_mxfp4_to_mxfp8(const bsq_tensor* in, bsq_tensor* out, void* stream) {
    bsq_status s = check_tensor(in, false);
    if (s != BSQ_OK) return s;
    if ((s = check_tensor(out, false)) != BSQ_OK) return s;
    if (in->fmt != BSQ_MXFP4_E2M1 || out->fmt != BSQ_MXFP8_E4M3) return BSQ_ERR_UNSUPPORTED;
    if (in->rows != out->rows || in->cols != out->cols) return BSQ_ERR_INVALID_ARG;
    bsq::RepackArgs a{};
    a.in_codes = static_cast<const uint8_t*>(in->codes);
    a.in_scales = in->scales;
    a.out_codes = static_cast<uint8_t*>(out->codes);
    a.out_scales = out->scales;
    a.rows = in->rows;
    a.cols = in->cols;
    a.scales_bytes = scales_bytes(BSQ_MXFP8_E4M3, in->rows, in->cols);
    a.scales_pad = scales_padded(BSQ_MXFP8_E4M3, in->rows, in->cols);
    a.num_sms = num_sms();
    return from_cuda(bsq::run_repack(a, static_cast<cudaStream_t>(stream)));
}

bsq_status bsq_mxfp4_to_mxfp8_col(const bsq_tensor* in, bsq_tensor* out, void* stream) {
    bsq_status s = check_tensor(in, false);
    if (s != BSQ_OK) return s;
    if ((s = check_tensor(out, false)) != BSQ_OK) return s;
    if (in->fmt != BSQ_MXFP4_E2M1 || out->fmt != BSQ_MXFP8_E4M3) return BSQ_ERR_UNSUPPORTED;
    if (out->rows != in->cols || out->cols != in->rows) return BSQ_ERR_INVALID_ARG;
    if (in->rows % 32 || in->cols % 32) return BSQ_ERR_INVALID_ARG;
    bsq::RepackArgs a{};
    a.in_codes = static_cast<const uint8_t*>(in->codes);
    a.in_scales = in->scales;
    a.out_codes = static_cast<uint8_t*>(out->codes);
    a.out_scales = out->scales;
    a.rows = in->rows;
    a.cols = in->cols;
    a.scales_bytes = scales_bytes(BSQ_MXFP8_E4M3, out->rows, out->cols);
    a.scales_pad = scales_padded(BSQ_MXFP8_E4M3, out->rows, out->cols);
    a.num_sms = num_sms();
    return from_cuda(bsq::run_repack_col(a, static_cast<cudaStream_t>(stream)));
}

bsq_status bsq_mxfp4_to_fp8_1x128(const bsq_tensor* in, void* out_codes, void* out_scales, void* stream) {
    bsq_status s = check_tensor(in, false);
    if (s != BSQ_OK) return s;
    if (in->fmt != BSQ_MXFP4_E2M1) return BSQ_ERR_UNSUPPORTED;
    if (!out_codes || !out_scales) return BSQ_ERR_INVALID_ARG;
    if (!al16(out_codes)) return BSQ_ERR_ALIGNMENT;
    bsq::RepackArgs a{};
    a.in_codes = static_cast<const uint8_t*>(in->codes);
    a.in_scales = in->scales;
    a.out_codes = static_cast<uint8_t*>(out_codes);
    a.out_scales = static_cast<uint8_t*>(out_scales);
    a.rows = in->rows;
    a.cols = in->cols;
    a.num_sms = num_sms();
    return from_cuda(bsq::run_repack_1x128(a, static_cast<cudaStream_t>(stream)));
}

bsq_status bsq_sync_status(void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // take-and-clear in one device-side atomic exchange, ordered after the
    // stream's work; then read the taken value back
    status_take_kernel<<<1, 1, 0, st>>>();
    if (cudaGetLastError() != cudaSuccess) return BSQ_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_taken, sizeof(v), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return BSQ_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return BSQ_ERR_CUDA;
    if (v & bsq::kStatusTimeout) return BSQ_ERR_TIMEOUT;
    return BSQ_OK;
}

bsq_status bsq_debug_timeout_probe(uint64_t limit_ns, void* stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return BSQ_ERR_INVALID_ARG;
    unsigned* st = status_ptr();
    if (!st) return BSQ_ERR_CUDA;
    return from_cuda(bsq::run_timeout_probe(st, limit_ns, static_cast<cudaStream_t>(stream)));
}

const char* bsq_status_string(int32_t s) {
    switch (s) {
    case BSQ_OK: return "ok";
    case BSQ_ERR_INVALID_ARG: return "invalid argument";
    case BSQ_ERR_UNSUPPORTED: return "unsupported request";
    case BSQ_ERR_ALIGNMENT: return "misaligned pointer or row pitch";
    case BSQ_ERR_CUDA: return "CUDA runtime error";
    case BSQ_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

const char* bsq_version(void) { return "bsq 0.1 sm_103a"; }

}  // extern "C"
