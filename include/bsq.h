/*
 * bsq.h -- C ABI of libbsq.so: block-scaled low-precision linear layer on
 * NVIDIA GB300 (sm_103a).
 *
 * What the library computes (the pages give the method in prose only):
 *  - Quantize BF16 tensors to MXFP8 (E4M3 for forward activations and
 *    weights, E5M2 for gradients), to MXFP4 and to NVFP4, row-wise and
 *    column-wise ("FP8 Training Infrastructure", sections "O panorama da
 *    precisao numerica" and "Estrategias de escalonamento"; "Practical FP4
 *    Training for Large-Scale MoE Models on Hopper GPUs", section 2,
 *    kernel BF16ToFP4Row and the transposed FP4RowToFP8Col layout).
 *  - A block-scaled GEMM with FP32 accumulation that consumes codes and
 *    scales directly on the tensor cores (MoE FP4 page, section 2, heavy
 *    GEMMs stay on native FP8 tensor cores), dense and grouped over ragged
 *    expert batches (same section, "tensores ragged").
 *  - The direct integer-domain MXFP4 -> MXFP8 re-encode (same section,
 *    "Algoritmo de Conversao Direta"; kernel FP4RowToFP8Row), also writing
 *    per-expert padded scales for the grouped GEMM.
 *  - Around that path: FP4RowToFP8Col (MXFP4 rows to MXFP8 columns in one
 *    pass, same section, "Kernels"), MXFP4 -> FP8 with 1 x 128 blocks (the
 *    Hopper FP8 block of the same section), NVFP4 with delayed scaling
 *    from an amax history (FP8 page, "Estrategias de escalonamento"), and
 *    the GEMM on MXFP4 x MXFP4 operands natively.
 *
 * Conventions shared by every entry point
 *  - Matrices are row-major.  A GEMM computes C[M,N] = A[M,K] * B[N,K]^T:
 *    both operands are stored K-major (K is the contiguous last axis).
 *  - "Row-wise" quantization puts blocks along the last (contiguous) axis.
 *    "Column-wise" puts blocks along axis 0 and stores the TRANSPOSE: the
 *    column-wise output of a [R, C] input is a [C, R] tensor whose blocks
 *    run along its last axis, so every GEMM operand is K-major.
 *  - Codes: FP8 formats one byte per element; FP4 formats two elements per
 *    byte, the even-index element in the low nibble.
 *  - Scales: one byte per block (E8M0 for the MX formats, UE4M3 for NVFP4),
 *    stored in 512-byte tiles of 128 rows x 4 scale columns: the byte of
 *    scale (r, c) of a [rows, S] scale matrix is at
 *        ((r/128) * ceil(S/4) + c/4) * 512 + (r%32)*16 + ((r/32)%4)*4 + c%4.
 *    Rows are padded to a multiple of 128, scale columns to a multiple of
 *    4, and padding bytes are zero.  This is the scale-operand layout the
 *    tcgen05 block-scaled MMA reads.
 *  - MX block scale: e = floor(log2(block amax)) - emax, emax = 8 (E4M3),
 *    15 (E5M2), 2 (E2M1), clamped to [-127, 127]; an all-zero block gets
 *    e = -127; a block holding NaN/Inf gets scale 0xFF and NaN codes
 *    (E2M1: zero codes).  Codes are round-to-nearest-even of x * 2^-e with
 *    saturation to +-448 / +-57344 / +-6; the sign of zero is kept.
 *  - NVFP4: s_t = amax(finite |x|) / 2688 in FP32 (1 when the amax is 0);
 *    per 16-block s_b = UE4M3(RNE((amax_b / 6) / s_t)); codes are
 *    E2M1(RNE(x / (s_b * s_t))) with each step an IEEE FP32 operation; a
 *    zero s_b gives zero codes; a block holding NaN/Inf gets s_b = 0x7F and
 *    zero codes.
 *
 * Ownership: the caller allocates and frees every buffer (sizes from
 * bsq_codes_bytes / bsq_scales_bytes / bsq_grouped_scales_bytes).  Pointers passed to the compute
 * calls are DEVICE pointers.  The library keeps no allocation between calls;
 * its only state is a device status word in static device memory.
 *
 * Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  All
 * compute calls are asynchronous on that stream.
 *
 * Errors: arguments are checked on the host before any launch; on failure
 * the call returns a status, launches nothing and writes nothing.  An empty
 * tensor (0 rows or 0 columns) is BSQ_ERR_INVALID_ARG; empty experts inside
 * a grouped batch (equal consecutive offsets) are valid.  The GEMMs and the
 * grouped re-encode take row counts up to 2^31 - 256 (their kernels index
 * rows in 32 bits; the grouped GEMM also bounds num_groups x B.rows);
 * larger ones are BSQ_ERR_UNSUPPORTED.  No C++
 * exception crosses this boundary.  Faults detected on the device (a wait
 * that exceeded its limit) set the device status word, which
 * bsq_sync_status() returns and clears.
 */
#ifndef BSQ_H
#define BSQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BSQ_OK = 0,
    BSQ_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, shape mismatch        */
    BSQ_ERR_UNSUPPORTED = 2,   /* valid request this library does not handle    */
    BSQ_ERR_ALIGNMENT = 3,     /* a pointer or a row pitch is not 16-byte aligned */
    BSQ_ERR_CUDA = 4,          /* a CUDA runtime call failed                    */
    BSQ_ERR_TIMEOUT = 5        /* a device-side wait ran past its limit         */
} bsq_status;

typedef enum {
    BSQ_MXFP8_E4M3 = 0,        /* E4M3 codes, 32-element blocks, E8M0 scales    */
    BSQ_MXFP8_E5M2 = 1,        /* E5M2 codes, 32-element blocks, E8M0 scales    */
    BSQ_MXFP4_E2M1 = 2,        /* E2M1 codes, 32-element blocks, E8M0 scales    */
    BSQ_NVFP4_E2M1 = 3         /* E2M1 codes, 16-element blocks, UE4M3 scales,
                                  plus one FP32 tensor scale                    */
} bsq_format;

typedef enum { BSQ_ROWWISE = 1, BSQ_COLWISE = 2, BSQ_BOTH = 3 } bsq_axis;

typedef enum { BSQ_OUT_F32 = 0, BSQ_OUT_BF16 = 1 } bsq_out;

/* A quantized tensor as stored: `rows` x `cols` logical elements with blocks
 * along `cols`.  codes / scales / tensor_scale are device pointers;
 * tensor_scale (one float) is used by NVFP4 only and may be NULL otherwise. */
typedef struct {
    int32_t fmt;               /* bsq_format */
    int32_t reserved;          /* must be 0  */
    int64_t rows;
    int64_t cols;
    void* codes;
    uint8_t* scales;
    float* tensor_scale;
} bsq_tensor;

/* Bytes of the code buffer of a rows x cols tensor (0 on a bad format). */
size_t bsq_codes_bytes(int32_t fmt, int64_t rows, int64_t cols);

/* Bytes of the tiled scale buffer: ceil(rows/128)*128 * ceil(S/4)*4 with
 * S = cols / block (0 on a bad format or when cols is not a block multiple). */
size_t bsq_scales_bytes(int32_t fmt, int64_t rows, int64_t cols);

/* Quantize a row-major BF16 matrix src[rows, cols] (device).
 *   axis BSQ_ROWWISE: out_row gets a [rows, cols] tensor (cols % block == 0).
 *   axis BSQ_COLWISE: out_col gets the transposed [cols, rows] tensor
 *                     (rows % block == 0).
 *   axis BSQ_BOTH:    both, from one read of src.
 * The caller fills the out tensors' fmt / rows / cols / pointers; they must
 * match the request.  For NVFP4 each written tensor's tensor_scale must be a
 * device float; the call computes the tensor amax first (two passes).
 * Citations: FP8 page "Estrategias de escalonamento" (block scaling); MoE
 * FP4 page section 2, BF16ToFP4Row (row quantize and pack) and the
 * transposed operand of FP4RowToFP8Col. */
bsq_status bsq_quantize(const void* src_bf16, int64_t rows, int64_t cols, int32_t fmt, int32_t axis,
                        bsq_tensor* out_row, bsq_tensor* out_col, void* stream);

/* NVFP4 quantize with delayed scaling: one pass instead of two.  The tensor
 * scale is taken from the amax of previous steps instead of this tensor:
 *   s_t = max(amax_history) / 2688 (FP32; positive finite entries only;
 *         1 when there is none),
 * the blocks are then encoded as by bsq_quantize with that s_t (values
 * beyond its range saturate to the largest block scale and code), each
 * written tensor_scale receives s_t, and last this tensor's amax (largest
 * finite |x|) is pushed to the front of amax_history and its oldest entry
 * dropped.  amax_history: DEVICE float[history_len], 4-byte aligned, owned
 * by the caller, read and updated in stream order (zero-filled before the
 * first step); 1 <= history_len <= 4096.  Arguments and outputs otherwise
 * as bsq_quantize with fmt = BSQ_NVFP4_E2M1; on an argument error nothing
 * is launched and the history is unchanged.  Citation: FP8 page,
 * "Transformer Engine: a fundacao de software" (DelayedScaling recipe:
 * amax_history_len = 16, amax_compute_algo = "max", margin = 0) and
 * "Estrategias de escalonamento e estabilidade" (scale factors from the
 * statistics of previous iterations). */
bsq_status bsq_quantize_nvfp4_delayed(const void* src_bf16, int64_t rows, int64_t cols, int32_t axis,
                                      bsq_tensor* out_row, bsq_tensor* out_col, float* amax_history,
                                      int32_t history_len, void* stream);

/* Exact dequantization dst[rows, cols] = code * scale (* tensor scale),
 * rounded once to FP32 or BF16 (nearest-even).  dst is device memory,
 * 16-byte aligned.  Citation: MoE FP4 page section 2 (the dequantization
 * step that FP4RowToFP8Row replaces). */
bsq_status bsq_dequantize(const bsq_tensor* in, void* dst, int32_t dst_type, void* stream);

/* C[M,N] = A[M,K] * B[N,K]^T with FP32 accumulation on tcgen05 block-scaled
 * tensor-core MMAs; C row-major with leading dimension N, FP32 or BF16.
 * Supported pairs: any of MXFP8 E4M3 / E5M2 with each other; NVFP4 with
 * NVFP4 (the result is multiplied by both tensor scales); MXFP4 with MXFP4
 * (native FP4 MMA with UE8M0 scales, no re-encode).  K = A.cols =
 * B.cols; K % 32 == 0.  M, N >= 1 of any size.  Citation: MoE FP4 page
 * section 2 ("Calculo Intenso": GEMMs stay on native FP8 tensor cores);
 * FP8 page "MXFP8 e NVFP4 do Blackwell" (hardware block scaling). */
bsq_status bsq_gemm(const bsq_tensor* A, const bsq_tensor* B, void* C, int32_t out_type, void* stream);

/* Grouped GEMM over ragged expert batches: for g in [0, num_groups)
 *   C[o_g:o_{g+1}, :] = A[o_g:o_{g+1}, :] * B_g^T
 * where o = group_offsets_dev (DEVICE int64[num_groups+1], o_0 = 0,
 * non-decreasing, o_G = A.rows).  B_groups is a HOST array of num_groups
 * tensors of identical shape [N, K] and format; their code buffers must be
 * consecutive slices of one allocation (B_g.codes = B_0.codes + g * codes
 * bytes); scale buffers may be anywhere.  A's scales use the plain tiled
 * layout of the whole [A.rows, K] matrix.  num_groups <= 256; MXFP8
 * (any mix of E4M3 / E5M2) or MXFP4 x MXFP4; for MXFP4 the experts' scale
 * buffers must also be evenly spaced (BSQ_ERR_UNSUPPORTED otherwise).
 * Citation: MoE FP4 page section 2, ragged tensors whose per-expert token
 * counts vary. */
bsq_status bsq_grouped_gemm(const bsq_tensor* A, const int64_t* group_offsets_dev, int32_t num_groups,
                            const bsq_tensor* B_groups, void* C, int32_t out_type, void* stream);

/* Per-expert padded scale layout of a grouped activation tensor A[rows, cols]
 * with expert row offsets o (o_0 = 0, non-decreasing, o_G = rows): the scales
 * of expert g's rows start at scale row P_g = sum over earlier experts of
 * their row counts rounded up to 128, so no 128x4 scale tile holds two
 * experts (the tile layout itself is the plain one, over P_G rows; bytes
 * between experts are zero).  Codes keep their plain row-major layout.
 * This returns the buffer size that holds it for any offsets:
 * (ceil(rows/128)*128 + 128*num_groups) * ceil(S/4)*4, S = cols / block;
 * 0 on a bad format, shape or group count (1..256). */
size_t bsq_grouped_scales_bytes(int32_t fmt, int64_t rows, int64_t cols, int32_t num_groups);

/* MXFP4 -> MXFP8 re-encode (as bsq_mxfp4_to_mxfp8) whose output scales are
 * written in the per-expert padded layout for the given DEVICE offsets
 * (int64[num_groups+1]); out->scales must hold
 * bsq_grouped_scales_bytes(BSQ_MXFP8_E4M3, rows, cols, num_groups) bytes
 * (zero-filled by the call).  Offsets are clamped to [0, rows] and made
 * non-decreasing on the device.  Citation: MoE FP4 page section 2
 * (FP4RowToFP8Row feeding the per-expert FP8 GEMM). */
bsq_status bsq_mxfp4_to_mxfp8_grouped(const bsq_tensor* in_mxfp4, bsq_tensor* out_e4m3,
                                      const int64_t* group_offsets_dev, int32_t num_groups, void* stream);

/* Grouped GEMM as bsq_grouped_gemm, with A's scales in the per-expert padded
 * layout (as written by bsq_mxfp4_to_mxfp8_grouped).  Output tiles then start
 * at each expert's first row, so only the last tile of an expert is partly
 * idle (with the plain layout a 128-row scale tile shared by two experts is
 * computed for both).  Same formats, limits and errors as
 * bsq_grouped_gemm. */
bsq_status bsq_grouped_gemm_padded(const bsq_tensor* A, const int64_t* group_offsets_dev, int32_t num_groups,
                                   const bsq_tensor* B_groups, void* C, int32_t out_type, void* stream);

/* Direct MXFP4 -> MXFP8 (E4M3) re-encode in the integer domain, same shape
 * and block grid.  Per 32-block with scale exponent e and largest code
 * magnitude exponent e_c: new scale e + e_c - 8 (clamped at -127), every
 * code moved to the E4M3 code of the same value.  The result equals the
 * E4M3 MX quantization of the exactly dequantized MXFP4 block.  Citation:
 * MoE FP4 page section 2, "Algoritmo de Conversao Direta" and kernel
 * FP4RowToFP8Row. */
bsq_status bsq_mxfp4_to_mxfp8(const bsq_tensor* in_mxfp4, bsq_tensor* out_e4m3, void* stream);

/* FP4RowToFP8Col: dequantize a row-wise MXFP4 tensor in[R, C], transpose and
 * re-quantize column-wise to MXFP8 E4M3: out[C, R] holds the K-major codes
 * of the transpose with E8M0 scales over 32-row blocks of each column.  The
 * result equals the column-wise E4M3 MX quantization of the exactly
 * dequantized input (computed in the integer domain, no BF16 or FP32
 * intermediate that could round); a NaN row scale makes its blocks NaN.
 * R % 32 == 0 and C % 32 == 0; out->rows == C, out->cols == R; buffers as
 * for bsq_mxfp4_to_mxfp8 (device, caller-owned, 16-byte aligned).
 * Citation: MoE FP4 page section 2, "Kernels" (FP4RowToFP8Col: fused
 * dequantization, transposition and requantization for the weight
 * gradient). */
bsq_status bsq_mxfp4_to_mxfp8_col(const bsq_tensor* in_mxfp4, bsq_tensor* out_e4m3, void* stream);

/* MXFP4 -> FP8 E4M3 with 1 x 128 blocks, the FP8 block of the pages'
 * Hopper path.  Per row, each group of four 32-blocks (128 elements; the
 * last group of a row may hold fewer) takes the largest of their E8M0 scale
 * bytes S as its scale, and every element becomes the E4M3 code (RNE) of
 * its exact value code * 2^(s - 127) over 2^(S - 127), s its own block's
 * scale.  Exact while s >= S - 5; blocks further below round into E4M3's
 * subnormals and then to zero.  A NaN scale byte (0xFF) in a group makes
 * its scale 0xFF and all its codes NaN (0x7F).
 *   in_mxfp4:   row-wise MXFP4 tensor [rows, cols], cols % 32 == 0 (device)
 *   out_codes:  DEVICE [rows, cols] E4M3 bytes, row-major, 16-byte aligned
 *               (BSQ_ERR_ALIGNMENT otherwise), caller-owned
 *   out_scales: DEVICE [rows, ceil(cols / 128)] E8M0 bytes, row-major,
 *               caller-owned
 * Asynchronous on `stream`.  Citation: MoE FP4 page section 2, "Algoritmo
 * de Conversao Direta" (FP8 blocks of 128, the largest of four FP4 block
 * scales, exponents adjusted locally). */
bsq_status bsq_mxfp4_to_fp8_1x128(const bsq_tensor* in_mxfp4, void* out_codes, void* out_scales, void* stream);

/* Take and clear the device status word (one atomic exchange on the
 * device, ordered after the work already on `stream`), synchronize
 * `stream`, and return BSQ_ERR_TIMEOUT if any kernel recorded a timed-out
 * wait since the word was last taken, BSQ_ERR_CUDA if the stream reported an
 * error, else BSQ_OK.  The word is shared by every stream of the device: a
 * timeout recorded by a kernel on another stream is reported by whichever
 * call takes the word first. */
bsq_status bsq_sync_status(void* stream);

/* Test hook for the failure path: launches one kernel that waits on a
 * barrier nothing ever arrives on, gives up after `limit_ns` nanoseconds
 * (capped at 1e9) and records BSQ_ERR_TIMEOUT in the status word.  It
 * touches no memory besides the status word. */
bsq_status bsq_debug_timeout_probe(uint64_t limit_ns, void* stream);

/* Test hook for the GEMM kernels' failure path: bsq_gemm with every wait of
 * the kernel limited to `timeout_ns` nanoseconds (1 .. 4e9; bsq_gemm uses
 * 4e9) instead of the default.  With a limit shorter than the GEMM takes,
 * the kernel gives up part-way: it records BSQ_ERR_TIMEOUT in the status
 * word, lets every stage load, scale copy and MMA it issued land, releases
 * tensor memory and exits; C is then partly written.  `kernel` 0 runs the
 * kernel bsq_gemm would choose, 1 the single-CTA kernel (not for MXFP4,
 * BSQ_ERR_UNSUPPORTED).  Argument rules and errors as for bsq_gemm. */
bsq_status bsq_debug_gemm_timeout(const bsq_tensor* A, const bsq_tensor* B, void* C, int32_t out_type,
                                  uint64_t timeout_ns, int32_t kernel, void* stream);

/* Static description of a status code. */
const char* bsq_status_string(int32_t status);

/* Library version string. */
const char* bsq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BSQ_H */
