// Block-scaled GEMM on the sm_103a tensor cores (tcgen05), dense and grouped.
//
// C[M,N] = A[M,K] * B[N,K]^T, both operands K-major codes with per-block
// scales, FP32 accumulation in tensor memory.  This is the heavy GEMM of the
// low-precision linear layer ("Practical FP4 Training for Large-Scale MoE
// Models on Hopper GPUs", section 2, "Calculo Intenso": GEMMs run on native
// FP8 tensor cores; "FP8 Training Infrastructure", section "MXFP8 e NVFP4 do
// Blackwell": block scaling is done by the hardware).  The grouped variant
// walks ragged expert batches (MoE page, section 2, "tensores ragged").
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: A tile 128 x 128 B and B tile 256 x 128 B per
//               stage (128-byte swizzle) plus the stage's scale atoms (bulk
//               copies of 512-byte 128x4 tiles), into a 4-stage smem ring.
//   warp 1      TMEM owner and MMA issuer: per stage copies the scale atoms
//               into a per-stage TMEM slot (tcgen05.cp 32x128b.warpx4) and
//               issues four tcgen05.mma ... block_scale with M=128, N=256;
//               commits free the smem stage and, per tile, signal the
//               epilogue.
//   warps 2-9   epilogue: drain the 128 x 256 FP32 accumulator from TMEM to
//               registers, release TMEM to the MMA warp, then scale (NVFP4
//               tensor scales), convert and store C.
// Every wait is bounded: past the time limit the kernel records a timeout in
// the status word, drains its own in-flight copies and MMAs and exits.
#include <cuda.h>
#include "common.cuh"
#include "internal.h"

namespace bsq {
namespace {

constexpr int BM = 128;            // tile rows (A)
constexpr int BN = 256;            // tile columns (B rows)
constexpr int BKB = 128;           // K bytes per stage (one 128-byte swizzle row)
constexpr int STAGES = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;  // scale slots start after the accumulator
constexpr int A_BYTES = BM * BKB;
constexpr int B_BYTES = BN * BKB;
constexpr int kRasterGroup = 16;   // m-tiles per raster group (L2 reuse)

template <bool FP4>
struct Cfg {
    static constexpr int SF_ATOMS = FP4 ? 4 : 1;         // 512-byte atoms per 128 rows per stage
    static constexpr int SFA_BYTES = SF_ATOMS * 512;
    static constexpr int SFB_BYTES = 2 * SF_ATOMS * 512;
    static constexpr int SF_STAGE = SFA_BYTES + SFB_BYTES;
    static constexpr uint32_t SF_COLS = FP4 ? 48 : 12;   // TMEM columns per stage slot
    static constexpr int SMEM = 1024 + STAGES * (A_BYTES + B_BYTES + SF_STAGE) + 256 + 8 * (kMaxGroups + 1) + 8 * kMaxGroups;
};

struct Params {
    const uint8_t* sfa;
    const uint8_t* sfb;
    int64_t sfa_band;              // bytes per 128-row band of A scales
    int64_t sfb_band;
    int32_t n_atoms;               // scale atoms along K
    int32_t M, N;
    int32_t k_stages;
    int32_t mma_last;              // MMAs in the last stage (1..4)
    int32_t m_tiles, n_tiles, total_tiles;
    int32_t b_bands;               // 128-row bands of B (per group)
    void* C;
    int64_t ldc;
    int32_t out_bf16, vec_ok;
    const float* ts_a;
    const float* ts_b;
    uint32_t idesc;
    int32_t num_groups;
    const int64_t* offsets;
    unsigned* status;
    uint64_t timeout_ns;
    const uint8_t* sfb_group[kMaxGroups];
};

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred P;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, P;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait: false when the CTA is aborting or the time limit passed.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       unsigned* status, uint64_t limit_ns) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 255u) == 255u) {
            if (*abort_flag) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > limit_ns) {
                *abort_flag = 1;
                record_status(status, kStatusTimeout);
                return false;
            }
        }
    }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y, uint32_t bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar) : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}
template <bool FP4>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc) {
    if (FP4) {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
                     :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
    } else {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
                     :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
    }
}
#define BSQ_LD32(r, taddr)                                                                              \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"  \
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"              \
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),   \
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),            \
                   "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),         \
                   "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),         \
                   "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),         \
                   "=r"(r[31])                                                                           \
                 : "r"(taddr))

// Shared-memory matrix descriptor, K-major operand tile with 128-byte
// swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Descriptor of one 512-byte scale atom: 32 rows of 16 bytes, no swizzle,
// 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

struct TileInfo {
    int32_t a_row0;       // first A row of the tile (multiple of 128)
    int32_t band;         // A scale band
    int32_t b_row0;       // first B row (in the [groups*N, K] view)
    int32_t n0;           // first output column
    int32_t row_lo, row_hi;   // rows of C this tile may write
    int32_t group;
};

struct GroupTable {
    int32_t prefix[kMaxGroups + 1];
    int32_t band0[kMaxGroups];
    int32_t lo[kMaxGroups];
    int32_t hi[kMaxGroups];
};

__device__ __forceinline__ TileInfo tile_info(const Params& p, int t, const GroupTable* gt, int& gcur) {
    TileInfo ti;
    if (p.num_groups == 0) {
        const int per_group = kRasterGroup * p.n_tiles;
        const int g = t / per_group;
        const int first_m = g * kRasterGroup;
        const int gm = min(kRasterGroup, p.m_tiles - first_m);
        const int local = t - g * per_group;
        const int mt = first_m + local % gm, nt = local / gm;
        ti.a_row0 = mt * BM; ti.band = mt; ti.b_row0 = nt * BN; ti.n0 = nt * BN;
        ti.row_lo = mt * BM; ti.row_hi = min(p.M, mt * BM + BM);
        ti.group = 0;
    } else {
        while (t >= gt->prefix[gcur + 1]) ++gcur;
        const int g = gcur;
        const int cnt = (gt->prefix[g + 1] - gt->prefix[g]) / p.n_tiles;
        const int local = t - gt->prefix[g];
        const int nt = local / cnt, band = gt->band0[g] + local % cnt;
        ti.a_row0 = band * BM; ti.band = band; ti.b_row0 = g * p.N + nt * BN; ti.n0 = nt * BN;
        ti.row_lo = max(gt->lo[g], band * BM); ti.row_hi = min(gt->hi[g], band * BM + BM);
        ti.group = g;
    }
    return ti;
}

template <bool FP4>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ Params p) {
    using CF = Cfg<FP4>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smA = base;
    uint8_t* smB = base + STAGES * A_BYTES;
    uint8_t* smSF = smB + STAGES * B_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smSF + STAGES * CF::SF_STAGE);
    // bars: full[STAGES], empty[STAGES], tfull, tempty, drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    GroupTable* gt = reinterpret_cast<GroupTable*>(bars + 32);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t tfull = smem_u32(bars + 2 * STAGES), tempty = smem_u32(bars + 2 * STAGES + 1);
    const uint32_t drain = smem_u32(bars + 2 * STAGES + 2);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, kEpiWarps);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    int total = p.total_tiles;
    if (p.num_groups > 0 && warp == 2 && lane == 0) {
        int acc = 0;
        gt->prefix[0] = 0;
        for (int g = 0; g < p.num_groups; g++) {
            const int lo = (int)p.offsets[g], hi = (int)p.offsets[g + 1];
            const int b0 = lo / BM, b1 = (hi + BM - 1) / BM;
            const int cnt = hi > lo ? b1 - b0 : 0;
            gt->band0[g] = b0; gt->lo[g] = lo; gt->hi[g] = hi;
            acc += cnt * p.n_tiles;
            gt->prefix[g + 1] = acc;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (p.num_groups > 0) total = gt->prefix[p.num_groups];
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int gcur = 0;
            int issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileInfo ti = tile_info(p, t, gt, gcur);
                const uint8_t* sfb_base = p.num_groups ? p.sfb_group[ti.group] : p.sfb;
                const int nb = ti.n0 / 128;                       // first B scale band of the tile
                for (int kb = 0; kb < p.k_stages; kb++) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
                    const uint32_t fb = full0 + 8 * stage;
                    const int atom0 = kb * CF::SF_ATOMS;
                    const int natoms = min(CF::SF_ATOMS, p.n_atoms - atom0);
                    const int bands = min(2, p.b_bands - nb);
                    const uint32_t sf_bytes = (uint32_t)(natoms * 512 * (1 + bands));
                    mbar_expect_tx(fb, A_BYTES + B_BYTES + sf_bytes);
                    tma_load_2d(smem_u32(smA + stage * A_BYTES), &tmA, kb * BKB, ti.a_row0, fb);
                    tma_load_2d(smem_u32(smB + stage * B_BYTES), &tmB, kb * BKB, ti.b_row0, fb);
                    uint8_t* sf = smSF + stage * CF::SF_STAGE;
                    bulk_load(smem_u32(sf), p.sfa + ti.band * p.sfa_band + atom0 * 512, natoms * 512, fb);
                    for (int rt = 0; rt < bands; rt++)
                        bulk_load(smem_u32(sf + CF::SFA_BYTES + rt * CF::SF_ATOMS * 512),
                                  sfb_base + (int64_t)(nb + rt) * p.sfb_band + atom0 * 512, natoms * 512, fb);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                const int pending = min(issued, STAGES);
                int s = stage;
                uint32_t ph = phase;
                for (int i = 0; i < pending; i++) {
                    if (--s < 0) { s = STAGES - 1; ph ^= 1; }
                    volatile int no_abort = 0;
                    mbar_wait(full0 + 8 * s, ph, &no_abort, nullptr, 100000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int iter = 0;
            bool ok = true, any = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++iter) {
                if (!mbar_wait(tempty, (iter & 1) ^ 1, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                for (int kb = 0; kb < p.k_stages; kb++) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem + kSfCol0 + stage * CF::SF_COLS;
                    const uint32_t sfb_t = sfa_t + (FP4 ? 16 : 4);
                    const uint32_t sf_s = smem_u32(smSF + stage * CF::SF_STAGE);
                    for (int a = 0; a < CF::SF_ATOMS; a++) {
                        tc_cp_sf(sfa_t + 4 * a, desc_sf(sf_s + a * 512));
                        for (int rt = 0; rt < 2; rt++)
                            tc_cp_sf(sfb_t + 8 * a + 4 * rt, desc_sf(sf_s + CF::SFA_BYTES + (rt * CF::SF_ATOMS + a) * 512));
                    }
                    const uint32_t a_s = smem_u32(smA + stage * A_BYTES), b_s = smem_u32(smB + stage * B_BYTES);
                    const int nk = kb == p.k_stages - 1 ? p.mma_last : 4;
                    for (int k = 0; k < nk; k++) {
                        const uint64_t ad = desc_sw128(a_s + 32 * k), bd = desc_sw128(b_s + 32 * k);
                        if (FP4) {
                            tc_mma<true>(tmem, ad, bd, p.idesc, sfa_t + 4 * k, sfb_t + 8 * k, (kb | k) != 0);
                        } else {
                            const uint32_t id = p.idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29);
                            tc_mma<false>(tmem, ad, bd, id, sfa_t, sfb_t, (kb | k) != 0);
                        }
                    }
                    any = true;
                    tc_commit(empty0 + 8 * stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit(tfull);
            }
            if (!ok && any) {
                // wait for the MMAs already issued before TMEM is released
                tc_commit(drain);
                volatile int no_abort = 0;
                mbar_wait(drain, 0, &no_abort, nullptr, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int h = (warp - 2) >> 2;          // column half
        float alpha = 1.0f;
        if (FP4) alpha = __fmul_rn(*p.ts_a, *p.ts_b);
        int iter = 0, gcur = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++iter) {
            const TileInfo ti = tile_info(p, t, gt, gcur);
            if (!mbar_wait(tfull, iter & 1, abort_flag, p.status, p.timeout_ns)) break;
            tc_fence_after();
            uint32_t r[4][32];
            const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128);
            BSQ_LD32(r[0], ta);
            BSQ_LD32(r[1], ta + 32);
            BSQ_LD32(r[2], ta + 64);
            BSQ_LD32(r[3], ta + 96);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);

            const int row = ti.a_row0 + q * 32 + lane;
            const int col0 = ti.n0 + h * 128;
            if (row < ti.row_lo || row >= ti.row_hi || col0 >= p.N) continue;
            if (p.out_bf16) {
                __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc + col0;
                if (p.vec_ok && col0 + 128 <= p.N) {
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
                        if (col0 + j < p.N) out[j] = __float2bfloat16_rn(__uint_as_float(r[j >> 5][j & 31]) * alpha);
                }
            } else {
                float* out = reinterpret_cast<float*>(p.C) + (int64_t)row * p.ldc + col0;
                if (p.vec_ok && col0 + 128 <= p.N) {
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
                        if (col0 + j < p.N) out[j] = __uint_as_float(r[j >> 5][j & 31]) * alpha;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ----------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t row_bytes, uint32_t box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)BKB, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// tcgen05 instruction descriptor (block-scaled kinds), without scale ids:
// bits 7-9 A type, 10-12 B type, 17-22 N>>3, 23 scale type (1 = UE8M0),
// 24-28 M>>4; K-major A and B, no negation, dense.
uint32_t make_idesc(uint32_t atype, uint32_t btype, bool ue8m0) {
    return (atype << 7) | (btype << 10) | ((uint32_t)(BN >> 3) << 17) | ((ue8m0 ? 1u : 0u) << 23) |
           ((uint32_t)(BM >> 4) << 24);
}

template <bool FP4>
cudaError_t launch(const GemmArgs& a, const Params& p, const CUtensorMap& ta, const CUtensorMap& tb, int grid,
                   cudaStream_t st) {
    static bool attr_done = false;
    cudaError_t e;
    if (!attr_done) {
        e = cudaFuncSetAttribute(gemm_kernel<FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<FP4>::SMEM);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    gemm_kernel<FP4><<<grid, kThreads, Cfg<FP4>::SMEM, st>>>(ta, tb, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t run_gemm(const GemmArgs& a, cudaStream_t st) {
    const bool fp4 = a.fmt_a == kNVFP4;
    const int64_t kbytes = fp4 ? a.K / 2 : a.K;
    const int blk = fp4 ? 16 : 32;
    Params p{};
    const int64_t S = a.K / blk;
    p.n_atoms = (int32_t)((S + 3) / 4);
    p.sfa = a.a_scales;
    p.sfb = a.b_scales;
    p.sfa_band = (int64_t)p.n_atoms * 512;
    p.sfb_band = p.sfa_band;
    p.M = (int32_t)a.M;
    p.N = (int32_t)a.N;
    p.k_stages = (int32_t)((kbytes + BKB - 1) / BKB);
    p.mma_last = (int32_t)((kbytes - (int64_t)(p.k_stages - 1) * BKB + 31) / 32);
    p.m_tiles = (int32_t)((a.M + BM - 1) / BM);
    p.n_tiles = (int32_t)((a.N + BN - 1) / BN);
    p.total_tiles = p.m_tiles * p.n_tiles;
    p.b_bands = (int32_t)((a.N + 127) / 128);
    p.C = a.C;
    p.ldc = a.N;
    p.out_bf16 = a.out_bf16;
    const int esz = a.out_bf16 ? 2 : 4;
    p.vec_ok = ((reinterpret_cast<uintptr_t>(a.C) & 15) == 0) && ((a.N * esz) % 16 == 0);
    p.ts_a = a.ts_a;
    p.ts_b = a.ts_b;
    if (fp4) p.idesc = make_idesc(1, 1, false);
    else p.idesc = make_idesc(a.fmt_a == kE5M2 ? 1 : 0, a.fmt_b == kE5M2 ? 1 : 0, true);
    p.num_groups = a.num_groups;
    p.offsets = a.offsets;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    for (int g = 0; g < a.num_groups; g++) p.sfb_group[g] = a.b_group_scales[g];

    CUtensorMap ta, tb;
    const int64_t b_rows = a.num_groups ? a.N * a.num_groups : a.N;
    if (!make_map(&ta, a.a_codes, a.M, kbytes, BM)) return cudaErrorInvalidValue;
    if (!make_map(&tb, a.b_codes, b_rows, kbytes, BN)) return cudaErrorInvalidValue;
    int grid = a.num_sms;
    if (a.num_groups == 0 && p.total_tiles < grid) grid = p.total_tiles;
    if (grid < 1) grid = 1;
    return fp4 ? launch<true>(a, p, ta, tb, grid, st) : launch<false>(a, p, ta, tb, grid, st);
}

// ------------------------------------------------------------ timeout probe
__global__ void timeout_probe_kernel(unsigned* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // nothing ever arrives on `bar`: the wait must give up and report
        mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
    }
}

cudaError_t run_timeout_probe(unsigned* status, uint64_t limit_ns, cudaStream_t st) {
    timeout_probe_kernel<<<1, 32, 0, st>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace bsq
