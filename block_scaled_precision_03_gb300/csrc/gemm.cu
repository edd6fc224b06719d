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
//   warp 1      TMEM owner and MMA issuer: per stage four tcgen05.mma ...
//               block_scale with M=128, N=256; commits free the smem stage
//               and, per tile, signal the epilogue.
//   warps 2-9   epilogue: drain the 128 x 256 FP32 accumulator from TMEM to
//               registers, release TMEM to the MMA warp, then scale (NVFP4
//               tensor scales), convert and store C.
//   warp 10     scale copies: each stage's atoms into a per-stage TMEM slot
//               (tcgen05.cp 32x128b.warpx4) as soon as the stage lands, apart
//               from the MMA thread so that copies and MMAs overlap.
// Every wait is bounded: past the time limit the kernel records a timeout in
// the status word, drains its own in-flight copies and MMAs and exits.
#include <cuda.h>
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "epilogue.cuh"
#include "tmap.h"

namespace bsq {
namespace {
using namespace tc;

constexpr int BM = 128;            // tile rows (A)
constexpr int BN = 256;            // tile columns (B rows)
constexpr int BKB = 128;           // K bytes per stage (one 128-byte swizzle row)
constexpr int STAGES = 4;
constexpr int kEpiWarps = 8;
constexpr int kCopyWarp = 2 + kEpiWarps;   // scale-copy issuer
constexpr int kThreads = 32 * (3 + kEpiWarps);
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
    // epilogue staging for TMA stores (FP8 only: the NVFP4 ring leaves no room)
    static constexpr int OUT_STAGE = FP4 ? 0 : kEpiWarps * 2048;
    static constexpr int SMEM = 1024 + STAGES * (A_BYTES + B_BYTES + SF_STAGE) + OUT_STAGE + 256 + 8 * (kMaxGroups + 1) +
                                8 * kMaxGroups;
    static_assert(SMEM <= 232448, "shared memory per block");
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
    int32_t out_bf16, vec_ok, tma_store;
    const float* ts_a;
    const float* ts_b;
    uint32_t idesc;
    int32_t num_groups;
    int32_t gsf;                   // grouped: A's scales in the per-expert padded layout
    const int64_t* offsets;
    unsigned* status;
    uint64_t timeout_ns;
    const uint8_t* sfb_group[kMaxGroups];
};

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
        ti.a_row0 = p.gsf ? gt->lo[g] + (local % cnt) * BM : band * BM;
        ti.band = band; ti.b_row0 = g * p.N + nt * BN; ti.n0 = nt * BN;
        ti.row_lo = max(gt->lo[g], ti.a_row0); ti.row_hi = min(gt->hi[g], ti.a_row0 + BM);
        ti.group = g;
    }
    return ti;
}

template <bool FP4>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, const __grid_constant__ Params p) {
    using CF = Cfg<FP4>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smA = base;
    uint8_t* smB = base + STAGES * A_BYTES;
    uint8_t* smSF = smB + STAGES * B_BYTES;
    uint8_t* smOut = smSF + STAGES * CF::SF_STAGE;      // epilogue staging, 2 KB per warp (FP8)
    uint64_t* bars = reinterpret_cast<uint64_t*>(smOut + CF::OUT_STAGE);
    // bars: full[STAGES], empty[STAGES], sfready[STAGES], tfull, tempty, drain (MMAs), cdrain (copies)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    GroupTable* gt = reinterpret_cast<GroupTable*>(bars + 32);
    static_assert(8 * (3 * STAGES + 4) + 8 <= 256, "barrier area");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES), sfr0 = smem_u32(bars + 2 * STAGES);
    const uint32_t tfull = smem_u32(bars + 3 * STAGES), tempty = smem_u32(bars + 3 * STAGES + 1);
    const uint32_t drain = smem_u32(bars + 3 * STAGES + 2), cdrain = smem_u32(bars + 3 * STAGES + 3);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
            mbar_init(sfr0 + 8 * s, 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, kEpiWarps);
        mbar_init(drain, 1);
        mbar_init(cdrain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), kTmemCols);
    }
    int total = p.total_tiles;
    if (p.num_groups > 0 && warp == 2 && lane == 0) {
        // boundaries clamped to [0, M] and non-decreasing (expert 0 starts at 0)
        int acc = 0, prev = 0, pband = 0;
        gt->prefix[0] = 0;
        for (int g = 0; g < p.num_groups; g++) {
            const int lo = prev;
            const int hi = max(lo, clamp_rows(p.offsets[g + 1], 0, p.M));
            prev = hi;
            int b0, cnt;
            if (p.gsf) {
                // per-expert padded scale layout: tiles start at the expert's first row
                cnt = (hi - lo + BM - 1) / BM;
                b0 = pband;
                pband += cnt;
            } else {
                b0 = lo / BM;
                cnt = hi > lo ? (hi + BM - 1) / BM - b0 : 0;
            }
            gt->band0[g] = b0; gt->lo[g] = lo; gt->hi[g] = hi;
            acc += cnt * p.n_tiles;
            gt->prefix[g + 1] = acc;
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (p.num_groups > 0) total = gt->prefix[p.num_groups];
    const uint32_t tmem = *tmem_slot;

    // producer state kept for the drain at exit
    int stage = 0, issued = 0;
    uint32_t phase = 0;
    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int gcur = 0;
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
            if (!ok) *abort_flag = 1;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // Per stage: wait for the operands (full) and for the stage's scales in
        // tensor memory (sfready, committed by the scale-copy warp), issue the
        // stage's four MMAs, commit the stage back to the producer.
        if (lane == 0) {
            constexpr int MPS = 4;
            const uint64_t ad_base = desc_sw128(smem_u32(smA));
            const uint64_t bd_base = desc_sw128(smem_u32(smB));
            const uint32_t sf_t0 = tmem + kSfCol0;
            int stage = 0;
            uint32_t phase = 0;
            int iter = 0;
            bool ok = true, any = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++iter) {
                if (!mbar_wait(tempty, (iter & 1) ^ 1, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
                fence_after();
                for (int kb = 0; kb < p.k_stages; kb++) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status, p.timeout_ns) ||
                        !mbar_wait(sfr0 + 8 * stage, phase, abort_flag, p.status, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const int nk = kb == p.k_stages - 1 ? p.mma_last : MPS;
                    const uint32_t sfa_t = sf_t0 + stage * CF::SF_COLS, sfb_t = sfa_t + (FP4 ? 16 : 4);
                    const uint64_t ad = ad_base + (uint64_t)((stage * A_BYTES) >> 4);
                    const uint64_t bd = bd_base + (uint64_t)((stage * B_BYTES) >> 4);
#pragma unroll
                    for (int m = 0; m < MPS; m++) {
                        if (m < nk) {
                            const uint32_t acc = (kb | m) != 0;
                            // +32 bytes along K inside the 128-byte swizzle row = +2 in the address field
                            if (FP4) mma<1, kMmaNV>(tmem, ad + 2 * m, bd + 2 * m, p.idesc, sfa_t + 4 * m, sfb_t + 8 * m, acc);
                            else mma<1, kMmaFP8>(tmem, ad + 2 * m, bd + 2 * m,
                                                 p.idesc | ((uint32_t)m << 4) | ((uint32_t)m << 29), sfa_t, sfb_t, acc);
                        }
                    }
                    any = true;
                    commit<1>(empty0 + 8 * stage);
                    if (kb == p.k_stages - 1) commit<1>(tfull);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) *abort_flag = 1;
            if (any) {
                // every MMA issued finishes before TMEM is released (the epilogue,
                // which otherwise sees the last tile finish, may have given up)
                commit<1>(drain);
                volatile int no_abort = 0;
                mbar_wait(drain, 0, &no_abort, nullptr, 100000000ull);
            }
        }
    } else if (warp == kCopyWarp) {
        // ------------------------------------------------ scale copies
        // Copies each stage's scale atoms into the stage's TMEM slot as soon as
        // the stage has landed (the slot is free: the producer reloads a stage
        // only after the MMAs that read it completed) and commits sfready.
        // Issued apart from the MMAs, the copies overlap with them instead of
        // holding up the next MMA.
        if (lane == 0) {
            constexpr int NCP = 3 * CF::SF_ATOMS;
            const uint64_t sfd_base = desc_sf(smem_u32(smSF));
            const uint32_t sf_t0 = tmem + kSfCol0;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, any = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                for (int kb = 0; kb < p.k_stages; kb++) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
                    fence_after();
                    const uint64_t sd = sfd_base + (uint64_t)((stage * CF::SF_STAGE) >> 4);
                    const uint32_t sfa_t = sf_t0 + stage * CF::SF_COLS, sfb_t = sfa_t + (FP4 ? 16 : 4);
                    // copy c: atom c / 3, part c % 3 (A; B rows 0-127; B rows 128-255)
#pragma unroll
                    for (int c = 0; c < NCP; c++) {
                        const int at = c / 3, part = c % 3;
                        if (part == 0) cp_sf<1>(sfa_t + 4 * at, sd + 32 * at);
                        else cp_sf<1>(sfb_t + 8 * at + 4 * (part - 1),
                                      sd + ((CF::SFA_BYTES + ((part - 1) * CF::SF_ATOMS + at) * 512) >> 4));
                    }
                    commit<1>(sfr0 + 8 * stage);
                    any = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) *abort_flag = 1;
            if (any) {
                // every copy lands before TMEM is released
                commit<1>(cdrain);
                volatile int no_abort = 0;
                mbar_wait(cdrain, 0, &no_abort, nullptr, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2-9)
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int h = (warp - 2) >> 2;          // column half
        // NVFP4 tensor scales, applied one after the other (their product alone can underflow)
        float alpha = 1.0f, beta = 1.0f;
        if (FP4) {
            alpha = *p.ts_a;
            beta = *p.ts_b;
        }
        int iter = 0, gcur = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++iter) {
            const TileInfo ti = tile_info(p, t, gt, gcur);
            if (!mbar_wait(tfull, iter & 1, abort_flag, p.status, p.timeout_ns)) break;
            fence_after();
            uint32_t r[4][32];
            const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128);
            BSQ_TMEM_LD32(r[0], ta);
            BSQ_TMEM_LD32(r[1], ta + 32);
            BSQ_TMEM_LD32(r[2], ta + 64);
            BSQ_TMEM_LD32(r[3], ta + 96);
            tmem_wait_ld();
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);

            // this warp's 32 rows, clipped to the rows the tile may write
            const int row0 = ti.a_row0 + q * 32;
            const int col0 = ti.n0 + h * 128;
            const int lo = max(row0, ti.row_lo), hi = min(row0 + 32, ti.row_hi);
            if (lo >= hi || col0 >= p.N) continue;
            if (!FP4 && p.tma_store && lo == row0 && hi == row0 + 32) {
                const uint32_t buf = smem_u32(smOut + (warp - 2) * 2048);
                if (p.out_bf16) store_tile_tma<true>(r, buf, &tmC, col0, row0, alpha, beta, lane);
                else store_tile_tma<false>(r, buf, &tmC, col0, row0, alpha, beta, lane);
            } else if (row0 + lane >= lo && row0 + lane < hi) {
                store_row128(r, p.C, p.ldc, row0 + lane, col0, p.N, p.out_bf16, p.vec_ok, alpha, beta);
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0 && *abort_flag) {
        // some role gave up: the stage loads still in flight (at most the last
        // STAGES issued; an older stage was reloaded only after it had landed)
        // land before the CTA exits
        const int pending = min(issued, STAGES);
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < pending; i++) {
            if (--s < 0) { s = STAGES - 1; ph ^= 1; }
            volatile int no_abort = 0;
            mbar_wait(full0 + 8 * s, ph, &no_abort, nullptr, 100000000ull);
        }
    }
    __syncthreads();
    if (warp == 1) {
        fence_after();
        tmem_dealloc<1>(tmem, kTmemCols);
    }
}

// ----------------------------------------------------------------- host
template <bool FP4>
cudaError_t launch(const GemmArgs& a, const Params& p, const CUtensorMap& ta, const CUtensorMap& tb,
                   const CUtensorMap& tc_, int grid, cudaStream_t st) {
    static bool attr_done = false;
    cudaError_t e;
    if (!attr_done) {
        e = cudaFuncSetAttribute(gemm_kernel<FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<FP4>::SMEM);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    gemm_kernel<FP4><<<grid, kThreads, Cfg<FP4>::SMEM, st>>>(ta, tb, tc_, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t run_gemm(const GemmArgs& a, cudaStream_t st) {
    // Grouped GEMMs go to CTA pairs whenever their layout allows (one tensor
    // map over the experts' scales) and A's scales are in the per-expert
    // padded layout: the pair's 256 x 256 tiles halve the operand traffic per
    // FLOP, which outweighs the half tile an expert with an odd number of
    // 128-row bands leaves idle (measured on the 64-expert Zipf workload:
    // 0.405 ms against 0.435 ms).  With the plain layout a pair tile starts on
    // A's own bands, idles more rows, and is chosen only when the experts
    // average at least kPairRowsPerGroup rows.
    constexpr int64_t kPairRowsPerGroup = 1024;
    // MXFP4 x MXFP4 exists only on the CTA-pair kernel (kind::mxf4)
    if (a.fmt_a == kMXFP4) return run_gemm_pair(a, st);
    if (!a.single_cta) {
        if (a.num_groups == 0) return run_gemm_pair(a, st);
        if (gemm_pair_grouped_ok(a) &&
            (a.grouped_pair || a.a_grouped_sf || a.M >= kPairRowsPerGroup * a.num_groups))
            return run_gemm_pair(a, st);
    }
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
    if (fp4) p.idesc = make_idesc(1, 1, false, BM, BN);
    else p.idesc = make_idesc(a.fmt_a == kE5M2 ? 1 : 0, a.fmt_b == kE5M2 ? 1 : 0, true, BM, BN);
    p.num_groups = a.num_groups;
    p.gsf = a.num_groups > 0 && a.a_grouped_sf;
    p.offsets = a.offsets;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    for (int g = 0; g < a.num_groups; g++) p.sfb_group[g] = a.b_group_scales[g];

    CUtensorMap ta, tb;
    const int64_t b_rows = a.num_groups ? a.N * a.num_groups : a.N;
    if (!tmap::codes_2d(&ta, a.a_codes, a.M, kbytes, BM)) return cudaErrorInvalidValue;
    if (!tmap::codes_2d(&tb, a.b_codes, b_rows, kbytes, BN)) return cudaErrorInvalidValue;
    // TMA stores of whole 32-row boxes when the output's base and row pitch allow them
    CUtensorMap tcm = ta;
    p.tma_store = !fp4 && p.vec_ok && tmap::out_2d(&tcm, a.C, a.M, a.N, a.N, a.out_bf16 != 0);
    if (!p.tma_store) tcm = ta;
    int grid = a.num_sms;
    if (a.num_groups == 0 && p.total_tiles < grid) grid = p.total_tiles;
    if (grid < 1) grid = 1;
    return fp4 ? launch<true>(a, p, ta, tb, tcm, grid, st) : launch<false>(a, p, ta, tb, tcm, grid, st);
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
