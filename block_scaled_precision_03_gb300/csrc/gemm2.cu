// Block-scaled GEMM on a CTA pair (tcgen05 cta_group::2), sm_103a: dense,
// and grouped over experts; MXFP8 (E4M3 / E5M2), NVFP4 and MXFP4 operands.
//
// C[M,N] = A[M,K] * B[N,K]^T with per-block scales and FP32 accumulation
// ("Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// section 2, "Calculo Intenso": the heavy GEMMs run on the native low-
// precision tensor cores; "FP8 Training Infrastructure", section "MXFP8 e
// NVFP4 do Blackwell": hardware block scaling).
//
// Two CTAs of a cluster (one per SM of a TPC) compute one 256 x 256 output
// tile with M=256 MMAs issued by the even CTA.  Each CTA stages only its
// own 128 rows of A and its own 128 rows of B per K step, so a CTA holds
// 32 KB of operands per stage (a 1-CTA 128 x 256 tile needs 48 KB) and the
// ring holds 3 stages of 256 K-bytes (MXFP4: 5 of 128, NVFP4: 4 of 128).
// The tcgen05 instruction queue is about one MMA deep, so the issuing
// thread runs in lockstep with the tensor pipe; every barrier handshake
// costs pipe time, and larger stages (8 MMAs per handshake) amortize it.
// Each CTA also keeps the full 256-row B scale tile so its tensor memory
// holds the scales its half of the MMA reads (a pair's scale copy fills each
// CTA's tensor memory from that CTA's own shared memory).
//
// Roles (both CTAs, 11 warps each):
//   warp 0      TMA producer: own A / B halves and scale atoms; completion is
//               signalled on the even CTA's stage barrier (cta_group::2 TMA)
//   warp 1      TMEM owner (both CTAs); the even CTA's lane 0 issues the MMAs
//               and multicasts the commits that free stages and tiles
//   warps 2-9   epilogue on each CTA's own 128 accumulator rows
//   warp 10     the even CTA's lane 0 copies each stage's scales into tensor
//               memory (tcgen05.cp) as soon as the stage lands, apart from the
//               MMA thread: a scale copy costs the issuing thread about as
//               long as an MMA, and from a second thread the copies overlap
//               with the MMAs instead of queueing between them
// Every wait is bounded; a CTA that gave up records the status, and before
// the pair exits every MMA, scale copy and stage load it issued has landed.
#include <algorithm>
#include <cuda.h>
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "epilogue.cuh"
#include "tmap.h"

namespace bsq {
namespace {

constexpr int BN = 256;              // output columns per pair
constexpr int BKB = 128;             // K bytes per stage
constexpr int HALF = 128 * BKB;      // 16 KB: one CTA's 128 rows of A (or B)
constexpr int kEpiWarps = 8;
constexpr int kCopyWarp = 2 + kEpiWarps;           // scale-copy issuer
constexpr int kThreads = 32 * (3 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;
constexpr int kRasterGroup = 8;      // default tiles per raster group
constexpr int64_t kL2Resident = 48ll << 20;   // operand bytes that stay in L2 while the other streams

// Grouped mode: per expert g its rows [lo, hi) of A and C, its first 128-row
// band of A and the number of 256-row tiles (pairs of bands) covering it;
// prefix[g] = tiles of the experts before g.
struct GroupTable2 {
    int32_t prefix[kMaxGroups + 1];
    int32_t band0[kMaxGroups];
    int32_t pairs[kMaxGroups];
    int32_t lo[kMaxGroups];
    int32_t hi[kMaxGroups];
};
constexpr int kGroupTableBytes = (int)sizeof(GroupTable2);

// Operand kinds: MXFP8 (E4M3 / E5M2), NVFP4, MXFP4 (E2M1 with UE8M0 scales
// per 32, the MoE page's activation format, multiplied natively).
constexpr int kKindFP8 = tc::kMmaFP8, kKindNV = tc::kMmaNV, kKindMX4 = tc::kMmaMX4;

template <int KIND>
struct Cfg2 {
    static constexpr bool FP4 = KIND != kKindFP8;
    // KSUB 128-byte K sub-steps per stage: more MMAs per barrier handshake.
    // FP4 stages stay at 128 bytes: the scales of a 256-byte MXFP4 stage
    // (6 KB) would not leave room for three stages and the epilogue.
    static constexpr int KSUB = FP4 ? 1 : 2;
    // NVFP4 (one scale atom per MMA) takes B's scales four times over, laid
    // out for one 128x256b copy per atom instead of two 32x128b.warpx4: 8
    // scale copies per stage instead of 12, for 12 KB more scale bytes per
    // stage and one stage less.  (The same for A's scales, or for MXFP4's B
    // scales, costs more in loads and stages than it saves in copies.)
    static constexpr bool SFB_QUARTERS = KIND == kKindNV;
    static constexpr int STAGES = FP4 ? (SFB_QUARTERS ? 4 : 5) : 3;
    static constexpr int MPS = 4 * KSUB;                  // MMAs per stage
    static constexpr int OP_BYTES = KSUB * HALF;          // one CTA's A (or B) bytes per stage
    // 512-byte scale atoms (4 scale columns x 128 rows) per 128 rows per stage
    static constexpr int SF_ATOMS = KSUB * (KIND == kKindNV ? 4 : (KIND == kKindMX4 ? 2 : 1));
    static constexpr int SFA_BYTES = SF_ATOMS * 512;
    static constexpr int SFB_BYTES = SFB_QUARTERS ? SF_ATOMS * 4096 : 2 * SF_ATOMS * 512;
    static constexpr int SF_STAGE = SFA_BYTES + SFB_BYTES;
    static constexpr uint32_t SFA_COLS = 4 * SF_ATOMS;    // TMEM columns: SFA atoms, then SFB atom pairs
    static constexpr uint32_t SF_COLS = 12 * SF_ATOMS;
    static constexpr uint32_t OP_TX = 2 * OP_BYTES;       // operand bytes one CTA loads per stage
    static constexpr uint32_t SF_TX = SF_STAGE;           // scale bytes one CTA loads per stage
    static constexpr int SMEM = 1024 + STAGES * (2 * OP_BYTES + SF_STAGE) + kEpiWarps * 2048 + 256 + kGroupTableBytes;
    static_assert(kSfCol0 + STAGES * SF_COLS <= kTmemCols, "TMEM columns");
    static_assert(SMEM <= 232448, "shared memory per block");
};

struct Params2 {
    int32_t M, N;
    int32_t k_stages, mma_last;
    int32_t m_tiles, n_tiles, total_tiles;
    void* C;
    int64_t ldc;
    int32_t out_bf16, vec_ok, tma_store;
    const float* ts_a;
    const float* ts_b;
    uint32_t idesc;
    int32_t raster, raster_n;
    int32_t num_groups;            // 0 = dense
    int32_t gsf;                   // grouped: A's scales in the per-expert padded layout
    int32_t group_bands;           // 128-row bands of one expert's B
    const int64_t* offsets;        // grouped: device row offsets, num_groups + 1
    unsigned* status;
    uint64_t timeout_ns;
};

// Tile order: groups of `raster` tiles along one dimension, swept along the
// other (raster_n: the groups run along n).  A group spanning the whole of
// the smaller operand keeps that operand resident in L2 while the other one
// streams through once.
__device__ __forceinline__ void tile_mn(const Params2& p, int t, int& mt, int& nt) {
    const int MT = p.raster_n ? p.n_tiles : p.m_tiles, NT = p.raster_n ? p.m_tiles : p.n_tiles;
    const int per_group = p.raster * NT;
    const int g = t / per_group;
    const int first = g * p.raster;
    const int gm = min(p.raster, MT - first);
    const int local = t - g * per_group;
    const int a = first + local % gm, b = local / gm;
    if (p.raster_n) { mt = b; nt = a; } else { mt = a; nt = b; }
}

// After an abort: the even CTA's producer makes every stage load still in
// flight land before the pair exits.  Load k (k-th stage load of a CTA) goes
// to stage k % S, barrier phase (k / S) & 1, on the even CTA; the even CTA
// arms each load with both CTAs' bytes.  A load one CTA issued and the other
// did not gets its barrier accounting completed here (the missing half's
// bytes retired with complete_tx, or the arrival and the odd half's bytes
// expected), then its phase is awaited with a time limit.  Loads older than
// the last S of the CTA that issued more have landed already: a stage is
// reloaded only after the MMAs that read its previous load completed.
__device__ __noinline__ void drain_pair_loads(uint32_t full0, int S, int n_own, int n_peer, uint32_t cta_tx) {
    const int n = max(n_own, n_peer);
    for (int k = max(0, n - S); k < n; k++) {
        const uint32_t bar = full0 + 8 * (uint32_t)(k % S);
        const uint32_t parity = (uint32_t)((k / S) & 1);
        const bool own = k < n_own, peer = k < n_peer;
        if (own && !peer) tc::mbar_complete_tx(bar, cta_tx);
        if (peer && !own) tc::mbar_expect_tx(bar, cta_tx);
        volatile int no_abort = 0;
        tc::mbar_wait(bar, parity, &no_abort, nullptr, 100000000ull);
    }
}

// What one CTA of the pair loads and stores for tile t.  The two CTAs own
// one 128-row band of A each; in grouped mode both bands belong to the same
// expert (any two of its bands: each CTA loads its own), so a tile never
// mixes experts and at most half a tile is idle when an expert covers an odd
// number of bands.
struct Tile2 {
    int32_t a_row;         // this CTA's first row of A (and of C)
    int32_t a_band;        // its 128-row band of A's scale tiles
    int32_t nt;            // 256-column tile of C
    int32_t b_row;         // this CTA's first B row
    int32_t sfb_band;      // first of the tile's two B scale bands
    int32_t row_lo, row_hi;    // rows of C this CTA may write
};

__device__ __forceinline__ Tile2 tile2(const Params2& p, int t, const GroupTable2* gt, int& gcur, uint32_t rank) {
    Tile2 ti;
    if (p.num_groups == 0) {
        int mt, nt;
        tile_mn(p, t, mt, nt);
        ti.a_band = mt * 2 + (int)rank;
        ti.a_row = ti.a_band * 128;
        ti.nt = nt;
        ti.b_row = nt * BN + (int)rank * 128;
        ti.sfb_band = nt * 2;
        ti.row_lo = ti.a_band * 128;
        ti.row_hi = min(p.M, ti.row_lo + 128);
    } else {
        while (t >= gt->prefix[gcur + 1]) ++gcur;
        const int g = gcur;
        const int pairs = gt->pairs[g];
        const int local = t - gt->prefix[g];
        const int pi = local % pairs;
        ti.nt = local / pairs;
        ti.a_band = gt->band0[g] + 2 * pi + (int)rank;
        // plain scale layout: tiles sit on A's own 128-row bands; per-expert
        // padded layout: tiles start at the expert's first row
        ti.a_row = p.gsf ? gt->lo[g] + 128 * (2 * pi + (int)rank) : ti.a_band * 128;
        ti.b_row = g * p.N + ti.nt * BN + (int)rank * 128;
        ti.sfb_band = g * p.group_bands + ti.nt * 2;
        ti.row_lo = max(gt->lo[g], ti.a_row);
        ti.row_hi = min(gt->hi[g], ti.a_row + 128);
    }
    return ti;
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
gemm2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
             const __grid_constant__ CUtensorMap tmC, const __grid_constant__ Params2 p) {
    using CF = Cfg2<KIND>;
    constexpr int S = CF::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smSF = base;                                 // scales first: stage sizes are 1 KB multiples
    uint8_t* smA = base + S * CF::SF_STAGE;
    uint8_t* smB = smA + S * CF::OP_BYTES;
    uint8_t* smOut = smB + S * CF::OP_BYTES;              // epilogue staging, 2 KB per warp
    uint64_t* bars = reinterpret_cast<uint64_t*>(smOut + kEpiWarps * 2048);
    GroupTable2* gt = reinterpret_cast<GroupTable2*>(bars + 32);
    // bars: full[S] (operands), empty[S], sfready[S], sfull[S] (scales), sfree[S] (scales
    // read into tensor memory), tfull, tempty, drain (MMAs), cdrain (scale copies)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 5 * S + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* issued_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);   // operand loads this CTA issued
    volatile int* sf_issued_slot = reinterpret_cast<volatile int*>(tmem_slot + 3);   // scale loads it issued
    static_assert(8 * (5 * S + 4) + 16 <= 256, "barrier area");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_rank();
    const bool leader = rank == 0;
    const uint32_t full0 = tc::smem_u32(bars), empty0 = tc::smem_u32(bars + S), sfr0 = tc::smem_u32(bars + 2 * S);
    const uint32_t sfull0 = tc::smem_u32(bars + 3 * S), sfree0 = tc::smem_u32(bars + 4 * S);
    const uint32_t tfull = tc::smem_u32(bars + 5 * S), tempty = tc::smem_u32(bars + 5 * S + 1);
    const uint32_t drain = tc::smem_u32(bars + 5 * S + 2), cdrain = tc::smem_u32(bars + 5 * S + 3);
    const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < S; s++) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, 1);
            tc::mbar_init(sfr0 + 8 * s, 1);
            tc::mbar_init(sfull0 + 8 * s, 1);
            tc::mbar_init(sfree0 + 8 * s, 1);
        }
        tc::mbar_init(tfull, 1);
        tc::mbar_init(tempty, 2 * kEpiWarps);
        tc::mbar_init(drain, 1);
        tc::mbar_init(cdrain, 1);
        *abort_flag = 0;
        *issued_slot = 0;
        *sf_issued_slot = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tc::prefetch_tmap(&tmA);
        tc::prefetch_tmap(&tmB);
        tc::prefetch_tmap(&tmSFA);
        tc::prefetch_tmap(&tmSFB);
    }
    if (warp == 1) tc::tmem_alloc<2>(tc::smem_u32(tmem_slot), kTmemCols);
    if (p.num_groups > 0 && warp == 2) {
        // Expert table, 32 boundaries per pass.  Boundaries are clamped to
        // [0, M] and made non-decreasing (running max; expert 0 starts at 0),
        // so the experts never hold more than M rows in total.  Entry g of a
        // pass is boundary g; expert g - 1 is [boundary g - 1, boundary g).
        int carry = 0, bcarry = 0, prev = 0;
        for (int g0 = 0; g0 <= p.num_groups; g0 += 32) {
            const int g = g0 + lane;
            int om = (g >= 1 && g <= p.num_groups) ? clamp_rows(p.offsets[g], 0, p.M) : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, om, d);
                if (lane >= d) om = max(om, u);
            }
            om = max(om, prev);
            const int up = __shfl_up_sync(0xffffffffu, om, 1);
            const int lo = lane == 0 ? prev : up;
            const bool expert = g >= 1 && g <= p.num_groups;
            int nb = 0, pairs = 0;
            if (expert && om > lo) {
                nb = (om - lo + 127) / 128;                                  // 128-row tiles of the expert
                pairs = p.gsf ? (nb + 1) / 2 : ((om - 1) / 128 - lo / 128 + 2) / 2;
            }
            int vt = pairs * p.n_tiles, vb = nb;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int ut = __shfl_up_sync(0xffffffffu, vt, d), ub = __shfl_up_sync(0xffffffffu, vb, d);
                if (lane >= d) { vt += ut; vb += ub; }
            }
            if (expert) {
                const int e = g - 1;
                gt->lo[e] = lo;
                gt->hi[e] = om;
                gt->pairs[e] = pairs;
                gt->band0[e] = p.gsf ? bcarry + vb - nb : lo / 128;     // padded layout: 128-row tiles per expert
                gt->prefix[e + 1] = carry + vt;
            }
            carry += __shfl_sync(0xffffffffu, vt, 31);
            bcarry += __shfl_sync(0xffffffffu, vb, 31);
            prev = __shfl_sync(0xffffffffu, om, 31);
        }
        if (lane == 0) gt->prefix[0] = 0;
    }
    tc::fence_before();
    __syncthreads();
    tc::cluster_sync();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total = p.num_groups > 0 ? gt->prefix[p.num_groups] : p.total_tiles;
    const uint32_t sf_t0 = tmem + kSfCol0;

    if (warp == 0) {
        // ------------------------------------------------ TMA producers (both CTAs)
        // Lane 0 loads the operands of a stage once the MMAs that read its
        // previous contents completed (empty).  Lane 1 loads the stage's scales
        // once the scale copies read their previous contents into tensor
        // memory (sfree), which is up to a whole ring ahead of the operands, so
        // the copies of a stage are done long before its MMAs are issued.
        // Completion of both is signalled on the even CTA's barriers.
        if (lane == 0) {
            const uint32_t full_c0 = tc::mapa(full0, 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int gcur = 0, issued = 0;
            for (int t = cid; t < total && ok; t += ncl) {
                const Tile2 ti = tile2(p, t, gt, gcur, rank);
                const int arow = ti.a_row, brow = ti.b_row;
                for (int kb = 0; kb < p.k_stages; kb++) {
                    if (!tc::mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.status, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_c0 + 8 * stage;
                    if (leader) tc::mbar_expect_tx(full0 + 8 * stage, 2 * CF::OP_TX);
#pragma unroll
                    for (int j = 0; j < CF::KSUB; j++) {
                        const int kx = (kb * CF::KSUB + j) * BKB;
                        tc::tma_load_2d_pair(tc::smem_u32(smA + stage * CF::OP_BYTES + j * HALF), &tmA, kx, arow, fb);
                        tc::tma_load_2d_pair(tc::smem_u32(smB + stage * CF::OP_BYTES + j * HALF), &tmB, kx, brow, fb);
                    }
                    ++issued;
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            *issued_slot = issued;
            if (!ok) *abort_flag = 1;
        } else if (lane == 1) {
            const uint32_t sfull_c0 = tc::mapa(sfull0, 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int gcur = 0, issued = 0;
            for (int t = cid; t < total && ok; t += ncl) {
                const Tile2 ti = tile2(p, t, gt, gcur, rank);
                for (int kb = 0; kb < p.k_stages; kb++) {
                    if (!tc::mbar_wait(sfree0 + 8 * stage, phase ^ 1, abort_flag, p.status, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sb = sfull_c0 + 8 * stage;
                    if (leader) tc::mbar_expect_tx(sfull0 + 8 * stage, 2 * CF::SF_TX);
                    uint8_t* sf = smSF + stage * CF::SF_STAGE;
                    tc::tma_load_3d_pair(tc::smem_u32(sf), &tmSFA, 0, kb * CF::SF_ATOMS, ti.a_band, sb);
                    if (CF::SFB_QUARTERS) {
                        // both CTAs need the same B scale tile: the even CTA loads it once
                        // into both (multicast); the barrier still counts both copies
                        if (leader)
                            tc::tma_load_4d_pair_mc(tc::smem_u32(sf + CF::SFA_BYTES), &tmSFB, 0, 0, ti.sfb_band,
                                                    kb * CF::SF_ATOMS, sb, (uint16_t)0x3);
                    }
                    else
                        tc::tma_load_3d_pair(tc::smem_u32(sf + CF::SFA_BYTES), &tmSFB, 0, kb * CF::SF_ATOMS,
                                             ti.sfb_band, sb);
                    ++issued;
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            *sf_issued_slot = issued;
            if (!ok) *abort_flag = 1;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA)
        // Per stage: wait for the operands (full) and for the stage's scales in
        // tensor memory (sfready, committed by the scale-copy warp), issue the
        // stage's MMAs, commit the stage back to the producers.
        if (lane == 0 && leader) {
            constexpr int MPS = CF::MPS;
            constexpr uint32_t OP_STEP = CF::OP_BYTES >> 4, SUB_STEP = HALF >> 4;  // descriptor address units
            const uint64_t ad_base = tc::desc_sw128(tc::smem_u32(smA));
            const uint64_t bd_base = tc::desc_sw128(tc::smem_u32(smB));
            int stage = 0;
            uint32_t phase = 0;
            int iter = 0;
            bool ok = true, any = false;
            for (int t = cid; t < total && ok; t += ncl, ++iter) {
                // both CTAs' epilogue warps arrive here after their TMEM loads completed
                // (tcgen05.wait::ld); a CTA-scope acquire suffices
                if (!tc::mbar_wait(tempty, (iter & 1) ^ 1, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
                tc::fence_after();
                for (int kb = 0; kb < p.k_stages; kb++) {
                    if (!tc::mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status, p.timeout_ns) ||
                        !tc::mbar_wait(sfr0 + 8 * stage, phase, abort_flag, p.status, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t sfa_t = sf_t0 + stage * CF::SF_COLS, sfb_t = sfa_t + CF::SFA_COLS;
                    const uint64_t ad = ad_base + (uint64_t)(stage * OP_STEP), bd = bd_base + (uint64_t)(stage * OP_STEP);
                    const int nk = kb == p.k_stages - 1 ? p.mma_last : MPS;
#pragma unroll
                    for (int m = 0; m < MPS; m++) {
                        if (m < nk) {
                            const int sub = m >> 2, k = m & 3;
                            // +32 bytes along K inside a 128-byte swizzle row = +2 in the address field
                            const uint64_t adm = ad + sub * SUB_STEP + 2 * k, bdm = bd + sub * SUB_STEP + 2 * k;
                            const uint32_t acc = (kb | m) != 0;
                            // FP8 takes scale byte k of the sub-step's atom (1X), NVFP4 one atom
                            // per MMA (4X), MXFP4 the byte pair 2 (m & 1) of atom m >> 1 (2X)
                            if (KIND == kKindNV) {
                                tc::mma<2, tc::kMmaNV>(tmem, adm, bdm, p.idesc, sfa_t + 4 * m, sfb_t + 8 * m, acc);
                            } else if (KIND == kKindMX4) {
                                const uint32_t id = (uint32_t)(m & 1) * 2u;
                                tc::mma<2, tc::kMmaMX4>(tmem, adm, bdm, p.idesc | (id << 4) | (id << 29),
                                                        sfa_t + 4 * (m >> 1), sfb_t + 8 * (m >> 1), acc);
                            } else {
                                tc::mma<2, tc::kMmaFP8>(tmem, adm, bdm, p.idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29),
                                                        sfa_t + 4 * sub, sfb_t + 8 * sub, acc);
                            }
                        }
                    }
                    any = true;
                    tc::commit<2>(empty0 + 8 * stage, 3);
                    if (kb == p.k_stages - 1) tc::commit<2>(tfull, 3);
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) *abort_flag = 1;
            if (any) {
                // every MMA issued finishes before tensor memory is released (the
                // epilogue, which otherwise sees the last tile finish, may have given up)
                tc::commit<2>(drain, 1);
                volatile int no_abort = 0;
                tc::mbar_wait(drain, 0, &no_abort, nullptr, 100000000ull);
            }
        }
    } else if (warp < kCopyWarp) {
        // ------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const uint32_t tempty_c0 = tc::mapa(tempty, 0);
        // NVFP4: the two tensor scales are applied one after the other, so that
        // their product is never formed on its own (it can underflow FP32)
        float alpha = 1.0f, beta = 1.0f;
        if (KIND == kKindNV) {
            alpha = *p.ts_a;
            beta = *p.ts_b;
        }
        int iter = 0, gcur = 0;
        for (int t = cid; t < total; t += ncl, ++iter) {
            const Tile2 ti = tile2(p, t, gt, gcur, rank);
            if (!tc::mbar_wait(tfull, iter & 1, abort_flag, p.status, p.timeout_ns)) break;
            tc::fence_after();
            uint32_t r[4][32];
            const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128);
            BSQ_TMEM_LD32(r[0], ta);
            BSQ_TMEM_LD32(r[1], ta + 32);
            BSQ_TMEM_LD32(r[2], ta + 64);
            BSQ_TMEM_LD32(r[3], ta + 96);
            tc::tmem_wait_ld();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster(tempty_c0);
            // this warp's 32 rows, clipped to the rows the CTA may write
            const int row0 = ti.a_row + q * 32;
            const int col0 = ti.nt * BN + h * 128;
            const int lo = max(row0, ti.row_lo), hi = min(row0 + 32, ti.row_hi);
            if (lo >= hi || col0 >= p.N) continue;
            if (p.tma_store && (hi == row0 + 32 || hi == p.M) && lo == row0) {
                // whole box (rows past M are clipped by the tensor map)
                const uint32_t buf = tc::smem_u32(smOut + (warp - 2) * 2048);
                if (p.out_bf16) store_tile_tma<true>(r, buf, &tmC, col0, row0, alpha, beta, lane);
                else store_tile_tma<false>(r, buf, &tmC, col0, row0, alpha, beta, lane);
            } else if (row0 + lane >= lo && row0 + lane < hi) {
                store_row128(r, p.C, p.ldc, row0 + lane, col0, p.N, p.out_bf16, p.vec_ok, alpha, beta);
            }
        }
        if (lane == 0) tc::bulk_wait_all();
    } else {
        // ------------------------------------------------ scale copies (even CTA)
        // Copies each stage's scale atoms from shared memory into the stage's
        // tensor-memory slot as soon as the stage's scales have landed (they
        // load on their own barrier, ahead of the operands; a slot is free once
        // its stage was loaded again: the producer reloads a stage only after
        // the MMAs that read it completed), then commits sfready.  Issued apart
        // from the MMAs, the copies overlap with them.
        if (lane == 0 && leader) {
            constexpr int NCP = 3 * CF::SF_ATOMS;
            const uint32_t sf_smem = tc::smem_u32(smSF);
            const uint64_t sfd_base = tc::desc_sf(sf_smem);
            constexpr uint32_t SF_STEP = CF::SF_STAGE >> 4;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, any = false;
            for (int t = cid; t < total && ok; t += ncl) {
                for (int kb = 0; kb < p.k_stages; kb++) {
                    // the stage's scales have landed, and the MMAs that read the stage's
                    // tensor-memory slot last time have completed
                    if (!tc::mbar_wait(sfull0 + 8 * stage, phase, abort_flag, p.status, p.timeout_ns) ||
                        !tc::mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.status, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint64_t sd = sfd_base + (uint64_t)(stage * SF_STEP);
                    const uint32_t sfa_t = sf_t0 + stage * CF::SF_COLS, sfb_t = sfa_t + CF::SFA_COLS;
                    if (CF::SFB_QUARTERS) {
                        // per atom: A's 512-byte 128x4 tile broadcast to the four lane
                        // quarters, B's two tiles as one 128 x 32-byte matrix already
                        // laid out four times over ([band][quarter][row][16 bytes])
                        const uint32_t sfb_s = sf_smem + stage * CF::SF_STAGE + CF::SFA_BYTES;
#pragma unroll
                        for (int a = 0; a < CF::SF_ATOMS; a++) {
                            tc::cp_sf<2>(sfa_t + 4 * a, sd + 32 * a);
                            tc::cp_sf_128x256<2>(sfb_t + 8 * a, tc::desc_sf_ns(sfb_s + a * 4096, 2048, 128));
                        }
                    } else {
                        // copy c: atom c / 3, part c % 3 (A; B rows 0-127; B rows 128-255), each
                        // one 512-byte 128x4 tile broadcast to the four lane quarters
#pragma unroll
                        for (int c = 0; c < NCP; c++) {
                            const int a = c / 3, part = c % 3;
                            if (part == 0) tc::cp_sf<2>(sfa_t + 4 * a, sd + 32 * a);
                            else tc::cp_sf<2>(sfb_t + 8 * a + 4 * (part - 1),
                                              sd + ((CF::SFA_BYTES + ((part - 1) * CF::SF_ATOMS + a) * 512) >> 4));
                        }
                    }
                    tc::commit<2>(sfr0 + 8 * stage, 1);
                    tc::commit<2>(sfree0 + 8 * stage, 3);         // both CTAs' scale slots are free again
                    any = true;
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) *abort_flag = 1;
            if (any) {
                // every scale copy issued lands before tensor memory is released
                tc::commit<2>(cdrain, 1);
                volatile int no_abort = 0;
                tc::mbar_wait(cdrain, 0, &no_abort, nullptr, 100000000ull);
            }
        }
    }

    // Both CTAs have stopped issuing.  If either gave up, the even CTA waits
    // (bounded) for every stage load still in flight: all loads report to its
    // barriers, and a CTA must not exit while copies into its shared memory
    // or onto its barriers may still land.
    tc::fence_before();
    __syncthreads();
    tc::cluster_sync();
    if (leader && warp == 0 && lane == 0) {
        const int peer_abort = tc::ld_cluster_s32(tc::mapa(tc::smem_u32((const void*)abort_flag), 1));
        if (*abort_flag || peer_abort) {
            const int n_own = *issued_slot;
            const int n_peer = tc::ld_cluster_s32(tc::mapa(tc::smem_u32((const void*)issued_slot), 1));
            const int sf_own = *sf_issued_slot;
            const int sf_peer = tc::ld_cluster_s32(tc::mapa(tc::smem_u32((const void*)sf_issued_slot), 1));
            // per scale load the odd CTA's bytes: its own scale tiles (NVFP4: A's only,
            // the even CTA's multicast carries B's into both)
            drain_pair_loads(sfull0, S, sf_own, sf_peer, CF::SFB_QUARTERS ? CF::SFA_BYTES : CF::SF_TX);
            drain_pair_loads(full0, S, n_own, n_peer, CF::OP_TX);
        }
    }
    tc::cluster_sync();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc<2>(tmem, kTmemCols);
    }
}

template <int KIND>
cudaError_t launch2(const Params2& p, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                    const CUtensorMap& tsb, const CUtensorMap& tc_, int grid, cudaStream_t st) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(gemm2_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg2<KIND>::SMEM);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    gemm2_kernel<KIND><<<grid, kThreads, Cfg2<KIND>::SMEM, st>>>(ta, tb, tsa, tsb, tc_, p);
    return cudaGetLastError();
}

}  // namespace

// True when a grouped GEMM can run on CTA pairs: MXFP8, whole 128-row scale
// bands per expert and the experts' scale buffers evenly spaced (one tensor
// map then spans all of them).
bool gemm_pair_grouped_ok(const GemmArgs& a) {
    if (a.num_groups < 1 || a.fmt_a == kNVFP4 || a.N % 128 != 0) return false;     // MXFP8 or MXFP4
    const int64_t n_atoms = (a.K / 32 + 3) / 4;
    const int64_t stride = (a.N / 128) * n_atoms * 512;
    for (int g = 0; g < a.num_groups; g++)
        if (a.b_group_scales[g] != a.b_group_scales[0] + g * stride) return false;
    return true;
}

// Block-scaled GEMM on CTA pairs: dense, or grouped over experts when
// gemm_pair_grouped_ok() holds.
cudaError_t run_gemm_pair(const GemmArgs& a, cudaStream_t st) {
    const int kind = a.fmt_a == kNVFP4 ? kKindNV : (a.fmt_a == kMXFP4 ? kKindMX4 : kKindFP8);
    const bool fp4 = kind != kKindFP8;
    const int64_t kbytes = fp4 ? a.K / 2 : a.K;
    const int64_t S = a.K / (kind == kKindNV ? 16 : 32);
    const int64_t n_atoms = (S + 3) / 4;
    Params2 p{};
    p.M = (int32_t)a.M;
    p.N = (int32_t)a.N;
    const int64_t stage_kb = (int64_t)BKB * (fp4 ? Cfg2<kKindNV>::KSUB : Cfg2<kKindFP8>::KSUB);
    p.k_stages = (int32_t)((kbytes + stage_kb - 1) / stage_kb);
    p.mma_last = (int32_t)((kbytes - (int64_t)(p.k_stages - 1) * stage_kb + 31) / 32);
    p.m_tiles = (int32_t)((a.M + 255) / 256);
    p.n_tiles = (int32_t)((a.N + BN - 1) / BN);
    p.total_tiles = p.m_tiles * p.n_tiles;
    p.C = a.C;
    p.ldc = a.N;
    p.out_bf16 = a.out_bf16;
    const int esz = a.out_bf16 ? 2 : 4;
    p.vec_ok = ((reinterpret_cast<uintptr_t>(a.C) & 15) == 0) && ((a.N * esz) % 16 == 0);
    p.ts_a = a.ts_a;
    p.ts_b = a.ts_b;
    // E2M1 operands are type 1 in the FP4 kinds; UE8M0 scales except NVFP4's UE4M3
    p.idesc = fp4 ? make_idesc(1, 1, kind == kKindMX4, 256, BN)
                  : make_idesc(a.fmt_a == kE5M2 ? 1 : 0, a.fmt_b == kE5M2 ? 1 : 0, true, 256, BN);
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    const bool grouped = a.num_groups > 0;
    p.num_groups = a.num_groups;
    p.gsf = grouped && a.a_grouped_sf;
    p.offsets = a.offsets;
    p.group_bands = (int32_t)(a.N / 128);
    // raster order: sweep the larger operand past the whole of the smaller one
    // when the smaller one fits in L2 with room to spare
    {
        const int64_t a_bytes = a.M * kbytes, b_bytes = a.N * kbytes;
        p.raster = kRasterGroup;
        p.raster_n = 0;
        if (std::min(a_bytes, b_bytes) <= kL2Resident) {
            p.raster_n = b_bytes < a_bytes;
            p.raster = p.raster_n ? p.n_tiles : p.m_tiles;
        }
    }

    const int sf_atoms = kind == kKindNV ? Cfg2<kKindNV>::SF_ATOMS
                       : (kind == kKindMX4 ? Cfg2<kKindMX4>::SF_ATOMS : Cfg2<kKindFP8>::SF_ATOMS);
    CUtensorMap ta, tb, tsa, tsb;
    if (!tmap::codes_2d(&ta, a.a_codes, a.M, kbytes, 128)) return cudaErrorInvalidValue;
    const int64_t b_rows = grouped ? a.N * a.num_groups : a.N;
    const uint8_t* b_sf = grouped ? a.b_group_scales[0] : a.b_scales;
    if (!tmap::codes_2d(&tb, a.b_codes, b_rows, kbytes, 128)) return cudaErrorInvalidValue;
    // the per-expert padded scale layout spans up to one extra 128-row tile per expert
    const int64_t a_bands = (a.M + 127) / 128 + (p.gsf ? a.num_groups : 0);
    if (!tmap::scales_3d(&tsa, a.a_scales, a_bands, n_atoms, sf_atoms, 1)) return cudaErrorInvalidValue;
    if (kind == kKindNV) {
        if (!tmap::scales_4d_quarters(&tsb, b_sf, (b_rows + 127) / 128, n_atoms, sf_atoms, 2))
            return cudaErrorInvalidValue;
    } else if (!tmap::scales_3d(&tsb, b_sf, (b_rows + 127) / 128, n_atoms, sf_atoms, 2)) {
        return cudaErrorInvalidValue;
    }
    // TMA stores of the output when its base and row pitch allow them
    CUtensorMap tcm = ta;
    p.tma_store = p.vec_ok && tmap::out_2d(&tcm, a.C, a.M, a.N, a.N, a.out_bf16 != 0);
    if (!p.tma_store) tcm = ta;
    int pairs = a.num_sms / 2;
    if (!grouped && p.total_tiles < pairs) pairs = p.total_tiles;
    if (pairs < 1) pairs = 1;
    if (kind == kKindNV) return launch2<kKindNV>(p, ta, tb, tsa, tsb, tcm, 2 * pairs, st);
    if (kind == kKindMX4) return launch2<kKindMX4>(p, ta, tb, tsa, tsb, tcm, 2 * pairs, st);
    return launch2<kKindFP8>(p, ta, tb, tsa, tsb, tcm, 2 * pairs, st);
}

}  // namespace bsq
