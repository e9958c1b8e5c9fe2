// hgemm_fp8bs.cuh - the block-scaled FP8 GEMM kernel for sm_103a:
//
//   C[i][j] = bf16( sum_kb  a_scale[i / bs][kb] * b_scale[kb][j / bs]
//                           * sum_{k in block kb} A[i][k] * B[k][j] )
//
// A (M x K) and B (K x N) are row-major E4M3 or E5M2 patterns, each
// bs x bs sub-block of A and of B carrying one fp32 factor (bs = 32 or 64):
// "深度学习加速核心：GEMM优化从分块到TensorCore的实战解析", section 4.3 (FP8 data
// is scaled block-wise, one factor per 32 x 32 or 64 x 64 sub-block) and
// section 5.2, the third mishap (the factors must be 32-bit: a 16-bit one
// overflowed). C is bfloat16, rounded once to nearest even.
//
// A factor that varies along K cannot be taken out of one tensor-core sum,
// and the hardware's own block-scaled MMA kinds take only power-of-two (UE8M0)
// factors. So the sum is split at the scale blocks:
//
//   MMA warp   for each scale block (bs / 32 kind::f8f6f4 MMAs of K = 32) it
//              writes the block's fp32 partial sum into one of four 128-column
//              TMEM buffers (accumulate flag off for the block's first MMA).
//              The buffers go back and forth in pairs: one wait and one commit
//              per two blocks, because every hand-off between two warps costs
//              about 300 cycles however little they do (a bare skeleton of
//              this ring, measured), against 128 cycles of tensor work in a
//              64-deep block. The tensor core runs up to two pairs ahead.
//   epilogue   kBsEpiWarps warps; warp w owns TMEM lane quarter w % 4 (32 rows
//              of C, one per thread) and the 128 / (kBsEpiWarps / 4) columns of
//              column group w / 4. For each scale block it loads its part of
//              the partial (tcgen05.ld), forms the factor a_scale * b_scale in
//              fp32 (one per 32-column load: the row block is warp-uniform
//              because a quarter's 32 rows lie in one scale block) and adds
//              factor x partial into fp32 registers (fmaf); a pair's buffers
//              go back once both are read. The factors come from a per-warp
//              ring in shared memory that cp.async fills several blocks ahead.
//              After the last block it rounds to bf16 and stores its row.
//   producers  as in the main kernel: TMA loads of 128 x 128-byte A boxes and
//              128-row B atoms (read MN-major in the 128-byte swizzle), two
//              warps on alternate stages of a 7-stage ring.
//
// The epilogue's fp32 work per scale block equals the tensor core's (128 x 128
// FMAs per CTA at 128 per clock against 128 cycles of MMA for 64-deep blocks),
// and each warp's block is a serial chain: a TMEM load (~200-240 cycles
// before its data can be used), then the FMAs. The next block's load cannot
// be issued before the current block's FMAs without a second 64-register
// buffer, which the register file does not hold beside the accumulators; so
// the chain sets the pace (measured about 600 cycles per 64-deep block, 0.24
// of the tensor rate). 8 warps of 64 columns measured 5-9 % faster than 16
// warps of 32 (kBsEpiWarps = 16 builds with HG_FP8BS_EPI_WARPS=16).
//
// Tiles are 128 x 128 per CTA, or 256 x 128 for a CTA pair (cta_group::2,
// each CTA feeding 64 B columns). Every wait is bounded as in the main kernel.
#pragma once

#include "hgemm_tc.cuh"

namespace hg {

// Warp roles of the block-scaled kernel: epilogue warps first, then the two
// producers and the MMA warp.
#ifndef HG_FP8BS_EPI_WARPS
#define HG_FP8BS_EPI_WARPS 8
#endif
constexpr int kBsEpiWarps = HG_FP8BS_EPI_WARPS;
constexpr int kBsCols = 128 / (kBsEpiWarps / 4);   // columns per epilogue warp
constexpr int kBsProducer = kBsEpiWarps;
constexpr int kBsMma = kBsEpiWarps + 1;
constexpr int kBsProducer2 = kBsEpiWarps + 2;
constexpr int kBsThreads = 32 * (kBsEpiWarps + 3);
constexpr int kBsScaleAhead = kBsEpiWarps == 16 ? 4 : 8;   // scale blocks fetched ahead per warp (even)
constexpr int kBsRingBytes = kBsEpiWarps * kBsScaleAhead * 16;  // 16-byte slots: a_scale, b_scale(s)
static_assert(kBsEpiWarps == 8 || kBsEpiWarps == 16, "epilogue warps");

struct Fp8bsParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n, num_tiles, group_m;
    int32_t num_kb;                 // stages of K: ceil(K / 128)
    int32_t num_sb;                 // scale blocks along K: ceil(K / bs)
    int32_t sa_rows;                // ceil(M / bs): rows of the a_scale grid
    int32_t sb_cols;                // ceil(N / bs): columns of the b_scale grid (its row pitch)
    uint32_t idesc;                 // tcgen05 instruction descriptor (kind::f8f6f4, N = 128)
    const float* a_scale;           // sa_rows x num_sb, row-major
    const float* b_scale;           // num_sb x sb_cols, row-major
    uint16_t* C;                    // bf16 C, ldc elements between rows
    int64_t ldc;
    int32_t c_vec;                  // 1: C 16-byte aligned and N a multiple of 8 (16-byte stores)
    uint64_t timeout_ns;
    unsigned long long* status;
    Schedule sched;                 // whole tiles only
    unsigned long long* trace;      // per-block clock64 records (builds with HG_TRACE only), or null
    int32_t pdl;                    // host: launched as a programmatic dependent of an operand copy
};

// Traced builds: clock64 stamps of the first 64 scale blocks of CTAs 0 and 1
// (record (cta, block), field f).
enum : int { kBsMmaWaited = 0, kBsMmaCommitted = 1, kBsEpiWaited = 2, kBsEpiLoaded = 3, kBsEpiDone = 4,
             kBsEpiLastWaited = 5, kBsProdIssued = 6, kBsMmaFull = 7 };
__device__ __forceinline__ void bs_trace(const Fp8bsParams& p, int blk, int field) {
#ifdef HG_TRACE
    if (p.trace && blockIdx.x < 2 && blk < 64)
        p.trace[(static_cast<int64_t>(blockIdx.x) * 64 + blk) * 8 + field] = static_cast<unsigned long long>(clock64());
#else
    (void)p; (void)blk; (void)field;
#endif
}

template <int CG>
struct Fp8bsCfg {
    static constexpr int BN = 128;
    using Base = TcCfg<CG, BN, 1, 1>;           // the fp8 stage layout of the main kernel
    static constexpr int kParts = 4;            // TMEM partial-sum buffers of BN columns
    static constexpr int kTmemCols = kParts * BN;
    static constexpr int kBarBytes = 256;
    static constexpr int kStagesFit = (kSmemLimit - 1024 - kBarBytes - kBsRingBytes) / Base::kStageBytes;
    static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
    static constexpr int kSmemBytes = 1024 + kStages * Base::kStageBytes + kBarBytes + kBsRingBytes;
    static_assert(kTmemCols <= 512, "tensor memory");
    static_assert((2 * kStages + 2 * kParts + 1) * 8 + 8 <= kBarBytes, "barrier area");
    static_assert(kSmemBytes <= kSmemLimit, "shared memory");
};

template <int CG, int kGs, int kDt>
__global__ void __launch_bounds__(kBsThreads, 1)
hgemm_fp8bs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB2, const Fp8bsParams p) {
#if defined(__CUDA_ARCH__) && defined(__CUDA_ARCH_FEAT_SM103_ALL)
    using Cfg = Fp8bsCfg<CG>;
    using Base = typename Cfg::Base;
    constexpr int S = Cfg::kStages;
    constexpr int R = Cfg::kParts;
    constexpr int BN = Cfg::BN;
    constexpr int kSbPerStage = Base::kBK / kGs;   // scale blocks in a 128-deep stage
    constexpr int kMmaPerSb = kGs / Base::kUK;     // K = 32 MMAs per scale block
    constexpr int kGroups = R / 2;                  // hand-offs in flight: pairs of buffers
    static_assert(kGs == 32 || kGs == 64, "scale block");
    static_assert(kDt == 3 || kDt == 4, "fp8 operands");
    static_assert(Base::kBAtoms == 1, "one B atom per stage");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = sA + S * Base::kABytes;
    const uint32_t sBar = sB + S * Base::kBBytes;
    const uint32_t bar_full = sBar;                  // [S]
    const uint32_t bar_empty = sBar + 8 * S;         // [S]
    const uint32_t bar_pfull = sBar + 16 * S;        // [R] partial buffer written
    const uint32_t bar_pempty = bar_pfull + 8 * R;   // [R] partial buffer read
    const uint32_t bar_drain = bar_pempty + 8 * R;
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + (bar_drain + 8 - base));
    const uint32_t sRing = sBar + Cfg::kBarBytes;    // epilogue warps' scale rings
    volatile uint32_t* const abort_flag = tmem_slot + 1;

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t rank = (CG > 1) ? cluster_ctarank() : 0u;   // rank in the CTA pair
    const int cluster_id = static_cast<int>(blockIdx.x) / CG;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < kGroups; ++b) {
            mbar_init(bar_pfull + 8 * b, 1);
            mbar_init(bar_pempty + 8 * b, kBsEpiWarps * CG);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init_cluster();
    }
    if (warp == kBsProducer && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (Base::kBPartial) tma_prefetch_desc(&tmB2);
    }
    if (warp == kBsMma) tmem_alloc<CG>(smem_addr(tmem_slot), Cfg::kTmemCols);
    tc_fence_before();
    __syncthreads();
    if constexpr (CG > 1) cluster_sync();
    tc_fence_after();
    grid_dependency_wait();   // after an operand copy launched just before this kernel
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    const Waiter w{abort_flag, p.timeout_ns, p.status};

    if (warp == kBsProducer || warp == kBsProducer2) {
        // ------------------------------------------------------------ producer
        const uint32_t pid = warp == kBsProducer ? 0u : 1u;
        uint32_t stage = pid, phase = 0, g = 0;
        bool ok = true;
        WorkUnit wu;
        for (int lu = 0; ok && next_unit(p.sched, cluster_id, lu, wu); ++lu) {
            int32_t tm, tn;
            tile_coord(wu.tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            const int32_t m0 = tm * kBlockMCta * CG + static_cast<int32_t>(rank) * kBlockMCta;
            const int32_t n0 = tn * BN + static_cast<int32_t>(rank) * Base::kBnCta;
            for (int kb = 0; kb < p.num_kb; ++kb, ++g) {
                if ((g & 1u) != pid) continue;
                if (!wait_bar_warp(bar_empty + 8 * stage, phase ^ 1u, w, kRoleProducer, stage)) {
                    ok = false;
                    break;
                }
                const uint32_t a_dst = sA + stage * Base::kABytes;
                const uint32_t b_dst = sB + stage * Base::kBBytes;
                const uint32_t fb = bar_full + 8 * stage;
                const int32_t k0 = kb * Base::kBK;
                const CUtensorMap* bmap = Base::kBPartial ? &tmB2 : &tmB;
                if (elect_one_sync()) {
                    if constexpr (CG == 1) {
                        mbar_arrive_expect_tx(fb, Base::kTxBytes);
                        tma_load_2d(a_dst, &tmA, fb, k0, m0);
                        tma_load_2d(b_dst, bmap, fb, n0, k0);
                    } else {
                        const uint32_t fb_leader = mapa_shared(fb, 0);
                        if (rank == 0) mbar_arrive_expect_tx(fb, Base::kTxBytes);
                        tma_load_2d_pair(a_dst, &tmA, fb_leader, k0, m0);
                        tma_load_2d_pair(b_dst, bmap, fb_leader, n0, k0);
                    }
                }
                __syncwarp();
                stage += 2;
                if (stage >= static_cast<uint32_t>(S)) {
                    stage -= S;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            // loads already issued still land in this CTA's shared memory
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 50000ull) {}
        }
    } else if (warp == kBsMma) {
        // ----------------------------------------------------------------- MMA
        if (rank == 0) {
            uint32_t stage = 0, phase = 0, pb = 0, pph = 0;
            int nblk = 0;
            bool ok = true, issued = false;
            const uint64_t a_desc0 = sdesc_sw128(sA, 16u, 1024u);
            const uint64_t b_desc0 = sdesc_sw128(sB, Base::kBAtomBytes, 1024u);
            WorkUnit wu;
            for (int it = 0; ok && next_unit(p.sched, cluster_id, it, wu); ++it) {
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar_warp(bar_full + 8 * stage, phase, w, kRoleMma, stage)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) bs_trace(p, nblk, kBsMmaFull);
                    tc_fence_after();
                    const uint64_t ad = a_desc0 + ((stage * Base::kABytes) >> 4);
                    const uint64_t bd = b_desc0 + ((stage * Base::kBBytes) >> 4);
                    const int rem = p.num_sb - kb * kSbPerStage;
                    const int nsb = rem < kSbPerStage ? rem : kSbPerStage;
                    // Groups of two scale blocks (a stage holds 2 or 4; the
                    // last group of a K loop with an odd block count has one):
                    // one wait for the group's two buffers, one commit.
                    for (int j0 = 0; j0 < nsb; j0 += 2) {
                        if (!wait_bar_warp(bar_pempty + 8 * pb, pph ^ 1u, w, kRoleMma, 32 + pb)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) bs_trace(p, nblk, kBsMmaWaited);
                        tc_fence_after();
                        const int nj = nsb - j0 < 2 ? nsb - j0 : 2;
                        if (elect_one_sync()) {
                            for (int jj = 0; jj < nj; ++jj) {
                                const uint32_t d_tmem = tmem_base + (2u * pb + static_cast<uint32_t>(jj)) * BN;
#pragma unroll
                                for (int mm = 0; mm < kMmaPerSb; ++mm) {
                                    const uint32_t kk = static_cast<uint32_t>((j0 + jj) * kMmaPerSb + mm);
                                    umma_f8<CG>(d_tmem, ad + 2u * kk, bd + 8u * Base::kUK * kk, p.idesc,
                                                mm > 0 ? 1u : 0u);
                                }
                            }
                            if constexpr (CG == 1) umma_commit(bar_pfull + 8 * pb);
                            else umma_commit_pair(bar_pfull + 8 * pb, static_cast<uint16_t>(0x3u));
                        }
                        __syncwarp();
                        if (lane == 0) bs_trace(p, nblk, kBsMmaCommitted);
                        ++nblk;
                        issued = true;
                        if (++pb == static_cast<uint32_t>(kGroups)) {
                            pb = 0;
                            pph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    if (elect_one_sync()) {
                        if constexpr (CG == 1) umma_commit(bar_empty + 8 * stage);
                        else umma_commit_pair(bar_empty + 8 * stage, static_cast<uint16_t>(0x3u));
                    }
                    __syncwarp();
                    if (++stage == static_cast<uint32_t>(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && issued) {
                // TMEM may only be freed once every issued MMA has completed.
                if (elect_one_sync()) {
                    if constexpr (CG == 1) umma_commit(bar_drain);
                    else umma_commit_pair(bar_drain, static_cast<uint16_t>(0x1u));
                }
                __syncwarp();
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar_drain, 0) && globaltimer_ns() - t0 < p.timeout_ns) {}
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        constexpr int kLoads = kBsCols / 32;    // 32-column TMEM loads per block
        const int quarter = warp & 3;
        const int colgrp = warp >> 2;
        uint32_t pb = 0, pph = 0;
        int nblk = 0;
        bool ok = true;
        WorkUnit wu;
        for (int it = 0; ok && next_unit(p.sched, cluster_id, it, wu); ++it) {
            int32_t tm, tn;
            tile_coord(wu.tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            const int32_t row_base = tm * kBlockMCta * CG + static_cast<int32_t>(rank) * kBlockMCta + quarter * 32;
            const int32_t col_base = tn * BN + kBsCols * colgrp;
            // Scale rows and columns of this warp (warp-uniform; clamped for
            // rows and columns past the matrix, whose partial sums are zero).
            int32_t rb = row_base / kGs;
            if (rb > p.sa_rows - 1) rb = p.sa_rows - 1;
            int32_t cb[kLoads];
#pragma unroll
            for (int l = 0; l < kLoads; ++l) {
                cb[l] = (col_base + 32 * l) / kGs;
                if (cb[l] > p.sb_cols - 1) cb[l] = p.sb_cols - 1;
            }
            const float* sa_row = p.a_scale + static_cast<int64_t>(rb) * p.num_sb;
            float acc[kBsCols];
#pragma unroll
            for (int i = 0; i < kBsCols; ++i) acc[i] = 0.0f;
            // Block blk's factors go to slot blk % kBsScaleAhead of this warp's
            // ring: lane 0 copies a_scale, lanes 1..kLoads the b_scale of each
            // 32-column load. One commit group per block, in every lane.
            const uint32_t ring = sRing + static_cast<uint32_t>(warp * kBsScaleAhead * 16);
            const int32_t my_cb = kLoads == 1 ? cb[0] : (lane == 1 ? cb[0] : cb[kLoads - 1]);
            auto fetch = [&](int blk) {
                if (blk < p.num_sb) {
                    const uint32_t slot = ring + static_cast<uint32_t>((blk % kBsScaleAhead) * 16);
                    if (lane == 0) cp_async_4(slot, sa_row + blk);
                    else if (lane <= static_cast<uint32_t>(kLoads))
                        cp_async_4(slot + 4u * lane, p.b_scale + static_cast<int64_t>(blk) * p.sb_cols + my_cb);
                }
                cp_async_commit();
            };
#pragma unroll
            for (int j = 0; j < kBsScaleAhead; ++j) fetch(j);
            const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
            const uint32_t t_cols = static_cast<uint32_t>(kBsCols * colgrp) + t_lane;
            // acc += factor * partial for one block held in r (kLoads 32-column loads)
            auto accumulate = [&](const uint32_t (&r)[kBsCols], float sa_f, const float (&sb_f)[kLoads]) {
#pragma unroll
                for (int l = 0; l < kLoads; ++l) {
                    const float sf = sa_f * sb_f[l];
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[32 * l + i] = fmaf(sf, __uint_as_float(r[32 * l + i]), acc[32 * l + i]);
                }
            };
            auto load_block = [&](uint32_t buf, uint32_t (&r)[kBsCols]) {
#pragma unroll
                for (int l = 0; l < kLoads; ++l)
                    tmem_ld_32x32b_x32(tmem_base + buf * BN + t_cols + 32u * l, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * l));
                tmem_ld_wait();
#pragma unroll
                for (int l = 0; l < kLoads; ++l) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(r + 32 * l));
            };
            // Blocks come in pairs (2g, 2g + 1) that share one hand-off; a K
            // loop with an odd block count ends in a pair of one.
            const int ngroups = (p.num_sb + 1) / 2;
            for (int g = 0; g < ngroups; ++g) {
                const int b0 = 2 * g;
                const bool two = b0 + 1 < p.num_sb;
                // both blocks' factor copies have landed once at most
                // kBsScaleAhead - 2 commit groups are pending
                cp_async_wait<kBsScaleAhead - 2>();
                __syncwarp();
                const uint32_t slot0 = ring + static_cast<uint32_t>((b0 % kBsScaleAhead) * 16);
                const uint32_t slot1 = ring + static_cast<uint32_t>(((b0 + 1) % kBsScaleAhead) * 16);
                const float sa0 = ld_shared_f32(slot0), sa1 = ld_shared_f32(slot1);
                float sb0[kLoads], sb1[kLoads];
#pragma unroll
                for (int l = 0; l < kLoads; ++l) {
                    sb0[l] = ld_shared_f32(slot0 + 4u * (l + 1));
                    sb1[l] = ld_shared_f32(slot1 + 4u * (l + 1));
                }
                __syncwarp();
                fetch(b0 + kBsScaleAhead);       // the two slots just read
                fetch(b0 + 1 + kBsScaleAhead);
                if (!wait_bar_warp(bar_pfull + 8 * pb, pph, w, kRoleEpilogue, 32 + pb)) {
                    ok = false;
                    break;
                }
                if (lane == 0 && warp == 0) bs_trace(p, nblk, kBsEpiWaited);
                if (lane == 0 && warp == kBsEpiWarps - 1) bs_trace(p, nblk, kBsEpiLastWaited);
                tc_fence_after();
                uint32_t r[kBsCols];
                load_block(2u * pb, r);
                if (lane == 0 && warp == 0) bs_trace(p, nblk, kBsEpiLoaded);
                accumulate(r, sa0, sb0);
                if (two) load_block(2u * pb + 1u, r);
                // the pair's reads are done: hand its two buffers back to the MMA warp
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_accumulator<CG>(bar_pempty + 8 * pb, 0);
                if (++pb == static_cast<uint32_t>(kGroups)) {
                    pb = 0;
                    pph ^= 1u;
                }
                if (two) accumulate(r, sa1, sb1);
                if (lane == 0 && warp == 0) {
                    asm volatile("" :: "f"(acc[0]), "f"(acc[kBsCols - 1]));
                    bs_trace(p, nblk, kBsEpiDone);
                }
                ++nblk;
            }
            cp_async_wait<0>();
            if (!ok) break;
            // Round to bf16 and store this thread's row: kBsCols columns from col_base.
            const int32_t row = row_base + static_cast<int32_t>(lane);
            if (row < p.M) {
                uint32_t pk[kBsCols / 2];
#pragma unroll
                for (int i = 0; i < kBsCols / 2; ++i)
                    pk[i] = pack_rn<kDt>(__float_as_uint(acc[2 * i]), __float_as_uint(acc[2 * i + 1]));
                uint16_t* crow = p.C + static_cast<int64_t>(row) * p.ldc;
                if (p.c_vec) {
#pragma unroll
                    for (int j = 0; j < kBsCols / 8; ++j) {
                        const int32_t col = col_base + 8 * j;
                        if (col < p.N)
                            *reinterpret_cast<uint4*>(crow + col) =
                                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < kBsCols; ++i) {
                        const int32_t col = col_base + i;
                        if (col < p.N)
                            crow[col] = static_cast<uint16_t>((i & 1) ? (pk[i >> 1] >> 16) : (pk[i >> 1] & 0xFFFFu));
                    }
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    __syncthreads();
    if constexpr (CG > 1) cluster_sync();
    if (warp == kBsMma) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, Cfg::kTmemCols);
    }
#endif
}

}  // namespace hg
