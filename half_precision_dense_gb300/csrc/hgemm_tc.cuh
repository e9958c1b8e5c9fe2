// hgemm_tc.cuh - the persistent, warp-specialised tcgen05 GEMM kernel for
// sm_103a: C = A.B, A (M x K) and B (K x N) row-major, fp32 accumulation in
// tensor memory. fp16/bf16 operands give C in the input dtype; the tf32 and
// fp8 kinds (fp32 C; scaled bf16 C) and the implicit-GEMM convolution (A read
// by TMA im2col copies) are instances of the same template.
//
// Prior art: "[CUDA 优化实战] hgemm - 超越 cuBLAS" builds the same product on an
// RTX 5060 mobile from cp.async + ldmatrix + mma.sync m16n8k16 (section 1),
// XOR-swizzled shared memory (section 2), a double-buffered cp.async pipeline
// (section 3) and a shared-memory-staged, coalesced C write-back (section 4).
// Each idea has a Blackwell-native counterpart here:
//
//   page (sm_80-class instructions)          this kernel (sm_103a)
//   cp.async 16 B per thread + commit/wait   TMA box loads, mbarrier transaction counts
//   SWIZZLE_A / SWIZZLE_B (16 B chunk XOR)   the TMA/UMMA 128-byte swizzle (chunk ^= row % 8)
//   double buffer                            an S-stage full/empty mbarrier ring
//   mma.sync m16n8k16, fp32 in registers     tcgen05.mma kind::f16, fp32 in tensor memory
//   grid swizzle (SWIZZLE_W)                 persistent CTAs walking a grouped raster
//   Cs staging + SWIZZLE_C + float4 stores   tcgen05.ld -> cvt.rn -> swizzled smem -> row stores
//
// Roles (352 threads with 8 epilogue warps, 608 with 16; one CTA per SM):
//   warps 0-7  epilogue: warp w reads TMEM lanes 32(w % 4)..+31 (C rows of the
//              tile) and every other 64-column chunk, starting at chunk w / 4
//              (16 epilogue warps, for a 16-bit C on 224- and 256-wide tiles,
//              take every fourth 32-column chunk; the other roles' warp
//              numbers then move up by 8)
//   warps 8,10 producers: each warp takes alternate stages (even / odd K
//              blocks); one elected lane issues the TMA loads of A and B
//   warp 9     MMA: allocates TMEM; in the leader CTA the warp runs the loop and
//              one elected lane issues tcgen05.mma and the commits
//
// CTA pairs (CG = 2, a cluster of two): the pair owns a 256-row tile. Each CTA
// loads its own 128 rows of A and its own half of the tile's B columns; the
// leader's elected lane issues tcgen05.mma.cta_group::2, which reads both
// CTAs' shared memory and accumulates each CTA's 128 rows in that CTA's TMEM.
//
// Larger clusters (MC > 1): 2, 4 or 8 single CTAs that split one tile's K
// loop and add their partial sums through distributed shared memory (the
// template's comment gives the details).
//
// Every wait is bounded (TcParams::timeout_ns). A wait that runs out records
// HGEMM_ERR_TIMEOUT with the role and barrier in the device status word, sets a
// CTA-wide abort flag that ends the other roles' loops, lets in-flight copies
// and MMAs finish, frees TMEM and returns; it never traps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"
#include "schedule.h"

namespace hg {

constexpr int kBlockMCta = 128;   // C rows per CTA = TMEM lanes
constexpr int kBlockK = 64;       // K per stage for 16-bit inputs: one 128 B swizzle row
constexpr int kUmmaK = 16;        // K of one kind::f16 MMA
// Input kinds: 0 = fp16, 1 = bf16 (kind::f16, C in the input type), 2 = tf32
// (kind::tf32 on fp32 operands, C in fp32), 3 = E4M3, 4 = E5M2 (kind::f8f6f4
// on 8-bit operands, C in bf16 after the per-channel scales). A stage row is
// always 128 B of K.
__host__ __device__ constexpr int elem_bytes(int dt) { return dt == 2 ? 4 : dt >= 3 ? 1 : 2; }
__host__ __device__ constexpr int block_k(int dt) { return 128 / elem_bytes(dt); }
constexpr int kEpiWarps = 8;      // default: two per TMEM lane quarter, splitting the columns
constexpr int kEpiQuarters = 4;   // TMEM lane quarters (32 rows each)
constexpr int kThreads = 32 * (kEpiWarps + 3);  // + two producers and the MMA warp
constexpr int kEpiBoxRows = 32;   // one epilogue warp's rows
constexpr int kEpiBoxCols = 64;   // 128 B of half-precision values
constexpr int kEpiBoxBytes = kEpiBoxRows * kEpiBoxCols * 2;
constexpr int kSmemLimit = 232448;  // 227 KiB: the opt-in maximum per block

constexpr uint32_t kStatusTimeout = 5;  // == HGEMM_ERR_TIMEOUT
enum : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3 };

struct TcParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n, num_tiles, group_m;
    int32_t num_kb;                 // ceil(K / K per stage): 64 16-bit, 128 8-bit or 32 fp32 values
    uint32_t idesc;                 // tcgen05 instruction descriptor
    int32_t store_mode;             // 1: TMA stores of C; 2: plain element stores through `C`;
                                    // 3: direct 16-byte stores through `C` (aligned C only);
                                    // 4: smem-staged, coalesced 16-byte stores (aligned C only);
                                    // 5: smem-staged 16-byte stores realigned to each row's
                                    //    start, element stores at the ragged ends (16-bit C,
                                    //    any pitch)
    uint16_t* C;                    // used by store modes 2-4 (fp32 elements for tf32)
    const float* a_scale;           // fp8: one factor per row of A, or null (1)
    const float* b_scale;           // fp8: one factor per column of B, or null (1)
    // Implicit-GEMM convolution (im2col != 0): A is not a matrix but the
    // channels-last activations behind an im2col-mode tensor map; row m of A
    // is output pixel (n, p, q) = (m / (P Q), m / Q % P, m % Q), and K block
    // kb is filter tap kb / cv_cblocks (r = tap / cv_S, s = tap % cv_S) at
    // channels (kb % cv_cblocks) * kBK ..
    int32_t im2col;
    int32_t cv_cblocks, cv_S, cv_P, cv_Q, cv_stride, cv_pad;
    int64_t ldc;                    // elements between C rows (store_mode 2)
    uint64_t timeout_ns;
    unsigned long long* status;     // device status word
    Schedule sched;                 // data-parallel tiles, then stream-K ranges (schedule.h)
    float* partials;                // per cluster: the fp32 partial sums of its first,
                                    // non-owning stream-K unit
    unsigned long long* flags;      // one per (partial block, column half): == epoch once written
    unsigned long long epoch;       // unique per launch (a captured launch clears the flags first)
    int32_t inject;                 // test hook: 1 = stream-K owners wait for partial sums
                                    // that are never published; 2 = a K-split cluster's rank 0
                                    // withholds its ring-free arrival (the waits run out)
    unsigned long long* trace;      // timeline records (builds with HG_TRACE only), or null
    int32_t pdl;                    // host: launched as a programmatic dependent of the kernel
                                    // before it on the stream (an operand copy)
};

// Timeline records of a traced build: per CTA, per unit it takes (up to
// kTraceUnits), kTraceFields %globaltimer stamps.
constexpr int kTraceUnits = 32;
constexpr int kTraceFields = 8;
enum : int { kTrProdFirst = 0, kTrMmaFirst = 1, kTrMmaLast = 2, kTrEpiStart = 3, kTrEpiTmemFree = 4,
             kTrEpiEnd = 5, kTrUnit = 6, kTrSetup = 7 };
// Epilogue detail of a CTA's first unit (warp 0): slot 16 + c, field f, in
// SM clock cycles (clock64; %globaltimer is too coarse for a chunk's steps).
enum : int { kTcLdDone = 0, kTcWaitRead = 1, kTcStaged = 2, kTcIssued = 3, kTcStart = 4, kTcPacked = 5,
             kTcStored = 6 };
__device__ __forceinline__ void trace_chunk(const TcParams& p, int it, int c, int field) {
#ifdef HG_TRACE
    if (p.trace && it == 0 && (c < 10 || c == 12))
        p.trace[(static_cast<int64_t>(blockIdx.x) * kTraceUnits + 16 + c) * kTraceFields + field] =
            static_cast<unsigned long long>(clock64());
#else
    (void)p; (void)it; (void)c; (void)field;
#endif
}

__device__ __forceinline__ void trace_stamp(const TcParams& p, int local_unit, int field) {
#ifdef HG_TRACE
    if (p.trace && local_unit < kTraceUnits)
        p.trace[(static_cast<int64_t>(blockIdx.x) * kTraceUnits + local_unit) * kTraceFields + field] =
            globaltimer_ns();
#else
    (void)p; (void)local_unit; (void)field;
#endif
}

// Wait-time counters of a traced build: per CTA, clock64 cycles the producers
// and the MMA thread spent in barrier waits (unit slot kTraceUnits - 1).
enum : int { kTwProdEmpty0 = 0, kTwProdEmpty1 = 1, kTwMmaFull = 2, kTwMmaTempty = 3, kTwMmaStages = 4,
             kTwMmaSpan = 5 };
__device__ __forceinline__ void trace_wait_total(const TcParams& p, int field, long long cycles) {
#ifdef HG_TRACE
    if (p.trace)
        p.trace[(static_cast<int64_t>(blockIdx.x) * kTraceUnits + kTraceUnits - 1) * kTraceFields + field] =
            static_cast<unsigned long long>(cycles);
#else
    (void)p; (void)field; (void)cycles;
#endif
}
// Stream-K fix-up stamps of a traced build: unit slot 30 = the owner unit
// (0: partners' marks seen, 1: chunk loop done, 2: last store drained, 3+j:
// warp 0's j-th chunk done), slot 29 = the first partner unit (0: epilogue
// start, 1: partial sums published).
// Launch-level stamps of a traced build (%globaltimer): kernel entry, all
// roles done, teardown barrier passed, tensor memory freed.
constexpr int kTrLaunchSlot = 26;
__device__ __forceinline__ void trace_slot(const TcParams& p, int slot, int field) {
#ifdef HG_TRACE
    if (p.trace)
        p.trace[(static_cast<int64_t>(blockIdx.x) * kTraceUnits + slot) * kTraceFields + field] = globaltimer_ns();
#else
    (void)p; (void)slot; (void)field;
#endif
}
#ifdef HG_TRACE
#define HG_TW_BEGIN() const long long hg_tw0 = clock64()
#define HG_TW_END(acc) (acc) += clock64() - hg_tw0
#else
#define HG_TW_BEGIN() do {} while (0)
#define HG_TW_END(acc) do {} while (0)
#endif

// Index of the partial block published by cluster `cluster` (its one
// non-owning stream-K unit) for the CTA of cluster rank `crank` and TMEM lane
// quarter `quarter`: 32 rows x BN fp32. Its two epilogue warps (column halves)
// each mark their own chunks with flag 2 * block + half.
template <int kCluster>
__device__ __forceinline__ int64_t partial_block(int32_t cluster, uint32_t crank, int quarter) {
    return (static_cast<int64_t>(cluster) * kCluster + crank) * kEpiQuarters + quarter;
}

constexpr int pow2_at_least(int x) {
    int p = 32;
    while (p < x) p *= 2;
    return p;
}

// kSplitK > 1: the K split within a cluster, whose epilogue adds the partial
// sums in the stage ring and stores C from registers, so it needs no staging
// boxes and the ring takes their space.
template <int CG, int BN, int kElem = 2, int kSplitK = 1>
struct TcCfg {
    static constexpr int kBK = 128 / kElem;                // K per stage: one 128 B row of A
    static constexpr int kUK = 32 / kElem;                 // K of one MMA (32 bytes of K)
    static constexpr int kAtomCols = 128 / kElem;          // columns of one B swizzle atom
    static constexpr int kBnCta = BN / CG;                 // B columns each CTA feeds the MMA
    static constexpr int kABytes = kBlockMCta * 128;
    static constexpr int kBAtoms = (kBnCta + kAtomCols - 1) / kAtomCols;  // B swizzle atoms loaded
    static constexpr int kBAtomBytes = kBK * 128;          // kAtomCols columns x kBK k-rows
    // B is read MN-major in swizzle atoms of kAtomCols columns (128 B rows)
    // by kBK k-rows, straight from the row-major matrix, for every dtype.
    static constexpr int kBBytes = kBAtoms * kBAtomBytes;
    static constexpr int kChunks = (BN + 63) / 64;         // epilogue chunks of 64 columns
    static constexpr bool kHalfLast = (BN % 64) != 0;      // the last chunk is 32 columns
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kEpiBytes = kSplitK > 1 ? 0 : kEpiWarps * kEpiBoxBytes;  // one staging box per warp
    static constexpr int kBarBytes = kSplitK > 1 ? 512 : 256;  // a K split adds its three barriers
    static constexpr int kStagesFit = (kSmemLimit - 1024 - kEpiBytes - kBarBytes) / kStageBytes;
    static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + kBarBytes;
    static constexpr int kTmemCols = pow2_at_least(2 * BN);  // two accumulators of BN fp32 columns
    // Columns of the last B atom a CTA uses (112 of a 224-wide pair tile's
    // columns leave it part-full); it is loaded with a box of that width, so a
    // stage brings only the bytes the MMA reads.
    static constexpr int kBLastCols = kBnCta - (kBAtoms - 1) * kAtomCols;
    static constexpr bool kBPartial = kBLastCols != kAtomCols;
    static constexpr int kBLoadBytes = (kBAtoms - 1) * kBAtomBytes + kBK * kBLastCols * kElem;
    static constexpr uint32_t kTxBytes = CG * (kABytes + kBLoadBytes); // bytes landing per stage on the leader's barrier
    static_assert(CG == 1 || CG == 2, "cta group");
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "tile width");
    static_assert(kBnCta % 16 == 0, "MMA N per CTA");
    static_assert(kTmemCols <= 512, "tensor memory");
    static_assert(kStages >= 2, "pipeline depth");
    static_assert(kSmemBytes <= kSmemLimit, "shared memory");
    // full[S], empty[S], tmem_full[2], tmem_empty[2], drain, pre[2], the TMEM
    // slot and abort flag, one partial-sum barrier per epilogue warp
    static_assert((2 * kStages + 7) * 8 + 8 + 8 * kEpiWarps <= kBarBytes, "barrier area");
    // A stream-K owner's epilogue lands its partners' partial sums in the
    // (then idle) stage ring: per epilogue warp and partner one 8 KiB chunk.
    static constexpr int kBulkPartners = kStages * kStageBytes / (kEpiWarps * 8192);
};

// Shared-memory matrix descriptor (tcgen05), 128-byte swizzle.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-48  fixed 0b001
//   bits 49-51  base offset (0: every tile starts on a 1024 B boundary)
//   bits 61-63  layout: 2 = 128-byte swizzle
// K-major A (rows of 128 B holding 64 K values, 8-row swizzle atoms stacked
// along M): SBO = 1024 B between 8-row groups; LBO unused. The K offset of the
// j-th 16-wide MMA inside the 64-wide stage is +32 j bytes of start address.
// MN-major B (each atom is kAtomCols columns = 128 B wide and kBK k-rows
// deep: 64 x 64 for 16-bit, 128 x 128 for 8-bit): LBO = distance between
// atoms, SBO = 1024 B between 8-row k groups; the j-th MMA starts kUK j rows
// = 128 kUK j bytes further (2048 j for 16-bit, 4096 j for 8-bit).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
           (1ull << 46) | (2ull << 61);
}

// MN-major tf32 B: descriptor layout 1 (128-byte swizzle, 32-byte atomicity),
// LBO = distance between 32-column atoms, SBO = 512 B between 4-row cores.
__device__ __forceinline__ uint64_t sdesc_mn_tf32(uint32_t saddr, uint32_t lbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((512u >> 4) & 0x3FFFu) << 32) |
           (1ull << 46) | (1ull << 61);
}

template <int kDt>
__device__ __forceinline__ uint32_t pack_rn(uint32_t lo, uint32_t hi) {
    if constexpr (kDt == 1 || kDt >= 3) {
        __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(__uint_as_float(lo), __uint_as_float(hi));
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

struct Waiter {
    volatile uint32_t* abort;
    uint64_t timeout_ns;
    unsigned long long* status;
};

static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Waiter& w,
                                       uint32_t role, uint32_t which) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*w.abort) return false;
        if (globaltimer_ns() - t0 > w.timeout_ns) {
            const unsigned long long info =
                (static_cast<unsigned long long>(role) << 56) |
                (static_cast<unsigned long long>(which & 0xFFu) << 48) |
                (static_cast<unsigned long long>(blockIdx.x & 0xFFFFu) << 32);
            atomicCAS(w.status, 0ull, info | kStatusTimeout);
            *w.abort = 1;
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Waiter& w,
                                         uint32_t role, uint32_t which) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, w, role, which);
}

// wait_bar for a barrier that peer CTAs arrive on with release semantics at
// cluster scope: the wait acquires at cluster scope, so what they wrote into
// this CTA's shared memory before arriving is visible after it. Whole warp,
// lane 0's outcome.
static __device__ __noinline__ bool wait_bar_cluster_warp(uint32_t bar, uint32_t parity, const Waiter& w,
                                                          uint32_t role, uint32_t which) {
    bool got = mbar_try_wait_cluster(bar, parity);
    const uint64_t t0 = globaltimer_ns();
    while (!got) {
        for (int i = 0; i < 64 && !got; ++i) got = mbar_try_wait_cluster(bar, parity);
        if (got || *w.abort) break;
        if (globaltimer_ns() - t0 > w.timeout_ns) {
            const unsigned long long info =
                (static_cast<unsigned long long>(role) << 56) |
                (static_cast<unsigned long long>(which & 0xFFu) << 48) |
                (static_cast<unsigned long long>(blockIdx.x & 0xFFFFu) << 32);
            atomicCAS(w.status, 0ull, info | kStatusTimeout);
            *w.abort = 1;
            break;
        }
    }
    return __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
}

// wait_bar for a whole warp: every lane waits, and lane 0's outcome is the
// warp's (lanes could otherwise disagree when a wait runs out just as the
// phase completes), so the warp's control flow stays uniform.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Waiter& w,
                                              uint32_t role, uint32_t which) {
    const int got = wait_bar(bar, parity, w, role, which) ? 1 : 0;
    return __shfl_sync(0xffffffffu, got, 0) != 0;
}

// An epilogue warp hands its accumulator buffer back to the MMA warp. The
// arrive is relaxed: the warp's tcgen05.ld reads have completed
// (tcgen05.wait::ld) before it, which is all the MMA warp needs, whereas a
// release arrive at cluster scope also waits until the warp's earlier global
// stores of C are acknowledged (measured 0.6 us of a tile's epilogue).
template <int CG>
__device__ __forceinline__ void release_accumulator(uint32_t bar, uint32_t leader) {
    if constexpr (CG == 1) {
        asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
    } else {
        asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];"
                     :: "r"(mapa_shared(bar, leader)) : "memory");
    }
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* ptr) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ptr) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned long long* ptr, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(ptr), "l"(v) : "memory");
}

// Bounded wait until another CTA has published `epoch` at `flag`.
static __device__ __noinline__ bool wait_flag(const unsigned long long* flag, unsigned long long epoch,
                                              const Waiter& w, uint32_t which) {
    if (ld_acquire_gpu(flag) == epoch) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 16; ++i) {
            if (ld_acquire_gpu(flag) == epoch) return true;
            __nanosleep(32);
        }
        if (*w.abort) return false;
        if (globaltimer_ns() - t0 > w.timeout_ns) {
            const unsigned long long info =
                (static_cast<unsigned long long>(kRoleEpilogue) << 56) |
                (static_cast<unsigned long long>(which & 0xFFu) << 48) |
                (static_cast<unsigned long long>(blockIdx.x & 0xFFFFu) << 32);
            atomicCAS(w.status, 0ull, info | kStatusTimeout);
            *w.abort = 1;
            return false;
        }
    }
}

// Pins the 32 registers after tcgen05.wait::ld so no use is scheduled above it.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
#pragma unroll
    for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}

// Store mode 5, one warp's 32 rows x 64 (or 32, `half`) columns of 16-bit C
// from its swizzled staging box, for a C whose rows do not start on 16-byte
// boundaries (a row pitch that is not a multiple of 8 elements). A row's
// 16 * nseg bytes start at offset o (even) in a 16-byte segment: lane g of the
// row's nseg lanes writes the aligned segment g (g >= 1 when o > 0), assembled
// from box chunks g - 1 and g and shifted into place, and one of the row's
// eight edge elements (the head [0, 8 - o/2) and the tail, which share a
// segment with the neighbouring chunk of the row), so every lane does the
// same work and nothing outside these columns is written. Kept out of line:
// only an unaligned C calls it, and inlined it would take registers from the
// main loop of every instantiation.
// Element i (0..7) of eight 16-bit values packed in a 16-byte vector.
__device__ __forceinline__ uint16_t u16_of(const uint4& v, int32_t i) {
    const uint32_t w = (i >> 1) == 0 ? v.x : (i >> 1) == 1 ? v.y : (i >> 1) == 2 ? v.z : v.w;
    return static_cast<uint16_t>((i & 1) ? (w >> 16) : (w & 0xFFFFu));
}

static __device__ __noinline__ void store_chunk_realigned(const uint8_t* box_ptr, uint16_t* C, int64_t ldc,
                                                          int32_t M, int32_t N, int32_t row0, int32_t ccol,
                                                          bool half, uint32_t lane) {
    const uint32_t nseg = half ? 4u : 8u;       // 16-byte chunks per box row
    const int32_t nel = 8 * static_cast<int32_t>(nseg);
    const int32_t nvalid = N - ccol;            // columns of the chunk inside C
    if (nvalid <= 0) return;
#pragma unroll 2
    for (uint32_t piece = lane; piece < 32u * nseg; piece += 32u) {
        const uint32_t rr = piece / nseg, g = piece % nseg;
        const int32_t row = row0 + static_cast<int32_t>(rr);
        if (row >= M) continue;
        uint16_t* const crow = C + static_cast<int64_t>(row) * ldc + ccol;
        const uint32_t o = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(crow) & 15u);   // even
        const uint32_t sw = half ? ((rr >> 1) & 3u) : (rr & 7u);
        const uint8_t* const brow = box_ptr + rr * (half ? 64u : 128u);
        const uint4 cg = *reinterpret_cast<const uint4*>(brow + ((g ^ sw) << 4));
        if (o == 0) {
            const int32_t e0 = 8 * static_cast<int32_t>(g);
            if (e0 + 8 <= nvalid) {
                *reinterpret_cast<uint4*>(crow + e0) = cg;
            } else {
                for (int32_t e = e0; e < nvalid && e < e0 + 8; ++e) crow[e] = u16_of(cg, e - e0);
            }
            continue;
        }
        const int32_t half_o = static_cast<int32_t>(o >> 1);
        if (g > 0) {
            // the aligned segment holding elements [8g - o/2, 8g - o/2 + 8)
            const int32_t e0 = 8 * static_cast<int32_t>(g) - half_o;
            const uint4 cp = *reinterpret_cast<const uint4*>(brow + (((g - 1u) ^ sw) << 4));
            const uint4 v = bytes_from(cp, cg, 16u - o);
            if (e0 + 8 <= nvalid) {
                *reinterpret_cast<uint4*>(crow + e0) = v;
            } else {
                for (int32_t e = e0; e < nvalid && e < e0 + 8; ++e) crow[e] = u16_of(v, e - e0);
            }
        }
        // edge element k = g (and k = g + 4 for a 32-column chunk, whose row
        // has four lanes): head elements [0, 8 - o/2), then the tail
        for (uint32_t k = g; k < 8u; k += nseg) {
            const int32_t e = static_cast<int32_t>(k) < 8 - half_o ? static_cast<int32_t>(k)
                                                                   : nel - 8 + static_cast<int32_t>(k);
            if (e < nvalid) {
                const uint32_t ue = static_cast<uint32_t>(e);
                crow[e] = *reinterpret_cast<const uint16_t*>(brow + (((ue >> 3) ^ sw) << 4) + ((ue & 7u) << 1));
            }
        }
    }
}

// MC > 1 (single CTAs only: CG = 1, MC = 2, 4 or 8): the MC CTAs of a
// cluster split one 128 x BN tile's K loop (split-K within the cluster) and
// reduce their fp32 partial sums through distributed shared memory; that puts
// MC SMs on each tile of a shape with too few tiles to fill the GPU (a skinny
// M), each reading 1/MC of the tile's operands. Every operand copy lands in
// the issuing CTA's own shared memory (no cluster multicast).
template <int CG, int BN, int kDt, int MC, int kEW = kEpiWarps>
__global__ void __launch_bounds__(32 * (kEW + 3), 1)
hgemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC32,
                const __grid_constant__ CUtensorMap tmB2,
                const TcParams p) {
#if defined(__CUDA_ARCH__) && defined(__CUDA_ARCH_FEAT_SM103_ALL)
    using Cfg = TcCfg<CG, BN, elem_bytes(kDt), (CG == 1 && MC > 1) ? MC : 1>;
    // B is MN-major for every kind. kind::f16 and kind::f8f6f4 read it in the
    // 128-byte swizzle (descriptor layout 2). kind::tf32 reads an MN-major
    // operand only in the 128-byte swizzle with 32-byte atomicity (layout 1:
    // 4-row cores of 128 B rows whose 32-byte units sit at unit ^ (row % 4);
    // layout 2 multiplies as zero), which TMA writes with
    // CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B. Both checked exactly on this GPU.
    constexpr int S = Cfg::kStages;
    constexpr int kCluster = CG * MC;
    constexpr bool kSplit = CG == 1 && MC > 1;               // K split across the cluster
    static_assert(MC == 1 || (kSplit && (MC == 2 || MC == 4 || MC == 8)),
                  "a CTA pair, or a K split across 2, 4 or 8 single CTAs");
    // The split's reduction: 16-bit C, whole 64-column chunks, column slices
    // of at least eight 16-byte units, every CTA's slice received in the ring.
    static_assert(!kSplit || (kDt <= 1 && !Cfg::kHalfLast && BN / MC >= 32 &&
                              kBlockMCta * BN * 4 + kEpiWarps * 8192 <= S * Cfg::kStageBytes),
                  "K split shapes");
    // K split: the blocks of partial sums received from the cluster (MC of
    // them, 128 rows x BN / MC fp32 each) fill the ring from its start; each
    // epilogue warp's 8 KB staging area for the chunk it sends follows.
    constexpr uint32_t kSplitStageOffset = static_cast<uint32_t>(kBlockMCta * BN * 4);
    static_assert(!kSplit || (2 * S + 7) * 8 + 8 + 8 * kEpiWarps + 24 <= Cfg::kBarBytes, "barrier area");
    static_assert(S >= 2, "the two producers take alternate stages");
    // Epilogue warps: 8 (two per TMEM lane quarter, 64-column chunks), or 16
    // (four per quarter, 32-column chunks) on 224- and 256-wide tiles of a
    // 16-bit C (fp16, bf16, and the bf16 C of fp8). Each warp's chain of TMEM
    // load, conversion, staging and store is latency-bound, and the epilogue
    // sets the pace of short K loops and of a last wave: twice the warps keep
    // twice the chunks in flight. The producers and the MMA warp follow.
    constexpr int EW = kEW;
    static_assert(EW == 8 || (EW == 16 && MC == 1 && kDt != 2 && BN % 32 == 0),
                  "16 epilogue warps: 16-bit C, no K split");
    constexpr int kProd = EW, kMma = EW + 1, kProd2 = EW + 2;
    constexpr int kChunkCols = EW == 16 ? 32 : 64;           // columns of an epilogue chunk
    constexpr int NCH = (BN + kChunkCols - 1) / kChunkCols;  // chunks per tile
    constexpr int kColGroups = EW / 4;                       // warps per lane quarter
    constexpr uint32_t kBoxBytes = static_cast<uint32_t>(kEpiBoxRows * kChunkCols * 2);
    static_assert(EW * kBoxBytes == static_cast<uint32_t>(Cfg::kEpiBytes) || kSplit, "staging boxes");
    // One partial-sum barrier per epilogue warp, for stream-K owners (8
    // epilogue warps only: a 16-warp instance takes whole tiles).
    constexpr int kPartBars = EW == 8 ? EW : 0;
    static_assert((2 * S + 7) * 8 + 8 + 8 * kPartBars <= Cfg::kBarBytes, "barrier area");

    extern __shared__ uint8_t smem_raw[];
    if (threadIdx.x == 0) trace_slot(p, kTrLaunchSlot, 0);   // entry
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);
    const uint32_t sA = base;                                   // S x 16 KiB
    const uint32_t sB = sA + S * Cfg::kABytes;                  // S x kBBytes
    const uint32_t sEpi = sB + S * Cfg::kBBytes;                // 4 warps x 2 x 4 KiB
    const uint32_t sBar = sEpi + Cfg::kEpiBytes;
    const uint32_t bar_full = sBar;                             // [S]
    const uint32_t bar_empty = sBar + 8 * S;                    // [S]
    const uint32_t bar_tfull = sBar + 16 * S;                   // [2]
    const uint32_t bar_tempty = bar_tfull + 16;                 // [2]
    const uint32_t bar_drain = bar_tempty + 16;
    const uint32_t bar_pre = bar_drain + 8;                     // [2]
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + (bar_pre + 16 - base));
    volatile uint32_t* const abort_flag = tmem_slot + 1;
    const uint32_t bar_part = bar_pre + 24;                     // [kPartBars]
    const uint32_t bar_rok = bar_part + 8 * kPartBars;          // K split: peers' rings free
    const uint32_t bar_rdy = bar_rok + 8;                       // K split: all CTAs' sums landed
    const uint32_t bar_sent = bar_rdy + 8;                      // K split: this CTA's warps sent

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t crank = (kCluster > 1) ? cluster_ctarank() : 0u;  // rank in the cluster
    const uint32_t rank = crank & static_cast<uint32_t>(CG - 1);        // rank in the CTA pair
    const uint32_t pair = crank / CG;                                   // pair in the cluster
    const uint32_t leader = pair * CG;                                  // the pair's MMA CTA
    const int cluster_id = static_cast<int>(blockIdx.x) / kCluster;
    constexpr int kRowsPerUnit = kSplit ? kBlockMCta : kBlockMCta * kCluster;  // C rows per work unit
    // This CTA's first row within the unit.
    const int32_t m_in_unit = kSplit ? 0 : static_cast<int32_t>(pair * CG + rank) * kBlockMCta;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            // the one MMA issuer that reads the stage frees it (the pair
            // leader's, or this CTA's own)
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + 8 * a, 1);
            mbar_init(bar_tempty + 8 * a, EW * CG);
        }
        mbar_init(bar_drain, 1);
        for (int a = 0; a < 2; ++a) mbar_init(bar_pre + 8 * a, EW * CG);
        for (int e = 0; e < kPartBars; ++e) mbar_init(bar_part + 8 * e, 1);
        if constexpr (kSplit) {
            mbar_init(bar_rok, MC - 1);
            // 128-wide tiles: the peers' parts arrive by bulk copies counted
            // in bytes on bar_rdy, armed once by this CTA
            mbar_init(bar_rdy, Cfg::kChunks == 2 ? 1 : MC);
            mbar_init(bar_sent, EW);
        }
        *abort_flag = 0;
        fence_mbarrier_init_cluster();
    }
    if (warp == kProd && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (Cfg::kBPartial) tma_prefetch_desc(&tmB2);
        if (p.store_mode == 1) tma_prefetch_desc(&tmC);
        if (p.store_mode == 1 && (Cfg::kHalfLast || EW == 16) && kDt != 2) tma_prefetch_desc(&tmC32);  // 16-bit C only
    }
    if (warp == kMma) tmem_alloc<CG>(smem_addr(tmem_slot), Cfg::kTmemCols);
    tc_fence_before();
    __syncthreads();
    if constexpr (kCluster > 1) cluster_sync();
    tc_fence_after();
    // Launched as a programmatic dependent of an operand copy, the kernel has
    // run its set-up alongside the copy; global memory is read only after it.
    grid_dependency_wait();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    const Waiter w{abort_flag, p.timeout_ns, p.status};
    if (threadIdx.x == 0) trace_stamp(p, 0, kTrSetup);

    if (warp == kProd || warp == kProd2) {
        // ------------------------------------------------------------ producer
        // Two producer warps take alternate K blocks of the CTA's sequence
        // (block g of the sequence goes to stage g mod S): one warp needs
        // longer to issue a stage (a barrier wait, the expected-bytes arrive,
        // the TMA copies) than a 256-wide pair MMA takes to consume it, so a
        // single producer would starve the tensor core. The whole warp runs
        // the loop and one elected lane issues the copies: with warp-uniform
        // coordinates the copies issue faster than from a lone lane.
        {
            const uint32_t pid = warp == kProd ? 0u : 1u;
            uint32_t stage = pid, phase = 0;
            uint32_t g = 0;
            bool ok = true;
            long long tw_empty = 0;
            WorkUnit wu;
            for (int lu = 0; ok && next_unit(p.sched, cluster_id, lu, wu); ++lu) {
                if (pid == 0) trace_stamp(p, lu, kTrProdFirst);
                int32_t tm, tn;
                tile_coord(wu.tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
                const int32_t m0 = tm * kRowsPerUnit + m_in_unit;
                const int32_t n0 = tn * BN + static_cast<int32_t>(rank) * Cfg::kBnCta;
                int32_t kb_lo = wu.kb0, kb_hi = wu.kb1;
                if constexpr (kSplit) split_share(wu.kb0, wu.kb1, crank, MC, kb_lo, kb_hi);
                for (int kb = kb_lo; kb < kb_hi; ++kb, ++g) {
                    if ((g & 1u) != pid) continue;
                    HG_TW_BEGIN();
                    const bool got = wait_bar_warp(bar_empty + 8 * stage, phase ^ 1u, w, kRoleProducer, stage);
                    HG_TW_END(tw_empty);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_dst = sA + stage * Cfg::kABytes;
                    const uint32_t b_dst = sB + stage * Cfg::kBBytes;
                    const uint32_t fb = bar_full + 8 * stage;
                    const int32_t k0 = kb * Cfg::kBK;
                    // im2col: this CTA's 128 output pixels start at m0; the
                    // copy walks them from the first one's receptive-field
                    // origin, shifted by the K block's filter tap
                    int32_t ic = 0, iw = 0, ih = 0, in_ = 0;
                    uint16_t ow = 0, oh = 0;
                    if (p.im2col) {
                        const int32_t tap = kb / p.cv_cblocks;
                        ic = (kb - tap * p.cv_cblocks) * Cfg::kBK;
                        ow = static_cast<uint16_t>(tap % p.cv_S);
                        oh = static_cast<uint16_t>(tap / p.cv_S);
                        const int32_t q = m0 % p.cv_Q;
                        const int32_t pq = m0 / p.cv_Q;
                        iw = q * p.cv_stride - p.cv_pad;
                        ih = (pq % p.cv_P) * p.cv_stride - p.cv_pad;
                        in_ = pq / p.cv_P;
                    }
                    if (elect_one_sync()) {
                        if constexpr (CG == 1) {
                            mbar_arrive_expect_tx(fb, Cfg::kTxBytes);
                            if (p.im2col) tma_load_im2col_4d(a_dst, &tmA, fb, ic, iw, ih, in_, ow, oh);
                            else tma_load_2d(a_dst, &tmA, fb, k0, m0);
#pragma unroll
                            for (int j = 0; j < Cfg::kBAtoms; ++j)
                                tma_load_2d(b_dst + j * Cfg::kBAtomBytes,
                                            (Cfg::kBPartial && j == Cfg::kBAtoms - 1) ? &tmB2 : &tmB, fb,
                                            n0 + Cfg::kAtomCols * j, k0);
                        } else {
                            const uint32_t fb_leader = mapa_shared(fb, leader);
                            if (rank == 0) mbar_arrive_expect_tx(fb, Cfg::kTxBytes);
                            if (p.im2col) tma_load_im2col_4d_pair(a_dst, &tmA, fb_leader, ic, iw, ih, in_, ow, oh);
                            else tma_load_2d_pair(a_dst, &tmA, fb_leader, k0, m0);
#pragma unroll
                            for (int j = 0; j < Cfg::kBAtoms; ++j)
                                tma_load_2d_pair(b_dst + j * Cfg::kBAtomBytes,
                                                 (Cfg::kBPartial && j == Cfg::kBAtoms - 1) ? &tmB2 : &tmB,
                                                 fb_leader,
                                                 n0 + Cfg::kAtomCols * j, k0);
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
            trace_wait_total(p, pid == 0 ? kTwProdEmpty0 : kTwProdEmpty1, tw_empty);
            if (!ok) {
                // Loads already issued still land in this CTA's shared memory:
                // give them time before the CTA may exit.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 50000ull) {}
            }
        }
    } else if (warp == kMma) {
        // ----------------------------------------------------------------- MMA
        // The leader CTA's MMA warp runs the loop as a whole warp and one
        // elected lane issues each stage's tcgen05.mma and commit: with
        // warp-uniform descriptors and addresses the issue takes fewer cycles
        // than from a lone lane, which matters because a 256-wide stage leaves
        // the issuing thread little slack over the tensor core's 512 cycles.
        if (rank == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            bool issued = false;
            uint32_t pre_phase[2] = {0u, 0u};
            long long tw_full = 0, tw_tempty = 0, n_stages = 0;
#ifdef HG_TRACE
            const long long t_span0 = clock64();
#endif
            const uint64_t a_desc0 = sdesc_sw128(sA, 16u, 1024u);
            // MN-major B: atoms kBAtomBytes apart (tf32 in the 32-byte-atom
            // layout, the others in the 128-byte swizzle).
            const uint64_t b_desc0 = kDt == 2 ? sdesc_mn_tf32(sB, Cfg::kBAtomBytes)
                                              : sdesc_sw128(sB, Cfg::kBAtomBytes, 1024u);
            WorkUnit wu;
            for (int it = 0; next_unit(p.sched, cluster_id, it, wu); ++it) {
                const uint32_t acc = static_cast<uint32_t>(it) & 1u;
                const uint32_t acc_phase = (static_cast<uint32_t>(it) >> 1) & 1u;
                HG_TW_BEGIN();
                const bool got_acc = wait_bar_warp(bar_tempty + 8 * acc, acc_phase ^ 1u, w, kRoleMma, 32 + acc);
                HG_TW_END(tw_tempty);
                if (!got_acc) {
                    ok = false;
                    break;
                }
                if (wu.kind == 1) {
                    // A stream-K owner accumulates on top of its partners' partial
                    // sums, which the epilogue warps load into this buffer.
                    if (!wait_bar_warp(bar_pre + 8 * acc, pre_phase[acc], w, kRoleMma, 40 + acc)) {
                        ok = false;
                        break;
                    }
                    pre_phase[acc] ^= 1u;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                // An owner's first MMA adds to the preloaded partial sums.
                uint32_t accum = wu.kind == 1 ? 1u : 0u;
                int32_t kb_lo = wu.kb0, kb_hi = wu.kb1;
                if constexpr (kSplit) split_share(wu.kb0, wu.kb1, crank, MC, kb_lo, kb_hi);
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    HG_TW_BEGIN();
                    const bool got_full = wait_bar_warp(bar_full + 8 * stage, phase, w, kRoleMma, stage);
                    HG_TW_END(tw_full);
                    if (!got_full) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    ++n_stages;
                    if (kb == kb_lo) trace_stamp(p, it, kTrMmaFirst);
                    // Descriptor start addresses are in 16-byte units: stage s
                    // adds s * stage bytes / 16; each MMA step (32 bytes of K)
                    // moves 32 bytes along A's swizzled rows and kUK rows of
                    // 128 B down B's atoms.
                    const uint64_t ad = a_desc0 + ((stage * Cfg::kABytes) >> 4);
                    const uint64_t bd = b_desc0 + ((stage * Cfg::kBBytes) >> 4);
                    if (elect_one_sync()) {
#pragma unroll
                        for (int kk = 0; kk < Cfg::kBK / Cfg::kUK; ++kk) {
                            if constexpr (kDt == 2)
                                umma_tf32<CG>(d_tmem, ad + 2u * kk, bd + 8u * Cfg::kUK * kk, p.idesc, accum);
                            else if constexpr (kDt >= 3)
                                umma_f8<CG>(d_tmem, ad + 2u * kk, bd + 8u * Cfg::kUK * kk, p.idesc, accum);
                            else
                                umma_f16<CG>(d_tmem, ad + 2u * kk, bd + 8u * Cfg::kUK * kk, p.idesc, accum);
                            accum = 1u;
                        }
                        // A stage is free once the MMAs that read it are done; a
                        // pair's commit arrives on both CTAs' barriers.
                        if constexpr (CG == 1) umma_commit(bar_empty + 8 * stage);
                        else umma_commit_pair(bar_empty + 8 * stage, static_cast<uint16_t>(0x3u << leader));
                    }
                    __syncwarp();
                    accum = 1u;
                    issued = true;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (elect_one_sync()) {
                    if constexpr (CG == 1) umma_commit(bar_tfull + 8 * acc);
                    else umma_commit_pair(bar_tfull + 8 * acc, static_cast<uint16_t>(0x3u << leader));
                }
                __syncwarp();
                trace_stamp(p, it, kTrMmaLast);
            }
            trace_wait_total(p, kTwMmaFull, tw_full);
            trace_wait_total(p, kTwMmaTempty, tw_tempty);
            trace_wait_total(p, kTwMmaStages, n_stages);
#ifdef HG_TRACE
            trace_wait_total(p, kTwMmaSpan, clock64() - t_span0);
#endif
            if (!ok && issued) {
                // TMEM may only be freed once every issued MMA has completed.
                if (elect_one_sync()) {
                    if constexpr (CG == 1) umma_commit(bar_drain);
                    else umma_commit_pair(bar_drain, static_cast<uint16_t>(1u << leader));
                }
                __syncwarp();
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar_drain, 0) && globaltimer_ns() - t0 < p.timeout_ns) {}
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Warp w reads TMEM lane quarter w % 4 (rows 32(w % 4) .. +31 of the
        // CTA's tile) and every (EW / 4)-th chunk, starting at chunk w / 4:
        // every other 64-column chunk with 8 warps, every fourth 32-column
        // chunk with 16.
        const int quarter = warp & 3;
        const int colhalf = warp >> 2;        // the warp's column group (0 .. kColGroups - 1)
        const uint32_t box = sEpi + static_cast<uint32_t>(warp) * kBoxBytes;
        uint8_t* const box_ptr = smem + (box - base);
        // Stream-K owner unit `j` (the cluster's last): before its MMAs start,
        // put the partners' partial sums into its accumulator buffer (this
        // warp's lanes and chunks), so its own epilogue is a plain one. The
        // partners publish them with the first units of their ranges, usually
        // long before; if a partner's mark is not there yet the warp writes
        // zeros instead and adds the partial sums in the owner's epilogue (it
        // never blocks here, so no wait can chain across clusters). The
        // buffer's previous contents were read by this warp already.
        bool owner_preloaded = false;
        auto preload_owner = [&](int j, const WorkUnit& ou) {
            const uint32_t pacc = static_cast<uint32_t>(j) & 1u;
            const uint32_t p_row = tmem_base + pacc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
            const int32_t contrib_last = sk_last_contributor(p.sched, ou.tile);
            // Test hook: look for a mark no part ever writes.
            const unsigned long long want = p.inject == 1 ? ~p.epoch : p.epoch;
            bool have = true;
            for (int32_t q = cluster_id + 1; q <= contrib_last && have; ++q)
                have = ld_acquire_gpu(p.flags + 2 * partial_block<kCluster>(q, crank, quarter) + colhalf) == want;
            owner_preloaded = have;
#pragma unroll 1
            for (int c = colhalf; c < Cfg::kChunks; c += 2) {
                const bool half = Cfg::kHalfLast && c == Cfg::kChunks - 1;
                uint32_t r0[32], r1[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    r0[i] = 0u;
                    r1[i] = 0u;
                }
                for (int32_t q = cluster_id + 1; q <= contrib_last && have; ++q) {
                    const float4* src = reinterpret_cast<const float4*>(p.partials) +
                                        partial_block<kCluster>(q, crank, quarter) * (kEpiBoxRows * BN / 4);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const float4 a = __ldcg(src + (c * 16 + jj) * 32 + lane);
                        r0[4 * jj] = __float_as_uint(__uint_as_float(r0[4 * jj]) + a.x);
                        r0[4 * jj + 1] = __float_as_uint(__uint_as_float(r0[4 * jj + 1]) + a.y);
                        r0[4 * jj + 2] = __float_as_uint(__uint_as_float(r0[4 * jj + 2]) + a.z);
                        r0[4 * jj + 3] = __float_as_uint(__uint_as_float(r0[4 * jj + 3]) + a.w);
                        if (!half) {
                            const float4 b = __ldcg(src + (c * 16 + 8 + jj) * 32 + lane);
                            r1[4 * jj] = __float_as_uint(__uint_as_float(r1[4 * jj]) + b.x);
                            r1[4 * jj + 1] = __float_as_uint(__uint_as_float(r1[4 * jj + 1]) + b.y);
                            r1[4 * jj + 2] = __float_as_uint(__uint_as_float(r1[4 * jj + 2]) + b.z);
                            r1[4 * jj + 3] = __float_as_uint(__uint_as_float(r1[4 * jj + 3]) + b.w);
                        }
                    }
                }
                tmem_st_32x32b_x32(p_row + 64u * c, r0);
                if (!half) tmem_st_32x32b_x32(p_row + 64u * c + 32u, r1);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1) {
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar_pre + 8 * pacc) : "memory");
                } else {
                    mbar_arrive_cluster(mapa_shared(bar_pre + 8 * pacc, leader));
                }
            }
        };
        auto preload_if_owner = [&](int j) {
            if constexpr (EW == 8) {   // stream-K: 8 epilogue warps only
                WorkUnit ou;
                if (next_unit(p.sched, cluster_id, j, ou) && ou.kind == 1) preload_owner(j, ou);
            }
        };
        preload_if_owner(0);
        preload_if_owner(1);
        WorkUnit wu;
        for (int it = 0; next_unit(p.sched, cluster_id, it, wu); ++it) {
            const uint32_t acc = static_cast<uint32_t>(it) & 1u;
            const uint32_t acc_phase = (static_cast<uint32_t>(it) >> 1) & 1u;
            if (!wait_bar(bar_tfull + 8 * acc, acc_phase, w, kRoleEpilogue, 32 + acc)) break;
            tc_fence_after();
            if (warp == 0 && lane == 0) {
                trace_stamp(p, it, kTrEpiStart);
                trace_chunk(p, it, 12, kTcStart);
#ifdef HG_TRACE
                if (p.trace && it < kTraceUnits)
                    p.trace[(static_cast<int64_t>(blockIdx.x) * kTraceUnits + it) * kTraceFields + kTrUnit] =
                        (static_cast<unsigned long long>(wu.tile) << 32) |
                        (static_cast<unsigned long long>(wu.kb0) << 16) | static_cast<unsigned long long>(wu.kb1);
#endif
            }
            int32_t tm, tn;
            tile_coord(wu.tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            const int32_t row0 = tm * kRowsPerUnit + m_in_unit + quarter * kEpiBoxRows;
            const int32_t col0 = tn * BN;
            const uint32_t t_row = tmem_base + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
            if constexpr (kSplit) {
                // K split across the cluster (one tile per cluster): each CTA
                // holds the fp32 sum over its share of the K blocks. CTA j owns
                // the tile's columns [j S, (j + 1) S), S = BN / MC, and receives
                // every CTA's partial sums of them in its stage ring, idle once
                // its MMAs are done: block q (the sender's rank) of 128 rows x S
                // floats, 16-byte unit u of row r at unit u ^ (r % 8), so the
                // 8 lanes of each store phase cover the 32 banks once.
                constexpr uint32_t kSliceCols = BN / MC;
                constexpr uint32_t kRowBytes = kSliceCols * 4u;
                constexpr uint32_t kBlockBytes = kBlockMCta * kRowBytes;
                constexpr int kUnitsPerRow = static_cast<int>(kSliceCols / 4u);
                int32_t kb_lo, kb_hi;
                split_share(wu.kb0, wu.kb1, crank, MC, kb_lo, kb_hi);
                // 1. This CTA's MMAs have completed (tmem_full): its ring may
                //    be written by the peers. Test hook: rank 0 never says so,
                //    and its peers' waits run out.
                constexpr bool kBulkExchange = Cfg::kChunks == 2;   // one chunk per warp
                if (kBulkExchange && warp == 0 && lane == 0)
                    mbar_arrive_expect_tx(bar_rdy, static_cast<uint32_t>(MC - 1) * kBlockBytes);
                if (warp == 0 && lane == 0 && !(p.inject == 2 && crank == 0)) {
                    for (uint32_t q = 0; q < static_cast<uint32_t>(MC); ++q)
                        if (q != crank) mbar_arrive_cluster(mapa_shared(bar_rok, q));
                }
                // 2. Once every peer's ring is free, send each owner its columns.
                if (warp == 0 && lane == 0) {
                    trace_chunk(p, it, 12, kTcStart);
                    trace_chunk(p, it, 0, kTcStart);
                }
                bool ok = wait_bar_cluster_warp(bar_rok, 0, w, kRoleEpilogue, 96);
                if (warp == 0 && lane == 0) trace_chunk(p, it, 0, kTcLdDone);
                if (lane == 0) trace_chunk(p, it, 1 + warp, kTcLdDone);
                if constexpr (kBulkExchange) {
                    // 128-wide tiles: each warp holds one 64-column chunk, one
                    // or two owners' whole slice rows (32 rows each). Its own
                    // columns go straight into its own block; a peer's part is
                    // laid out in the staging area exactly as the owner's
                    // block holds it (row r at r * row bytes, unit u at
                    // u ^ (r % 8)), then moved by one bulk copy, which counts
                    // its bytes on the owner's bar_rdy.
                    const int c = colhalf;
                    uint32_t r0[32], r1[32];
                    tmem_ld_32x32b_x32(t_row + 64u * c, r0);
                    tmem_ld_32x32b_x32(t_row + 64u * c + 32u, r1);
                    tmem_ld_wait();
                    reg_fence(r0);
                    reg_fence(r1);
                    if (kb_hi == kb_lo) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            r0[i] = 0u;
                            r1[i] = 0u;
                        }
                    }
                    if (lane == 0) trace_chunk(p, it, 1 + warp, kTcPacked);
                    constexpr uint32_t kPartCols = kSliceCols >= 64u ? 64u : kSliceCols;
                    constexpr uint32_t kPartUnits = kPartCols / 4u;
                    constexpr uint32_t kPartBytes = 32u * kRowBytes;                // 32 rows of the owner's slice
                    static_assert(kRowBytes == kPartCols * 4u, "a part is whole slice rows");
                    const uint32_t stage = sA + kSplitStageOffset + static_cast<uint32_t>(warp) * 8192u;
                    const uint32_t rows_off = static_cast<uint32_t>(quarter * 32) * kRowBytes;
#pragma unroll
                    for (uint32_t part = 0; part < 64u / kPartCols; ++part) {
                        const uint32_t col = 64u * static_cast<uint32_t>(c) + part * kPartCols;
                        const uint32_t owner_cta = col / kSliceCols;
                        const bool own = owner_cta == crank;
                        const uint32_t dst = own ? sA + crank * kBlockBytes + rows_off : stage + part * kPartBytes;
#pragma unroll
                        for (uint32_t j = 0; j < kPartUnits; ++j) {
                            const uint32_t ju = part * kPartUnits + j;               // unit within the chunk
                            const uint32_t* v = ju < 8 ? r0 + 4 * ju : r1 + 4 * (ju - 8);
                            st_shared_v4(dst + lane * kRowBytes + ((j ^ (lane & 7u)) << 4), v[0], v[1], v[2], v[3]);
                        }
                        if (!own && ok) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0)
                                bulk_copy_to_peer(mapa_shared(sA + crank * kBlockBytes + rows_off, owner_cta), dst,
                                                  kPartBytes, mapa_shared(bar_rdy, owner_cta));
                        }
                        __syncwarp();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        trace_chunk(p, it, 1 + warp, kTcWaitRead);
                        if (warp == 0) trace_chunk(p, it, 0, kTcWaitRead);
                        release_accumulator<CG>(bar_tempty + 8 * acc, leader);
                        // 3. This warp's own columns are in its own block.
                        mbar_arrive_local(bar_sent);
                        trace_chunk(p, it, 1 + warp, kTcStaged);
                    }
                    // 4. Every warp's own columns, and every peer's bytes.
                    ok = wait_bar(bar_sent, 0, w, kRoleEpilogue, 98) && ok;
                    if (warp == 0 && lane == 0) trace_chunk(p, it, 0, kTcStaged);
                    ok = wait_bar(bar_rdy, 0, w, kRoleEpilogue, 97) && ok;
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                } else {
                for (int c = colhalf; c < Cfg::kChunks && ok; c += 2) {
                    uint32_t r0[32], r1[32];
                    tmem_ld_32x32b_x32(t_row + 64u * c, r0);
                    tmem_ld_32x32b_x32(t_row + 64u * c + 32u, r1);
                    tmem_ld_wait();
                    reg_fence(r0);
                    reg_fence(r1);
                    if (lane == 0) trace_chunk(p, it, 1 + warp, kTcPacked);
                    if (kb_hi == kb_lo) {
                        // no K block in this CTA's share: its partial sum is zero
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            r0[i] = 0u;
                            r1[i] = 0u;
                        }
                    }
                    // Stage the chunk in this warp's own 32 x 256-byte area, a
                    // row per lane (16-byte unit j of row l at j ^ (l % 8):
                    // each 8-lane phase covers the 32 banks once), then read it
                    // back row-contiguously: every cluster store then writes a
                    // whole 128- or 256-byte row slice of the owner's block, not
                    // 32 scattered 16-byte pieces (measured: 2700 cycles per
                    // warp for a chunk's stores the scattered way).
                    const uint32_t stage = sA + kSplitStageOffset + static_cast<uint32_t>(warp) * 8192u;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint32_t* v = j < 8 ? r0 + 4 * j : r1 + 4 * (j - 8);
                        st_shared_v4(stage + lane * 256u + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), v[0], v[1],
                                     v[2], v[3]);
                    }
                    __syncwarp();
                    // units of the chunk per owner row: 16 (the chunk lies in
                    // one owner's slice) or 8 (it spans two 32-column slices)
                    constexpr uint32_t kU = kSliceCols >= 64u ? 16u : kSliceCols / 4u;
                    constexpr uint32_t kRowsPerStore = 32u / kU;
                    const uint32_t uu = lane % kU;                       // unit within the owner's part
                    const uint32_t rsub = lane / kU;                     // row within the store
#pragma unroll
                    for (uint32_t part = 0; part < 16u / kU; ++part) {
                        const uint32_t col = 64u * static_cast<uint32_t>(c) + 4u * (part * kU);  // first column of the part
                        const uint32_t owner_cta = col / kSliceCols;
                        const uint32_t u_slice = (col % kSliceCols) / 4u + uu;   // unit within the slice row
                        const uint32_t u_chunk = part * kU + uu;                // unit within the chunk
                        const uint32_t dst_base = owner_cta == crank ? sA : mapa_shared(sA, owner_cta);
#pragma unroll 4
                        for (uint32_t i = 0; i < 32u / kRowsPerStore; ++i) {
                            const uint32_t rl = i * kRowsPerStore + rsub;                 // row in the warp's 32
                            const float4 q4 = ld_shared_f4(stage + rl * 256u + ((u_chunk ^ (rl & 7u)) << 4));
                            const uint32_t rt = static_cast<uint32_t>(quarter * 32) + rl;  // row in the tile
                            const uint32_t off = crank * kBlockBytes + rt * kRowBytes + ((u_slice ^ (rt & 7u)) << 4);
                            if (owner_cta == crank)
                                st_shared_v4(dst_base + off, __float_as_uint(q4.x), __float_as_uint(q4.y),
                                             __float_as_uint(q4.z), __float_as_uint(q4.w));
                            else
                                st_cluster_v4(dst_base + off, q4.x, q4.y, q4.z, q4.w);
                        }
                    }
                    __syncwarp();
                }
                tc_fence_before();
                __syncwarp();
                if (warp == 0 && lane == 0) trace_chunk(p, it, 0, kTcWaitRead);
                if (lane == 0) trace_chunk(p, it, 1 + warp, kTcWaitRead);
                if (lane == 0) {
                    release_accumulator<CG>(bar_tempty + 8 * acc, leader);
                    // 3. This warp's parts are sent (release at cluster scope).
                    if (ok) mbar_arrive_cluster(mapa_shared(bar_sent, crank));
                    trace_chunk(p, it, 1 + warp, kTcStaged);
                }
                // Warp 0 collects the eight warps' arrivals (a bounded wait: a
                // warp that gave up never arrives) and publishes the CTA's parts
                // to every CTA of the cluster, this one included: its own warps
                // read the block that its other warps wrote.
                if (warp == 0) {
                    const bool sent = wait_bar_cluster_warp(bar_sent, 0, w, kRoleEpilogue, 98);
                    if (sent && lane == 0) {
                        fence_acq_rel_cluster();
                        for (uint32_t q = 0; q < static_cast<uint32_t>(MC); ++q)
                            mbar_arrive_cluster(mapa_shared(bar_rdy, q));
                    }
                    ok = ok && sent;
                    if (lane == 0) trace_chunk(p, it, 0, kTcStaged);
                }
                // 4. Every CTA's block of this CTA's columns is in: sum the
                //    blocks in rank order (the same order on every run), round,
                //    store.
                ok = wait_bar_cluster_warp(bar_rdy, 0, w, kRoleEpilogue, 97) && ok;
                }   // per-thread cluster stores (256-wide tiles)
                if (warp == 0 && lane == 0) trace_chunk(p, it, 0, kTcIssued);
                if (ok) {
                    const int32_t row_base = tm * kBlockMCta;
                    const int32_t col_base = col0 + static_cast<int32_t>(crank * kSliceCols);
#pragma unroll 1
                    for (int f = warp * 32 + static_cast<int>(lane); f < kBlockMCta * kUnitsPerRow;
                         f += EW * 32) {
                        const uint32_t rr = static_cast<uint32_t>(f / kUnitsPerRow);
                        const uint32_t u = static_cast<uint32_t>(f % kUnitsPerRow);
                        const uint32_t off = rr * kRowBytes + ((u ^ (rr & 7u)) << 4);
                        float4 acc4 = ld_shared_f4(sA + off);
#pragma unroll
                        for (int q = 1; q < MC; ++q) {
                            const float4 t = ld_shared_f4(sA + static_cast<uint32_t>(q) * kBlockBytes + off);
                            acc4.x += t.x;
                            acc4.y += t.y;
                            acc4.z += t.z;
                            acc4.w += t.w;
                        }
                        const int32_t row = row_base + static_cast<int32_t>(rr);
                        const int32_t col = col_base + 4 * static_cast<int32_t>(u);
                        if (row < p.M && col < p.N) {
                            const uint32_t lo = pack_rn<kDt>(__float_as_uint(acc4.x), __float_as_uint(acc4.y));
                            const uint32_t hi = pack_rn<kDt>(__float_as_uint(acc4.z), __float_as_uint(acc4.w));
                            uint16_t* dst = p.C + static_cast<int64_t>(row) * p.ldc + col;
                            if (p.store_mode != 2 && p.store_mode != 5 && col + 4 <= p.N) {
                                // C 16-byte aligned with a 16-byte pitch, col a
                                // multiple of 4: an 8-byte aligned store
                                *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
                            } else {
                                const uint16_t e4[4] = {static_cast<uint16_t>(lo & 0xFFFFu), static_cast<uint16_t>(lo >> 16),
                                                        static_cast<uint16_t>(hi & 0xFFFFu), static_cast<uint16_t>(hi >> 16)};
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    if (col + e < p.N) dst[e] = e4[e];
                            }
                        }
                    }
                }
                if (warp == 0 && lane == 0) {
                    trace_chunk(p, it, 0, kTcStored);
                    trace_stamp(p, it, kTrEpiEnd);
                }
                continue;
            }
            const bool is_split = EW == 8 && wu.kind != 0;   // stream-K units: 8 epilogue warps only
            const bool owner = wu.kind != 2;
            if (colhalf >= NCH) {
                // No chunk for this warp (a 64-wide tile): release at once.
                __syncwarp();
                if (lane == 0) release_accumulator<CG>(bar_tempty + 8 * acc, leader);
                preload_if_owner(it + 2);
                continue;
            }
            const int32_t contrib_last = (is_split && owner) ? sk_last_contributor(p.sched, wu.tile)
                                                             : cluster_id;
            const bool owner_adds = is_split && owner && !owner_preloaded;
            if (owner_adds) {
                // The preload found a partner's mark missing: wait for the marks
                // now (this is the cluster's last unit; nothing else of this CTA
                // is in flight) and add the partial sums below. Test hook: wait
                // for a mark no part ever writes; the wait runs out.
                const unsigned long long want = p.inject == 1 ? ~p.epoch : p.epoch;
                for (int32_t q = cluster_id + 1; q <= contrib_last; ++q)
                    if (!wait_flag(p.flags + 2 * partial_block<kCluster>(q, crank, quarter) + colhalf, want, w,
                                   64 + ((q - cluster_id) & 63)))
                        break;
                if (warp == 0 && lane == 0) trace_slot(p, 30, 0);
            }
            if (is_split && !owner && warp == 0 && lane == 0) trace_slot(p, 29, 0);
            // An owner adding its partners' partial sums copies them, a chunk at
            // a time, into the stage ring by bulk copies: its unit is the
            // CTA's last, so once its MMAs are done (the tmem_full wait above)
            // the ring is idle and no load is in flight. The copies of a chunk
            // run while its TMEM loads do.
            const int32_t n_part = contrib_last - cluster_id;
            const bool bulk_adds = owner_adds && n_part <= Cfg::kBulkPartners;
            const uint32_t part_buf = sA + static_cast<uint32_t>(warp) * static_cast<uint32_t>(n_part) * 8192u;
            uint32_t part_phase = 0;
#pragma unroll 1
            for (int c = colhalf; c < NCH; c += kColGroups) {
                // A chunk is 64 columns (two 32-column TMEM loads), or 32 for the
                // last chunk of a tile whose width is an odd multiple of 32, and
                // for every chunk with 16 epilogue warps.
                const bool half = EW == 16 || (Cfg::kHalfLast && c == NCH - 1);
                const bool last = c + kColGroups >= NCH;
                if (warp == 0 && lane == 0) trace_chunk(p, it, c, kTcStart);
                if (bulk_adds && lane == 0) {
                    // chunk c of a partial block: float4s [16c * 32, 16(c + 1) * 32)
                    const uint32_t bytes = half ? 4096u : 8192u;
                    fence_proxy_async_all();
                    mbar_arrive_expect_tx(bar_part + 8 * warp, bytes * static_cast<uint32_t>(n_part));
                    for (int32_t q = 0; q < n_part; ++q)
                        bulk_load(part_buf + static_cast<uint32_t>(q) * 8192u,
                                  reinterpret_cast<const float4*>(p.partials) +
                                      partial_block<kCluster>(cluster_id + 1 + q, crank, quarter) * (kEpiBoxRows * BN / 4) +
                                      c * 16 * 32,
                                  bytes, bar_part + 8 * warp);
                }
                uint32_t r0[32], r1[32];
                tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(kChunkCols * c), r0);
                if (!half) tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(kChunkCols * c) + 32u, r1);
                tmem_ld_wait();
                reg_fence(r0);
                if (half) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r1[i] = 0u;
                }
                reg_fence(r1);
                if (warp == 0 && lane == 0) trace_chunk(p, it, c, kTcLdDone);
                if (last) {
                    // This warp's TMEM reads of the accumulator are done.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        release_accumulator<CG>(bar_tempty + 8 * acc, leader);
                        if (warp == 0) trace_stamp(p, it, kTrEpiTmemFree);
                    }
                }
                if (is_split) {
                    if (!owner) {
                        // A non-owning K part: publish this chunk's fp32 partial
                        // sums (lane-interleaved, so each warp store is 512
                        // contiguous bytes) instead of writing C.
                        float4* dst = reinterpret_cast<float4*>(p.partials) +
                                      partial_block<kCluster>(cluster_id, crank, quarter) * (kEpiBoxRows * BN / 4);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            dst[(c * 16 + j) * 32 + lane] =
                                make_float4(__uint_as_float(r0[4 * j]), __uint_as_float(r0[4 * j + 1]),
                                            __uint_as_float(r0[4 * j + 2]), __uint_as_float(r0[4 * j + 3]));
                            if (!half)
                                dst[(c * 16 + 8 + j) * 32 + lane] =
                                    make_float4(__uint_as_float(r1[4 * j]), __uint_as_float(r1[4 * j + 1]),
                                                __uint_as_float(r1[4 * j + 2]), __uint_as_float(r1[4 * j + 3]));
                        }
                        if (last) {
                            __threadfence();
                            __syncwarp();
                            if (lane == 0)
                                st_release_gpu(p.flags + 2 * partial_block<kCluster>(cluster_id, crank, quarter) + colhalf,
                                               p.epoch);
                            if (warp == 0 && lane == 0) trace_slot(p, 29, 1);
                        }
                        continue;
                    }
                    if (bulk_adds) {
                        if (wait_bar(bar_part + 8 * warp, part_phase, w, kRoleEpilogue, 80 + warp)) {
                            for (int32_t q = 0; q < n_part; ++q) {
                                const uint32_t src = part_buf + static_cast<uint32_t>(q) * 8192u + lane * 16u;
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const float4 a = ld_shared_f4(src + static_cast<uint32_t>(j) * 512u);
                                    r0[4 * j] = __float_as_uint(__uint_as_float(r0[4 * j]) + a.x);
                                    r0[4 * j + 1] = __float_as_uint(__uint_as_float(r0[4 * j + 1]) + a.y);
                                    r0[4 * j + 2] = __float_as_uint(__uint_as_float(r0[4 * j + 2]) + a.z);
                                    r0[4 * j + 3] = __float_as_uint(__uint_as_float(r0[4 * j + 3]) + a.w);
                                    if (!half) {
                                        const float4 b = ld_shared_f4(src + static_cast<uint32_t>(8 + j) * 512u);
                                        r1[4 * j] = __float_as_uint(__uint_as_float(r1[4 * j]) + b.x);
                                        r1[4 * j + 1] = __float_as_uint(__uint_as_float(r1[4 * j + 1]) + b.y);
                                        r1[4 * j + 2] = __float_as_uint(__uint_as_float(r1[4 * j + 2]) + b.z);
                                        r1[4 * j + 3] = __float_as_uint(__uint_as_float(r1[4 * j + 3]) + b.w);
                                    }
                                }
                            }
                        } else if (lane == 0) {
                            // The wait ran out (the status word says so): let the
                            // copies still in flight land before the CTA can exit.
                            const uint64_t t0 = globaltimer_ns();
                            while (globaltimer_ns() - t0 < 50000ull) {}
                        }
                        part_phase ^= 1u;
                        __syncwarp();
                    } else if (owner_adds) {
                        for (int32_t q = cluster_id + 1; q <= contrib_last; ++q) {
                            const float4* src = reinterpret_cast<const float4*>(p.partials) +
                                                partial_block<kCluster>(q, crank, quarter) * (kEpiBoxRows * BN / 4);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 a = __ldcg(src + (c * 16 + j) * 32 + lane);
                                r0[4 * j] = __float_as_uint(__uint_as_float(r0[4 * j]) + a.x);
                                r0[4 * j + 1] = __float_as_uint(__uint_as_float(r0[4 * j + 1]) + a.y);
                                r0[4 * j + 2] = __float_as_uint(__uint_as_float(r0[4 * j + 2]) + a.z);
                                r0[4 * j + 3] = __float_as_uint(__uint_as_float(r0[4 * j + 3]) + a.w);
                                if (!half) {
                                    const float4 b = __ldcg(src + (c * 16 + 8 + j) * 32 + lane);
                                    r1[4 * j] = __float_as_uint(__uint_as_float(r1[4 * j]) + b.x);
                                    r1[4 * j + 1] = __float_as_uint(__uint_as_float(r1[4 * j + 1]) + b.y);
                                    r1[4 * j + 2] = __float_as_uint(__uint_as_float(r1[4 * j + 2]) + b.z);
                                    r1[4 * j + 3] = __float_as_uint(__uint_as_float(r1[4 * j + 3]) + b.w);
                                }
                            }
                        }
                    }
                }
                if constexpr (kDt == 2) {
                    // fp32 C: the chunk goes out as two 32-column halves (r0, r1),
                    // each a 32 x 32 fp32 box of 128-byte rows in the same
                    // swizzle as the 16-bit boxes (16 B chunk j of row r at
                    // j ^ (r % 8)).
                    // A tile whose width is an odd multiple of 32 ends in a
                    // 32-column chunk: its first half only.
                    float* const Cf = reinterpret_cast<float*>(p.C);
#pragma unroll 1
                    for (int h = 0; h < (half ? 1 : 2); ++h) {
                        const uint32_t* v = h == 0 ? r0 : r1;
                        const int32_t hcol = col0 + 64 * c + 32 * h;
                        if (p.store_mode == 3) {
                            // C 16-byte aligned, pitch and N multiples of 4 floats
                            const int32_t row = row0 + static_cast<int32_t>(lane);
                            if (row < p.M) {
                                float* crow = Cf + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const int32_t col = hcol + 4 * j;
                                    if (col < p.N)
                                        *reinterpret_cast<uint4*>(crow + col) =
                                            make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                                }
                            }
                            continue;
                        }
                        if (p.store_mode == 1) {
                            if (lane == 0) bulk_wait_group_read<0>();
                            __syncwarp();
                        }
                        const uint32_t row_addr = box + lane * 128u;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4),
                                         v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        if (p.store_mode == 1) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                if (row0 < p.M && hcol < p.N) tma_store_2d(&tmC, box, hcol, row0);
                                bulk_commit_group();
                            }
                        } else if (p.store_mode == 4) {
                            // read back row-contiguously: 8 lanes per 128-byte row
                            __syncwarp();
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const uint32_t piece = static_cast<uint32_t>(i) * 32u + lane;
                                const uint32_t rr = piece >> 3, ch = piece & 7u;
                                const uint4 q4 = *reinterpret_cast<const uint4*>(
                                    box_ptr + rr * 128u + ((ch ^ (rr & 7u)) << 4));
                                const int32_t row = row0 + static_cast<int32_t>(rr);
                                const int32_t col = hcol + static_cast<int32_t>(ch * 4u);
                                if (row < p.M && col < p.N)
                                    *reinterpret_cast<uint4*>(Cf + static_cast<int64_t>(row) * p.ldc + col) = q4;
                            }
                            __syncwarp();
                        } else {
                            // plain stores, any pitch: lane = column of the half
                            __syncwarp();
                            const int32_t col = hcol + static_cast<int32_t>(lane);
#pragma unroll 1
                            for (int rr = 0; rr < kEpiBoxRows; ++rr) {
                                const int32_t row = row0 + rr;
                                if (row >= p.M) break;
                                const uint32_t urr = static_cast<uint32_t>(rr);
                                if (col < p.N)
                                    Cf[static_cast<int64_t>(row) * p.ldc + col] = *reinterpret_cast<const float*>(
                                        box_ptr + urr * 128u + (((lane >> 2) ^ (urr & 7u)) << 4) + ((lane & 3u) << 2));
                            }
                            __syncwarp();
                        }
                    }
                    if (is_split && owner && warp == 0 && lane == 0) trace_slot(p, 30, 3 + (c >> 1));
                    continue;
                } else {
                if constexpr (kDt >= 3) {
                    // fp8: C = bf16(acc * (a_scale[row] * b_scale[col])), the
                    // per-channel scales applied in fp32 once the sum is done
                    const int32_t srow = row0 + static_cast<int32_t>(lane);
                    const float sa = (p.a_scale && srow < p.M) ? __ldg(p.a_scale + srow) : 1.0f;
                    const int32_t scol = col0 + kChunkCols * c;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int32_t c0i = scol + i;
                        const float sb0 = (p.b_scale && c0i < p.N) ? __ldg(p.b_scale + c0i) : 1.0f;
                        r0[i] = __float_as_uint(__uint_as_float(r0[i]) * (sa * sb0));
                        if (!half) {
                            const int32_t c1i = scol + 32 + i;
                            const float sb1 = (p.b_scale && c1i < p.N) ? __ldg(p.b_scale + c1i) : 1.0f;
                            r1[i] = __float_as_uint(__uint_as_float(r1[i]) * (sa * sb1));
                        }
                    }
                }
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    pk[i] = pack_rn<kDt>(r0[2 * i], r0[2 * i + 1]);
                    pk[16 + i] = pack_rn<kDt>(r1[2 * i], r1[2 * i + 1]);
                }
                if (warp == 0 && lane == 0) trace_chunk(p, it, c, kTcPacked);
                const int32_t ccol = col0 + kChunkCols * c;
                if (p.store_mode == 3) {
                    // Direct 16-byte stores: thread `lane` writes its own row of the
                    // chunk (C is 16-byte aligned with a pitch of a multiple of 8
                    // elements, and N is a multiple of 8, so a vector is either
                    // wholly inside C or wholly outside).
                    const int32_t row = row0 + static_cast<int32_t>(lane);
                    if (row < p.M) {
                        uint16_t* crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int32_t col = ccol + 8 * j;
                            if ((!half || j < 4) && col < p.N)
                                *reinterpret_cast<uint4*>(crow + col) =
                                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                        }
                    }
                    continue;
                }
                if (p.store_mode == 1) {
                    // The TMA store issued from this box before must have read it.
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
                    if (warp == 0 && lane == 0) trace_chunk(p, it, c, kTcWaitRead);
                }
                // Row `lane` of the box. A 64-column box has 128-byte rows and
                // the 128-byte swizzle: 16 B chunk j goes to j ^ (row % 8). A
                // 32-column box has 64-byte rows and the 64-byte swizzle: chunk j
                // goes to j ^ ((row / 2) % 4). Either way each group of 8 lanes
                // covers all 32 banks once (the SWIZZLE_C idea of the page's
                // coalesced write-back), and the TMA store undoes the swizzle.
                if (!half) {
                    const uint32_t row_addr = box + lane * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4),
                                     pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                } else {
                    const uint32_t row_addr = box + lane * 64u;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ ((lane >> 1) & 3u)) << 4),
                                     pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                }
                if (p.store_mode == 1) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (warp == 0 && lane == 0) trace_chunk(p, it, c, kTcStaged);
                    if (lane == 0) {
                        if (row0 < p.M && ccol < p.N) {
                            if (half) tma_store_2d(&tmC32, box, ccol, row0);
                            else tma_store_2d(&tmC, box, ccol, row0);
                        }
                        bulk_commit_group();
                    }
                    if (warp == 0 && lane == 0) trace_chunk(p, it, c, kTcIssued);
                    if (is_split && owner && warp == 0 && lane == 0) trace_slot(p, 30, 3 + (c >> 1));
                } else if (p.store_mode == 4) {
                    // Read the box back row-contiguously: 8 lanes cover one row's
                    // 128 bytes (64-column box) or 4 lanes its 64 bytes (32-column
                    // box), so every warp store writes whole 128-byte lines.
                    __syncwarp();
                    const uint32_t per_row = half ? 4u : 8u;
                    const int n_inst = half ? 4 : 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (i < n_inst) {
                            const uint32_t piece = static_cast<uint32_t>(i) * 32u + lane;
                            const uint32_t rr = piece / per_row, ch = piece % per_row;
                            const uint32_t phys = half ? (ch ^ ((rr >> 1) & 3u)) : (ch ^ (rr & 7u));
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                box_ptr + rr * (half ? 64u : 128u) + (phys << 4));
                            const int32_t row = row0 + static_cast<int32_t>(rr);
                            const int32_t col = ccol + static_cast<int32_t>(ch * 8u);
                            if (row < p.M && col < p.N)
                                *reinterpret_cast<uint4*>(p.C + static_cast<int64_t>(row) * p.ldc + col) = v;
                        }
                    }
                    __syncwarp();
                    if (warp == 0 && lane == 0) trace_chunk(p, it, c, kTcStored);
                } else if (p.store_mode == 5) {
                    __syncwarp();
                    store_chunk_realigned(box_ptr, p.C, p.ldc, p.M, p.N, row0, ccol, half, lane);
                    __syncwarp();
                } else {
                    __syncwarp();
                    const uint32_t width = half ? 32u : 64u;
#pragma unroll 1
                    for (int rr = 0; rr < kEpiBoxRows; ++rr) {
                        const int32_t row = row0 + rr;
                        if (row >= p.M) break;
                        const uint32_t urr = static_cast<uint32_t>(rr);
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const uint32_t cc = lane * 2u + q;          // column in the box
                            const int32_t col = ccol + static_cast<int32_t>(cc);
                            if (cc < width && col < p.N) {
                                const uint32_t off =
                                    half ? urr * 64u + (((cc >> 3) ^ ((urr >> 1) & 3u)) << 4) + ((cc & 7u) << 1)
                                         : urr * 128u + (((cc >> 3) ^ (urr & 7u)) << 4) + ((cc & 7u) << 1);
                                p.C[static_cast<int64_t>(row) * p.ldc + col] =
                                    *reinterpret_cast<const uint16_t*>(box_ptr + off);
                            }
                        }
                    }
                    __syncwarp();
                }
                }  // 16-bit output
            }
            if (warp == 0 && lane == 0) {
                trace_stamp(p, it, kTrEpiEnd);
                trace_chunk(p, it, 12, kTcStored);
                if (is_split && owner) trace_slot(p, 30, 1);
            }
            preload_if_owner(it + 2);
        }
        if (lane == 0) bulk_wait_group<0>();
        if (warp == 0 && lane == 0) trace_slot(p, 30, 2);
        __syncwarp();
    }

    // ------------------------------------------------------------ teardown
    if (threadIdx.x == 0) trace_slot(p, kTrLaunchSlot, 1);   // roles done
    __syncthreads();
    if constexpr (kCluster > 1) cluster_sync();
    if (threadIdx.x == 0) trace_slot(p, kTrLaunchSlot, 2);   // teardown barrier passed
    if (warp == kMma) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, Cfg::kTmemCols);
        if (lane == 0) trace_slot(p, kTrLaunchSlot, 3);      // tensor memory freed
    }
#endif
}

}  // namespace hg
