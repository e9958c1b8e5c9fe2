// hgemm_api.cu - the C ABI (include/hgemm.h): argument checks, the planner,
// TMA descriptor encoding and the launch of the persistent tcgen05 kernel.
#include <atomic>
#include <chrono>
#include <cstring>
#include <mutex>
#include <string>

#include "hgemm.h"
#include "launch.h"

namespace {

using hg::TcParams;

thread_local std::string t_last_error;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_inject{0};
// hgemm_conv2d: 1 = implicit GEMM (TMA im2col) where the shape allows, 0 =
// always the explicit im2col matrix
std::atomic<bool> g_conv_implicit{true};
std::atomic<unsigned long long*> g_trace{nullptr};

hgemm_status_t cuda_fail(cudaError_t e, const char* where) {
    t_last_error = std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return HGEMM_ERR_CUDA;
}

// ------------------------------------------------------------ device facts
struct DeviceInfo {
    bool probed = false;
    int major = 0, minor = 0, sms = 0;
};

hgemm_status_t device_info(int* dev_out, DeviceInfo* out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        t_last_error = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return HGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (dev < 0 || dev >= 64) return HGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(mu);
    DeviceInfo& d = cache[dev];
    if (!d.probed) {
        if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
            t_last_error = std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e);
            return HGEMM_ERR_UNSUPPORTED_DEVICE;
        }
        d.probed = true;
    }
    *out = d;
    *dev_out = dev;
    if (d.major != 10 || d.minor != 3) {
        t_last_error = "device is compute capability " + std::to_string(d.major) + "." +
                       std::to_string(d.minor) + "; this library runs on 10.3 (sm_103a) only";
        return HGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    return HGEMM_OK;
}

// Element bytes and K per pipeline stage (one 128-byte row of A) of a dtype.
bool valid_dtype(int dt) {
    return dt == HGEMM_F16 || dt == HGEMM_BF16 || dt == HGEMM_TF32 || dt == HGEMM_E4M3 || dt == HGEMM_E5M2;
}
bool is_fp8(hgemm_dtype_t dt) { return dt == HGEMM_E4M3 || dt == HGEMM_E5M2; }
// operand bytes; C is fp32 for tf32, bf16 for fp8, else the operand type
int esize_of(hgemm_dtype_t dt) { return dt == HGEMM_TF32 ? 4 : is_fp8(dt) ? 1 : 2; }
hgemm_dtype_t c_dtype_of(hgemm_dtype_t dt) { return is_fp8(dt) ? HGEMM_BF16 : dt; }
int c_esize_of(hgemm_dtype_t dt) { return esize_of(c_dtype_of(dt)); }
int64_t bk_of(hgemm_dtype_t dt) { return 128 / esize_of(dt); }

// ------------------------------------------------- cuTensorMapEncodeTiled
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

using EncodeIm2colFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const int*, const int*, cuuint32_t, cuuint32_t,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeIm2colFn encode_im2col_fn() {
    static std::once_flag once;
    static EncodeIm2colFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeIm2colFn>(p);
    });
    return fn;
}

// The channels-last activations x (N x H x W x C) of a convolution as an
// im2col-mode tensor map: each copy brings `pixels` consecutive output pixels
// (walked W-fastest inside the bounding box of receptive-field origins,
// lower corner -pad, upper corner pad - (filter extent - 1), stepping by the
// stride) times `chans` channels, in the 128-byte swizzle.
hgemm_status_t encode_im2col(CUtensorMap* m, hgemm_dtype_t dt, const void* x, const hg::ConvShape& cs,
                             uint32_t chans, uint32_t pixels) {
    EncodeIm2colFn fn = encode_im2col_fn();
    if (!fn) {
        t_last_error = "cuTensorMapEncodeIm2col is not available from the driver";
        return HGEMM_ERR_CUDA;
    }
    const int64_t es = esize_of(dt);
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(cs.C), static_cast<cuuint64_t>(cs.W),
                                static_cast<cuuint64_t>(cs.H), static_cast<cuuint64_t>(cs.N)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(cs.C * es), static_cast<cuuint64_t>(cs.W) * cs.C * es,
                                   static_cast<cuuint64_t>(cs.H) * cs.W * cs.C * es};
    const int lower[2] = {-cs.pad, -cs.pad};
    const int upper[2] = {cs.pad - (cs.S - 1), cs.pad - (cs.R - 1)};
    const cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(cs.stride), static_cast<cuuint32_t>(cs.stride), 1};
    const CUtensorMapDataType type = dt == HGEMM_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : dt == HGEMM_TF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(m, type, 4, const_cast<void*>(x), dims, strides, lower, upper, chans, pixels, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_error = "cuTensorMapEncodeIm2col failed with CUresult " + std::to_string(static_cast<int>(r));
        return HGEMM_ERR_CUDA;
    }
    return HGEMM_OK;
}

// A 2-D row-major matrix of `dt` values: `cols` contiguous values per row,
// `ld` values between rows; box = box_cols x box_rows, 128-byte swizzle,
// out-of-range elements read as zero. 128-byte swizzle unless given.
hgemm_status_t encode_2d(CUtensorMap* m, hgemm_dtype_t dt, const void* base, int64_t rows,
                         int64_t cols, int64_t ld, uint32_t box_cols, uint32_t box_rows,
                         CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        t_last_error = "cuTensorMapEncodeTiled is not available from the driver";
        return HGEMM_ERR_CUDA;
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize_of(dt)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType type = dt == HGEMM_TF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : dt == HGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : is_fp8(dt)       ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(m, type,
                    2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_error = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(static_cast<int>(r));
        return HGEMM_ERR_CUDA;
    }
    return HGEMM_OK;
}

// ----------------------------------------------------------------- planner
bool valid_shape_config(int cg, int bn, hgemm_dtype_t dt) {
    (void)dt;
    return (cg == 1 && (bn == 64 || bn == 128 || bn == 256)) || (cg == 2 && (bn == 128 || bn == 224 || bn == 256));
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Relative throughput of one SM running each tile shape on a long K loop
// (1.0 = the pair 256x256 tile), measured on GB300 with L2 flushed, every SM
// busy (whole waves) and the slope of time over K: the pair tile halves each
// SM's B traffic through shared memory, and narrower tiles re-read A for
// fewer columns per MMA.
double shape_efficiency(int cg, int bn) {
    if (cg == 2 && bn == 256) return 1.00;
    if (cg == 2 && bn == 224) return 0.97;
    if (cg == 1 && bn == 256) return 0.845;
    if (cg == 1 && bn == 128) return 0.71;
    if (cg == 2 && bn == 128) return 0.83;
    return 0.385;  // cg 1, bn 64
}

// Measured time constants of the kernel on GB300: the mainloop rate of one SM
// at efficiency 1 (flop/s), the start-up plus last-epilogue time that no tile
// overlaps, and the owners' stream-K fix-up (reading and adding the partners'
// partial sums after the last unit) for a 256-wide tile.
constexpr double kSmFlops = 13.1e12;
constexpr double kFixedSec = 4.5e-6;
constexpr double kStreamKFixupSec = 3.0e-6;
// A CTA pair's extra start-up and hand-over latency per launch, visible on
// short problems (1024^3: single-CTA 128-wide tiles 12.7 us, pair tiles
// 13.9 us; 768^3: 12.1 against 12.5 us).
constexpr double kPairFixedSec = 1.0e-6;
// Epilogue time of a tile: a fixed part (the accumulator hand-over, the
// first TMEM load) plus a part per 64-column chunk that each epilogue warp
// converts and stores (a CTA's 8 warps take its chunks two at a time); a CTA
// pair hands tensor memory back across the pair, 1.75 times as long (1.6
// picked pair tiles for 8192 x 8192 x 64: 36.1 us against 32.3 for 1 x 256,
// interleaved; 4096 x 4096 x 64 and x 128 kept 1 x 256 either way). A tile
// takes at least this long even when its K loop is short: the epilogue of
// one tile overlaps the mainloop of the next, so the slower of the two sets
// the pace. Fitted on GB300 to K = 64 shapes with TMA stores of C (the
// planner's store path for short K loops), per tile and wave: 1x64 1.08 us,
// 1x128 1.18-1.23, 1x256 1.8-2.0, pair 256 1.83-1.98.
// With 16 epilogue warps (32-column chunks, four warps per lane quarter) a
// CTA's warps take its 32-column chunks four at a time, each costing half a
// 64-column chunk, and a pair's hand-over no longer shows: fitted to 16-warp
// tiles on GB300 (interleaved, TMA stores), 8192 x 8192 x 256 pair 256 35.3
// us against 1 x 256 39.1, 4096 x 4096 x 64 1 x 256 13.7 against pair 256
// 14.8, 2048 x 2048 x 1024 1 x 256 14.8 against pair 256 15.4.
constexpr double kEpiTileSec = 0.35e-6;
constexpr double kEpiChunkSec = 0.8e-6;

// The tiles that take 16 epilogue warps: a 16-bit C (fp16, bf16, and the
// bf16 C of fp8) on single 256-wide or pair 224- and 256-wide tiles (whole
// tiles, no K split).
bool epi16_tile(int cg, int bn, hgemm_dtype_t dt) {
    return c_esize_of(dt) == 2 && ((cg == 1 && bn == 256) || (cg == 2 && (bn == 224 || bn == 256)));
}

double tile_seconds(int cg, int bn, int64_t num_kb, int ew) {
    const double mainloop = 2.0 * 128 * bn * (num_kb * hg::kBlockK) / (kSmFlops * shape_efficiency(cg, bn));
    double epilogue;
    if (ew == 16) {
        const int chunks32_per_warp = (bn / 32 + 3) / 4;
        epilogue = kEpiTileSec + kEpiChunkSec * 0.5 * chunks32_per_warp;
    } else {
        const int chunks_per_warp = ((bn / cg + 63) / 64 + 1) / 2;
        epilogue = (kEpiTileSec + kEpiChunkSec * chunks_per_warp) * (cg == 2 ? 1.75 : 1.0);
    }
    return mainloop > epilogue ? mainloop : epilogue;
}

// Stream-K tiles for `tiles` tiles on `clusters` clusters: the leftover
// tiles of a partial last wave plus one full wave (mode 2) or the leftover
// tiles alone (mode 4); all tiles when there are fewer than clusters; 0 when
// the waves come out whole. mode 3 = all.
int64_t stream_k_tiles(int64_t tiles, int64_t clusters, int mode) {
    if (mode == 3) return tiles;
    const int64_t rem = tiles % clusters;
    if (rem == 0) return 0;
    if (tiles < clusters) return tiles;
    return mode == 4 ? rem : rem + clusters;
}

// Estimated seconds of a plan: data-parallel waves, then the stream-K phase
// (each cluster's equal share of K blocks, plus the owners' fix-up: reading
// the partners' partial sums after the last unit).
double schedule_seconds(int cg, int bn, int64_t tiles, int64_t clusters, int64_t num_kb,
                        int64_t sk_tiles, int ew) {
    const double tile_sec = tile_seconds(cg, bn, num_kb, sk_tiles > 0 ? 8 : ew);
    const int64_t dp = tiles - sk_tiles;
    double t = static_cast<double>((dp + clusters - 1) / clusters) * tile_sec;
    if (sk_tiles > 0) {
        const int64_t blocks = (sk_tiles * num_kb + clusters - 1) / clusters;
        t += tile_sec * static_cast<double>(blocks) / static_cast<double>(num_kb) +
             kStreamKFixupSec * bn / 256.0;
    }
    return t + kFixedSec + (cg == 2 ? kPairFixedSec : 0.0);
}

// CTAs per cluster: a CTA pair, or the CTAs splitting a tile's K loop.
int64_t cluster_ctas(const hgemm_plan_t& pl) {
    return static_cast<int64_t>(pl.cta_group) * (pl.split_k > 1 ? pl.split_k : 1);
}

// Fill the schedule fields of `pl` (tiles already set) for `clusters`
// resident clusters.
void schedule_plan(hgemm_plan_t* pl, int64_t clusters, int sk_mode, int64_t num_kb) {
    const int64_t tiles = pl->num_tiles;
    if (clusters < 1) clusters = 1;
    int64_t sk = 0;
    if (sk_mode >= 2) {
        sk = stream_k_tiles(tiles, clusters, sk_mode);
        if (sk == 0 && sk_mode == 2 && tiles % clusters == 0 && tiles >= clusters) sk = clusters;
    }
    // sk_mode 0 (the planner's choice) takes whole tiles. Measured on GB300
    // with the current kernel over 14 shapes from 512^3 to 4096x8192x2048,
    // including skinny 128 x 4096 x 4096 and 256 x 8192 x 8192, the best
    // stream-K schedule never beat the best whole-tile one by more than 1 %
    // and usually lost (by up to 30 %): the fix-up of shared tiles costs more
    // than the balance gains.
    if (sk * num_kb < clusters) sk = 0;  // fewer K blocks than clusters: nothing to share
    if (sk == 0) {
        // Whole waves only: spread them over as few clusters as give the same
        // wave count (less contention for L2 and HBM, same finish time).
        const int64_t waves = (tiles + clusters - 1) / clusters;
        clusters = (tiles + waves - 1) / waves;
    }
    const int64_t total = sk * num_kb;
    pl->dp_tiles = static_cast<int32_t>(tiles - sk);
    pl->sk_tiles = static_cast<int32_t>(sk);
    pl->sk_blocks = static_cast<int32_t>(sk ? total / clusters : 0);
    pl->sk_extra = static_cast<int32_t>(sk ? total % clusters : 0);
    pl->grid_ctas = static_cast<int32_t>(clusters * cluster_ctas(*pl));
    pl->num_kb = static_cast<int32_t>(num_kb);
}

// Bytes of fp32 partial sums (one block per CTA) and their flags.
int64_t partial_bytes(const hgemm_plan_t& pl) {
    if (pl.sk_tiles == 0) return 0;
    return static_cast<int64_t>(pl.grid_ctas) * hg::kEpiQuarters * hg::kEpiBoxRows * pl.block_n * 4;
}

int64_t flag_bytes(const hgemm_plan_t& pl) {
    if (pl.sk_tiles == 0) return 0;
    return static_cast<int64_t>(pl.grid_ctas) * hg::kEpiQuarters * 2 * 8;
}

int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

// Workspace layout: [A repack][B repack][partials][flags], each 256-aligned.
struct WorkspaceLayout {
    int64_t off_a, off_b, off_part, off_flags, total;
};

// Rows of an operand copy: padded to 128 bytes, so that every row of a TMA
// box starts on a 128-byte line. A pitch that is an odd multiple of 16 bytes
// costs the GEMM's loads 10-20 % (1000 x 4096 x K bf16, A read in place:
// K = 4104 33.6 us, 4112 29.3, 4128 28.6, 4160 28.3).
int64_t pitch128(int64_t cols, int esize) {
    const int64_t per = 128 / esize;
    return (cols + per - 1) / per * per;
}

// A's rows an odd multiple of 16 bytes apart: TMA can address them, but
// with 224-wide pair tiles, whose stages already ask for about as many bytes
// per cycle as the SM's loads deliver, the K-major A loads then run 10-20 %
// slower (every other 128-byte box row straddles two 32-byte sectors at both
// ends). The copy into 128-byte rows pays for itself once N is large enough.
// Measured on GB300 (bf16, L2 flushed, copied vs in place, same box):
// 4096 x 4096 x 4104 92.0 vs 98.9 us, 1000 x 4095 x 4104 52.3 vs 54.5,
// 1000 x 4096 x 4104 33.8 vs 34.5; 2048 x 2048 x 2056 27.1 vs 25.5 (a loss);
// with 256-wide tiles no cost to remove (8192 x 8192 x 8200 in place 595 us,
// as fast as 8192^3; copied 614). B (MN-major boxes) showed no such cost:
// 4096 x 4104 x 4096 83.6 us in place, 89.5 copied.
bool a_pitch_slow(int64_t N, int64_t K, int esize, int block_n, int split) {
    return ((K * esize) & 31) == 16 && N >= 3584 && block_n == 224 && split <= 1;
}

WorkspaceLayout workspace_layout(const hgemm_plan_t& pl, int64_t M, int64_t N, int64_t K, int esize) {
    WorkspaceLayout w{};
    const int64_t lda = pitch128(K, esize), ldb = pitch128(N, esize);
    int64_t off = 0;
    w.off_a = off;
    off += pl.repack_a ? align256(esize * M * lda) : 0;
    w.off_b = off;
    off += pl.repack_b ? align256(esize * K * ldb) : 0;
    w.off_part = off;
    off += align256(partial_bytes(pl));
    w.off_flags = off;
    off += align256(flag_bytes(pl));
    w.total = off;
    return w;
}

// Pick (cta_group, block_n) minimising the estimated time: whole waves of
// tiles over the resident clusters plus the (K-split) tail, each tile costing
// its padded area at the shape's efficiency, plus the fixed costs above. A
// problem with a single 128-row tile row keeps one CTA per tile (a pair would
// compute an empty half).
// A stage costs the same time for every dtype (128 bytes of K of A per row:
// 64 fp16/bf16 values, or 32 tf32 values at half the tensor rate).
double estimate_seconds(int64_t M, int64_t N, int64_t K, int cg, int bn, int64_t clusters, hgemm_dtype_t dt) {
    const int64_t kb = cdiv(K, bk_of(dt));
    const int64_t tiles = cdiv(M, 128 * cg) * cdiv(N, bn);
    hgemm_plan_t pl{};
    pl.cta_group = cg;
    pl.block_n = bn;
    pl.multicast = 1;
    pl.split_k = 1;
    pl.num_tiles = static_cast<int32_t>(tiles);
    schedule_plan(&pl, clusters, 0, kb);
    return schedule_seconds(cg, bn, tiles, pl.grid_ctas / cg, kb, pl.sk_tiles, epi16_tile(cg, bn, dt) ? 16 : 8);
}

void choose_shape(int64_t M, int64_t N, int64_t K, hgemm_dtype_t dt, int sms, int max_clusters, int* cg_out,
                  int* bn_out) {
    static const int cand[6][2] = {{2, 256}, {2, 224}, {1, 256}, {1, 128}, {2, 128}, {1, 64}};
    double best = 1e300;
    int bcg = 2, bbn = 256;
    for (const auto& c : cand) {
        const int cg = c[0], bn = c[1];
        if (cg == 2 && M <= 128) continue;
        if (!valid_shape_config(cg, bn, dt)) continue;
        // 8-bit B is read MN-major in 128-column atoms, which a CTA's 112
        // columns of a 224-wide pair tile leave part-full: E4M3 4096^3 runs
        // 51.6 us with 224-wide tiles on all SMs against 49.4 us with 256-wide
        // ones on 128 (the part-full atom loaded whole: 59.4 us; 8192^3 then
        // 2982 against 3649 TFLOP/s). The planner leaves it out for fp8 (a
        // config can still ask for it).
        if (is_fp8(dt) && cg == 2 && bn == 224) continue;
        // A single tile row on a long K loop is HBM-bound, which the time
        // model above (compute-bound tiles) does not see: the narrowest tile
        // that keeps every tile in one wave spreads B's stream over the most
        // SMs (128 x 4096 x 4096: 64-wide 23.1 us, 128-wide 24.6 us).
        if (M <= 128 && K >= 16 * bk_of(dt)) {
            const int skinny_bn = cdiv(N, 64) <= sms ? 64 : 128;
            if (cg != 1 || bn != skinny_bn) continue;
        }
        int64_t clusters = sms / cg;
        if (max_clusters > 0 && max_clusters < clusters) clusters = max_clusters;
        if (clusters <= 0) continue;
        const double t = estimate_seconds(M, N, K, cg, bn, clusters, dt);
        if (t < best * 0.999) {
            best = t;
            bcg = cg;
            bbn = bn;
        }
    }
    *cg_out = bcg;
    *bn_out = bbn;
}

// The planner's K split: clusters of `s` single CTAs on 128-wide tiles when
// the K loop is long (at least 64 blocks, 16 per CTA) and the tiles, s CTAs
// each, still fit on the SMs; the widest such s of 4 and 2. Measured on GB300
// (bf16, L2 flushed, interleaved, against the planner's whole tiles):
// 128 x 4096 x 14336 57.1 -> 40.7 us (split 4), 128 x 2048 x 8192 35.8 ->
// 25.9 (4), 1024 x 1024 x 8192 34.4 -> 29.2 (2), 128 x 8192 x 8192 45.1 ->
// 41.4 (2), 16 and 64 x 8192 x 8192 -10 % (2). Once the split's exchange
// sent whole row slices, K = 4096 gained too: 128 x 4096 x 4096 23.0 ->
// 20.7 (4), 256 x 4096 x 4096 23.1 -> 20.8 (2), 512 x 2048 x 4096 23.1 ->
// 20.9 (2), 1024 x 1024 x 4096 23.1 -> 21.0 (2), 64 x 8192 x 4096 24.1 ->
// 23.3 (2); K = 2048 still loses (128 x 8192 x 2048: 16.8 -> 18.6). 256-wide
// split tiles measured slower than 128-wide ones on every shape tried.
int auto_split(int64_t M, int64_t N, int64_t K, hgemm_dtype_t dt, int sms) {
    if (esize_of(dt) != 2) return 1;
    const int64_t num_kb = cdiv(K, bk_of(dt));
    if (num_kb < 64) return 1;
    const int64_t tiles = cdiv(M, 128) * cdiv(N, 128);
    for (int s : {4, 2})
        if (tiles * s <= sms && num_kb / s >= 16) return s;
    return 1;
}

hgemm_status_t make_plan(int64_t M, int64_t N, int64_t K, hgemm_dtype_t dt, const hgemm_config_t* cfg, int sms,
                         bool a_unaligned, bool b_unaligned, bool c_unaligned, hgemm_plan_t* pl,
                         bool allow_auto_split = true, bool a_copy_ok = true) {
    std::memset(pl, 0, sizeof(*pl));
    hgemm_config_t c{};
    if (cfg) c = *cfg;
    if (c.group_m < 0 || c.max_clusters < 0 || c.store_mode < 0 || c.store_mode > 5 || c.stream_k < 0 ||
        c.stream_k > 4 || c.split_k < 0 || c.split_k > 8) {
        t_last_error = "negative or unknown config field";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (c.multicast != 0 && c.multicast != 1) {
        // reserved: no operand is multicast across the CTAs of a cluster
        t_last_error = "multicast is reserved: 0 or 1 (no operand multicast is built)";
        return HGEMM_ERR_INVALID_ARG;
    }
    int cg = c.cta_group, bn = c.block_n;
    int split = c.split_k > 1 ? c.split_k : 1;
    if (c.split_k == 0 && allow_auto_split && cg == 0 && bn == 0 && c.stream_k <= 1 &&
        c.max_clusters == 0) {
        split = auto_split(M, N, K, dt, sms);
        if (split > 1) bn = 128;
    }
    if (split > 1) {
        // K split across a cluster: single CTAs, a tile of 128 or 256 columns
        if (cg == 0) cg = 1;
        if (bn == 0) bn = 256;
    }
    if (cg == 0 || bn == 0) {
        int acg, abn;
        choose_shape(M, N, K, dt, sms, c.max_clusters, &acg, &abn);
        if (cg == 0 && bn == 0) {
            cg = acg;
            bn = abn;
        } else if (cg == 0) {
            cg = (bn >= 128) ? acg : 1;
        } else {
            bn = (cg == 2 && abn < 128) ? 128 : abn;
        }
    }
    if (!valid_shape_config(cg, bn, dt)) {
        t_last_error = "unsupported (cta_group, block_n) pair";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (split > 1 && !((split == 2 || split == 4 || split == 8) && cg == 1 && (bn == 128 || bn == 256) &&
                       bn / split >= 32 && esize_of(dt) == 2 && c.stream_k <= 1)) {
        t_last_error = "split_k needs 2, 4 or 8 with cta_group 1, block_n 128 or 256 (at least 32 columns per "
                       "CTA), a 16-bit dtype and no stream-K";
        return HGEMM_ERR_INVALID_ARG;
    }
    pl->cta_group = cg;
    pl->multicast = 1;
    pl->split_k = split;
    pl->block_m = 128 * cg;
    pl->block_n = bn;
    pl->block_k = static_cast<int32_t>(bk_of(dt));
    pl->stages = hg::tc_stages(cg, bn, esize_of(dt), split);
    pl->smem_bytes = hg::tc_smem_bytes(cg, bn, esize_of(dt), split);
    pl->tmem_cols = hg::tc_tmem_cols(cg, bn);
    pl->tiles_m = static_cast<int32_t>(cdiv(M, pl->block_m));
    pl->tiles_n = static_cast<int32_t>(cdiv(N, bn));
    pl->num_tiles = pl->tiles_m * pl->tiles_n;
    // Raster groups of 8 tile rows keep the A and B panels of concurrent tiles
    // in L2 when the operands do not fit there (8192^3: 256 MiB); when they
    // do (up to ~96 MiB, L2 is 129 MB over two dies) groups of 2 measured
    // 1-2 % faster (4096^3 bf16/fp16, 8192x4096x4096: 28 of 30 interleaved
    // pairs).
    const double operand_bytes = static_cast<double>(esize_of(dt)) * (static_cast<double>(M) * K + static_cast<double>(K) * N);
    const int32_t gm_default = operand_bytes <= 96.0 * 1024 * 1024 ? 2 : 8;
    pl->group_m = c.group_m > 0 ? c.group_m
                                : (pl->tiles_m < gm_default ? (pl->tiles_m > 0 ? pl->tiles_m : 1) : gm_default);
    int64_t clusters = sms / cluster_ctas(*pl);
    if (c.max_clusters > 0 && c.max_clusters < clusters) clusters = c.max_clusters;
    if (split > 1 && pl->num_tiles > clusters) {
        // the K split's reduction reuses each CTA's stage ring: one tile per cluster
        t_last_error = "split_k needs one cluster per tile: " + std::to_string(pl->num_tiles) + " tiles, " +
                       std::to_string(clusters) + " clusters";
        return HGEMM_ERR_INVALID_ARG;
    }
    schedule_plan(pl, clusters, c.stream_k, cdiv(K, bk_of(dt)));
    pl->repack_a = (a_unaligned || (a_copy_ok && a_pitch_slow(N, K, esize_of(dt), bn, split))) ? 1 : 0;
    pl->repack_b = b_unaligned ? 1 : 0;
    // Default for an aligned C: rows written back from the swizzled staging box
    // with 16-byte vector stores (4). They go out through the load/store path,
    // so they do not queue in the SM's TMA unit ahead of the next tile's
    // operand loads, as TMA tensor stores (1) do: measured 0.5-1 % faster at
    // 4096^3 to 16384x14336x4096, in 33 of 36 interleaved pairs. A short K
    // loop (at most 8 blocks) leaves the epilogue setting the pace, and there
    // TMA stores are faster: 4096x4096x64 19.1 -> 16.6 us, 8192x8192x256
    // 53.2 -> 46.7, 16384x16384x64 156 -> 105. At K = 1024 the two modes
    // tie (4096x4096x1024: 30.8 us each). So is a single wave of tiles,
    // whose last epilogue nothing overlaps: 2048^3 22.9 -> 21.2 us,
    // 2048x2048x1024 15.2 -> 14.9 (3072^3, 1.3 waves: a tie).
    const int64_t num_kb_plan = cdiv(K, bk_of(dt));
    const bool one_wave = static_cast<int64_t>(pl->num_tiles) * cluster_ctas(*pl) <= pl->grid_ctas;
    // A C whose rows are not 16-byte aligned: 16-bit C takes realigned
    // 16-byte stores with element stores at the ragged ends (5); fp32 C (tf32)
    // plain element stores (2). Measured against element stores: 1000 x 4095
    // x 4104 53.2 against 55.4 us, 3000 x 1001 x 2048 32.8 against 34.6.
    const bool c16 = c_esize_of(dt) == 2;
    pl->store_mode = (c.store_mode != 0)   ? c.store_mode
                     : c_unaligned           ? (c16 ? 5 : 2)
                     : (num_kb_plan <= 8 || one_wave) ? 1
                                                      : 4;
    if (pl->store_mode == 5 && !c16) {
        t_last_error = "store_mode 5 is for 16-bit C";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (c_unaligned && pl->store_mode != 2 && pl->store_mode != 5) {
        t_last_error = "vector and TMA stores need a 16-byte aligned C with a 16-byte row pitch";
        return HGEMM_ERR_INVALID_ARG;
    }
    // Epilogue warps. A short K loop on single 256-wide tiles leaves the
    // epilogue setting the pace, and each warp's chain of TMEM load,
    // conversion, staging and store is latency-bound: 16 warps on 32-column
    // chunks keep twice the chunks in flight.
    const bool epi16_ok = epi16_tile(cg, bn, dt) && split == 1 && pl->sk_tiles == 0;
    if (c.epi_warps != 0 && c.epi_warps != 8 && !(c.epi_warps == 16 && epi16_ok)) {
        t_last_error = "epi_warps: 0, 8, or 16 with a 16-bit C on single 256-wide or pair 224- and 256-wide "
                       "tiles, no K split and no stream-K";
        return HGEMM_ERR_INVALID_ARG;
    }
    pl->epi_warps = c.epi_warps != 0 ? c.epi_warps : epi16_ok ? 16 : 8;
    const int mc = split > 1 ? split : 1;
    const bool compiled =
        dt == HGEMM_BF16   ? hg::tc_instance_exists_bf16(cg, bn, mc, pl->epi_warps)
        : dt == HGEMM_F16  ? hg::tc_instance_exists_f16(cg, bn, mc, pl->epi_warps)
        : dt == HGEMM_TF32 ? hg::tc_instance_exists_tf32(cg, bn, mc, pl->epi_warps)
                           : hg::tc_instance_exists_fp8(static_cast<int>(dt), cg, bn, mc, pl->epi_warps);
    if (!compiled) {
        t_last_error = "no kernel is compiled for cta_group " + std::to_string(cg) + ", block_n " +
                       std::to_string(bn) + ", split " + std::to_string(mc) + ", " +
                       std::to_string(pl->epi_warps) + " epilogue warps";
        return HGEMM_ERR_INVALID_ARG;
    }
    pl->workspace_bytes = workspace_layout(*pl, M, N, K, esize_of(dt)).total;
    return HGEMM_OK;
}

// --------------------------------------------------------------- workspace
// One stream-ordered pool per device, owned by the library, that keeps up to
// 256 MiB cached between calls so steady-state calls do not go to the driver.
hgemm_status_t pool_for_device(int dev, cudaMemPool_t* out) {
    static std::mutex mu;
    static cudaMemPool_t pools[64] = {};
    if (dev < 0 || dev >= 64) return HGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(mu);
    if (!pools[dev]) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        cudaError_t e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
        uint64_t keep = uint64_t{256} << 20;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return cuda_fail(e, "cudaMemPoolSetAttribute");
        }
        pools[dev] = pool;
    }
    *out = pools[dev];
    return HGEMM_OK;
}

// A number unique to each launch (split-K parts mark their partials with it).
unsigned long long next_epoch() {
    static std::atomic<unsigned long long> counter{
        (static_cast<unsigned long long>(
             std::chrono::steady_clock::now().time_since_epoch().count()) << 20) | (1ull << 63)};
    return counter.fetch_add(1, std::memory_order_relaxed);
}

bool misaligned16(const void* p, int64_t cols, int esize) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) != 0 || ((cols * esize) & 15) != 0;
}


bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

hgemm_status_t check_args(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                          hgemm_dtype_t dtype) {
    const int64_t kMax = 2147483647LL;
    if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax) {
        t_last_error = "dimensions must be in [0, 2^31 - 1]";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (!valid_dtype(dtype)) {
        t_last_error = "unknown dtype";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (M == 0 || N == 0) return HGEMM_OK;
    const int es = esize_of(dtype), ces = c_esize_of(dtype);
    const uintptr_t amask = static_cast<uintptr_t>(es - 1), cmask = static_cast<uintptr_t>(ces - 1);
    if (!C || (K > 0 && (!A || !B))) {
        t_last_error = "null pointer for a non-empty operand";
        return HGEMM_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(C) & cmask) ||
        (K > 0 && ((reinterpret_cast<uintptr_t>(A) & amask) || (reinterpret_cast<uintptr_t>(B) & amask)))) {
        t_last_error = "operands must be aligned to their element size";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (K > 0 && (overlaps(C, ces * M * N, A, es * M * K) || overlaps(C, ces * M * N, B, es * K * N))) {
        t_last_error = "C overlaps A or B";
        return HGEMM_ERR_INVALID_ARG;
    }
    return HGEMM_OK;
}

// Resident clusters of the kernel instance a plan launches, on the current
// device (0 if the query fails).
int resident_clusters(hgemm_dtype_t dtype, const hgemm_plan_t& q) {
    const int qm = q.split_k > 1 ? q.split_k : 1;
    const int ew = q.epi_warps == 16 ? 16 : 8;
    return dtype == HGEMM_BF16   ? hg::max_active_clusters_bf16(q.cta_group, q.block_n, qm, ew)
           : dtype == HGEMM_TF32 ? hg::max_active_clusters_tf32(q.cta_group, q.block_n, qm, ew)
           : is_fp8(dtype)       ? hg::max_active_clusters_fp8(static_cast<int>(dtype), q.cta_group, q.block_n, qm, ew)
                                 : hg::max_active_clusters_f16(q.cta_group, q.block_n, qm, ew);
}

// The planner's K split needs one resident cluster per tile. Where fewer
// clusters of that size fit on the current device (on a 152-SM GB300, 32
// clusters of 4 and 15 of 8), take half the split on the same tiles, then
// whole tiles. A split asked for in `cfg` is kept (the launch then fails
// with a message). *resident receives the resident clusters of the final plan.
hgemm_status_t fit_split_to_device(int64_t M, int64_t N, int64_t K, hgemm_dtype_t dtype, const hgemm_config_t* cfg,
                                   int sms, bool a_bad, bool b_bad, bool c_bad, hgemm_plan_t* pl, int* resident,
                                   bool a_copy_ok = true) {
    *resident = resident_clusters(dtype, *pl);
    while (pl->split_k > 1 && !(cfg && cfg->split_k > 1) && *resident > 0 && *resident < pl->num_tiles) {
        hgemm_config_t smaller{};
        if (cfg) smaller = *cfg;
        smaller.split_k = pl->split_k / 2 > 1 ? pl->split_k / 2 : 1;
        if (smaller.split_k > 1) {
            smaller.cta_group = 1;
            smaller.block_n = pl->block_n;
        }
        hgemm_status_t st = make_plan(M, N, K, dtype, &smaller, sms, a_bad, b_bad, c_bad, pl, false, a_copy_ok);
        if (st != HGEMM_OK) return st;
        *resident = resident_clusters(dtype, *pl);
    }
    return HGEMM_OK;
}

// `scratch` (nullptr: none) is caller-provided device memory of `scratch_bytes`
// used instead of the stream-ordered allocator for the repack workspace.
// `a_scale` / `b_scale` (fp8 only; nullptr = 1) are the per-channel factors.
// `lda_in` > 0: A's rows are lda_in elements apart (a 16-byte pitch, 16-byte
// aligned base: the library's own im2col matrix), so A needs no repack.
// `conv` (implicit-GEMM convolution): A is the activations x behind an
// im2col-mode tensor map; hgemm_conv2d has checked the operands.
// `bs_block` (32 or 64; 0 = none): the block-scaled fp8 GEMM, a_scale and
// b_scale being the fp32 grids of one factor per bs_block x bs_block
// sub-block of A and of B (hgemm_fp8_blockscaled has checked them).
hgemm_status_t run(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                   hgemm_dtype_t dtype, const hgemm_config_t* cfg, cudaStream_t stream,
                   void* scratch = nullptr, size_t scratch_bytes = 0, const float* a_scale = nullptr,
                   const float* b_scale = nullptr, int64_t lda_in = 0, const hg::ConvShape* conv = nullptr,
                   int bs_block = 0) {
    t_last_error.clear();
    hgemm_status_t st = conv ? HGEMM_OK : check_args(A, B, C, M, N, K, dtype);
    if (st != HGEMM_OK || M == 0 || N == 0) return st;
    int dev = 0;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != HGEMM_OK) return st;
    cudaError_t e;
    const int es = esize_of(dtype), ces = c_esize_of(dtype);
    const int64_t bk = bk_of(dtype);
    if (K == 0) {
        // zero bits are +0.0 in every dtype; the fill counts 16-bit words
        if ((e = hg::launch_zero(static_cast<uint16_t*>(C), M * N * (ces / 2), stream)) != cudaSuccess)
            return cuda_fail(e, "zero fill");
        return HGEMM_OK;
    }

    hgemm_plan_t pl;
    // A given as the library's im2col matrix (lda_in) or read by im2col copies is not copied
    const bool a_copy_ok = !(lda_in > 0 || conv);
    const bool a_bad = a_copy_ok && misaligned16(A, K, es);
    const bool b_bad = misaligned16(B, N, es), c_bad = misaligned16(C, N, ces);
    hgemm_config_t bs_cfg{};
    if (bs_block) {
        // block-scaled fp8: 128-column tiles, whole tiles; a CTA pair per
        // 256-row tile unless the problem has a single 128-row tile row
        if (cfg) bs_cfg = *cfg;   // fields checked by hgemm_fp8_blockscaled_ex
        if (bs_cfg.cta_group == 0) bs_cfg.cta_group = M > 128 ? 2 : 1;
        bs_cfg.block_n = 128;
        bs_cfg.split_k = 1;
        bs_cfg.stream_k = 1;
        cfg = &bs_cfg;
    }
    if ((st = make_plan(M, N, K, dtype, cfg, info.sms, a_bad, b_bad, c_bad, &pl, !conv && !bs_block, a_copy_ok)) !=
        HGEMM_OK)
        return st;
    if (bs_block) {
        pl.stages = hg::fp8bs_stages(pl.cta_group);
        pl.smem_bytes = hg::fp8bs_smem_bytes(pl.cta_group);
        pl.tmem_cols = hg::fp8bs_tmem_cols();
    }
    if (conv && pl.split_k > 1) {
        t_last_error = "split_k is not built for the convolution";
        return HGEMM_ERR_INVALID_ARG;
    }

    // Resident clusters bound the persistent grid: a K split that does not
    // fit shrinks, and the schedule is re-planned if fewer clusters fit than
    // the planner assumed. The kernel's cluster multiplier is the CTAs
    // splitting K.
    int resident = 0;
    if (bs_block)
        resident = hg::max_active_clusters_fp8bs(static_cast<int>(dtype), pl.cta_group, bs_block);
    else if ((st = fit_split_to_device(M, N, K, dtype, cfg, info.sms, a_bad, b_bad, c_bad, &pl, &resident,
                                       a_copy_ok)) != HGEMM_OK)
        return st;
    const int cg = pl.cta_group, bn = pl.block_n, mc = pl.split_k > 1 ? pl.split_k : 1;
    const int64_t num_kb = cdiv(K, bk);
    if (resident > 0 && resident < pl.grid_ctas / (cg * mc)) {
        if (pl.split_k > 1) {
            t_last_error = "split_k needs one cluster per tile: " + std::to_string(pl.num_tiles) + " tiles, " +
                           std::to_string(resident) + " clusters of " + std::to_string(mc) + " fit";
            return HGEMM_ERR_INVALID_ARG;
        }
        schedule_plan(&pl, resident, cfg ? cfg->stream_k : 0, num_kb);
        pl.workspace_bytes = workspace_layout(pl, M, N, K, es).total;
        if (pl.epi_warps == 16 && pl.sk_tiles > 0) {
            // stream-K units take the 8-warp epilogue
            if (cfg && cfg->epi_warps == 16) {
                t_last_error = "epi_warps 16 needs whole tiles, and stream-K remains on the resident clusters";
                return HGEMM_ERR_INVALID_ARG;
            }
            pl.epi_warps = 8;
        }
    }
    const int clusters = pl.grid_ctas / (cg * mc);

    // A copy of A made only for speed (a_pitch_slow) is dropped when it would
    // not fit in a caller's fixed scratch.
    if (scratch && pl.repack_a && !a_bad &&
        static_cast<size_t>(workspace_layout(pl, M, N, K, es).total) > scratch_bytes) {
        pl.repack_a = 0;
        pl.workspace_bytes = workspace_layout(pl, M, N, K, es).total;
    }
    // Workspace: 128-byte-pitched copies of operands TMA cannot address, and
    // the fp32 partial sums of a K-split tail.
    const WorkspaceLayout wl = workspace_layout(pl, M, N, K, es);
    const int64_t lda = lda_in > 0 ? lda_in : pl.repack_a ? pitch128(K, es) : K;
    const int64_t ldb = pl.repack_b ? pitch128(N, es) : N;
    void* work = nullptr;
    const void* a_use = A;
    const void* b_use = B;
    if (wl.total > 0) {
        const size_t need = static_cast<size_t>(wl.total);
        if (scratch) {
            if (need > scratch_bytes) {
                t_last_error = "this shape needs " + std::to_string(need) +
                               " bytes of workspace; the scratch holds " +
                               std::to_string(scratch_bytes);
                return HGEMM_ERR_INVALID_ARG;
            }
            work = scratch;
        } else {
            cudaMemPool_t pool = nullptr;
            if ((st = pool_for_device(dev, &pool)) != HGEMM_OK) return st;
            if ((e = cudaMallocFromPoolAsync(&work, need, pool, stream)) != cudaSuccess) {
                cuda_fail(e, "cudaMallocFromPoolAsync (workspace)");
                return HGEMM_ERR_ALLOC;
            }
        }
        uint8_t* w8 = static_cast<uint8_t*>(work);
        if (pl.repack_a || pl.repack_b) {
            // both copies in one launch
            hg::RepackJob ja{}, jb{};
            if (pl.repack_a) {
                ja = {static_cast<const uint8_t*>(A), M, es * K, w8 + wl.off_a, es * lda};
                a_use = w8 + wl.off_a;
            }
            if (pl.repack_b) {
                jb = {static_cast<const uint8_t*>(B), K, es * N, w8 + wl.off_b, es * ldb};
                b_use = w8 + wl.off_b;
            }
            if ((e = hg::launch_repack(ja, jb, stream)) != cudaSuccess) {
                if (work != scratch) cudaFreeAsync(work, stream);
                return cuda_fail(e, "repack");
            }
        }
    }

    CUtensorMap ta, tb, tb2, tc, tc32;
    std::memset(&tb2, 0, sizeof(tb2));
    std::memset(&tc, 0, sizeof(tc));
    std::memset(&tc32, 0, sizeof(tc32));
    // A CTA's B columns (bn / cg) in 128-byte swizzle atoms; a part-full
    // last atom is loaded with a box of its used columns only.
    const int64_t atom_cols = 128 / es, bn_cta = bn / cg;
    const int64_t b_last = bn_cta - ((bn_cta + atom_cols - 1) / atom_cols - 1) * atom_cols;
    // A boxes: 128 rows x one 128-byte row of K; B boxes: bk k-rows x one
    // 128-byte swizzle atom of columns (tf32 B in the 32-byte-atom swizzle,
    // which is how kind::tf32 reads an MN-major operand); C boxes: 32 rows x
    // 128 bytes.
    const uint32_t ubk = static_cast<uint32_t>(bk);
    if ((st = conv ? encode_im2col(&ta, dtype, A, *conv, ubk, hg::kBlockMCta)
                   : encode_2d(&ta, dtype, a_use, M, K, lda, ubk, hg::kBlockMCta)) != HGEMM_OK ||
        (st = encode_2d(&tb, dtype, b_use, K, N, ldb, ubk, ubk,
                        dtype == HGEMM_TF32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B)) !=
            HGEMM_OK ||
        (b_last != atom_cols &&
         (st = encode_2d(&tb2, dtype, b_use, K, N, ldb, static_cast<uint32_t>(b_last), ubk,
                         dtype == HGEMM_TF32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B)) !=
             HGEMM_OK) ||
        (pl.store_mode == 1 && !bs_block &&
         (st = encode_2d(&tc, c_dtype_of(dtype), C, M, N, N, static_cast<uint32_t>(128 / ces), hg::kEpiBoxRows)) !=
             HGEMM_OK) ||
        // the 32-column last chunk of a 16-bit C, or every chunk with 16
        // epilogue warps (fp32 C leaves in 32-column boxes throughout, through tc)
        (pl.store_mode == 1 && !bs_block && (bn % 64 != 0 || pl.epi_warps == 16) && ces == 2 &&
         (st = encode_2d(&tc32, c_dtype_of(dtype), C, M, N, N, 32, hg::kEpiBoxRows, CU_TENSOR_MAP_SWIZZLE_64B)) !=
             HGEMM_OK)) {
        if (work && work != scratch) cudaFreeAsync(work, stream);
        return st;
    }

    if (bs_block) {
        hg::Fp8bsParams q{};
        q.M = static_cast<int32_t>(M);
        q.N = static_cast<int32_t>(N);
        q.K = static_cast<int32_t>(K);
        q.tiles_m = pl.tiles_m;
        q.tiles_n = pl.tiles_n;
        q.num_tiles = pl.num_tiles;
        q.group_m = pl.group_m;
        q.num_kb = static_cast<int32_t>(cdiv(K, bk));
        q.num_sb = static_cast<int32_t>(cdiv(K, bs_block));
        q.sa_rows = static_cast<int32_t>(cdiv(M, bs_block));
        q.sb_cols = static_cast<int32_t>(cdiv(N, bs_block));
        // kind::f8f6f4: D fp32, A and B format (0 E4M3, 1 E5M2), A K-major,
        // B MN-major, N = 128, M = 128 per CTA
        const uint32_t f8 = dtype == HGEMM_E5M2 ? 1u : 0u;
        q.idesc = (1u << 4) | (f8 << 7) | (f8 << 10) | (1u << 16) | (static_cast<uint32_t>(bn >> 3) << 17) |
                  (static_cast<uint32_t>((128 * cg) >> 4) << 24);
        q.a_scale = a_scale;
        q.b_scale = b_scale;
        q.C = static_cast<uint16_t*>(C);
        q.ldc = N;
        q.c_vec = c_bad ? 0 : 1;
        q.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
        q.sched.num_tiles = pl.num_tiles;
        q.sched.dp_tiles = pl.dp_tiles;
        q.sched.num_kb = q.num_kb;
        q.sched.clusters = clusters;
        q.sched.sk_base = 0;
        q.sched.sk_extra = 0;
        q.trace = g_trace.load(std::memory_order_relaxed);
        q.pdl = (pl.repack_a || pl.repack_b) ? 1 : 0;
        if ((e = hg::status_word_ptr(&q.status)) != cudaSuccess) {
            if (work && work != scratch) cudaFreeAsync(work, stream);
            return cuda_fail(e, "status word");
        }
        e = hg::launch_fp8bs(static_cast<int>(dtype), cg, bs_block, ta, tb, tb2, q, clusters, stream);
        if (work && work != scratch) cudaFreeAsync(work, stream);
        if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
        return HGEMM_OK;
    }

    TcParams p{};
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.tiles_m = pl.tiles_m;
    p.tiles_n = pl.tiles_n;
    p.num_tiles = pl.num_tiles;
    p.group_m = pl.group_m;
    p.num_kb = static_cast<int32_t>(cdiv(K, bk));
    // operand format codes: kind::f16 0 f16, 1 bf16; kind::tf32 2; kind::f8f6f4
    // 0 E4M3, 1 E5M2
    const uint32_t fmt = dtype == HGEMM_BF16   ? 1u
                         : dtype == HGEMM_TF32 ? 2u
                         : dtype == HGEMM_E5M2 ? 1u
                                               : 0u;
    // Instruction descriptor, kind::f16 / kind::tf32: D fp32 (bits 4-5 = 1),
    // A and B format (bits 7-9, 10-12: 0 f16, 1 bf16, 2 tf32), A K-major
    // (bit 15 = 0), B MN-major (bit 16 = 1), N >> 3 (bits 17-22), M >> 4
    // (bits 24-28).
    p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (0u << 15) | (1u << 16) |
              (static_cast<uint32_t>(bn >> 3) << 17) | (static_cast<uint32_t>((128 * cg) >> 4) << 24);
    p.store_mode = pl.store_mode;
    p.C = static_cast<uint16_t*>(C);
    p.a_scale = a_scale;
    p.b_scale = b_scale;
    if (conv) {
        p.im2col = 1;
        p.cv_cblocks = static_cast<int32_t>(conv->C / bk);
        p.cv_S = conv->S;
        p.cv_P = conv->P;
        p.cv_Q = conv->Q;
        p.cv_stride = conv->stride;
        p.cv_pad = conv->pad;
    }
    p.ldc = N;
    p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    p.sched.num_tiles = pl.num_tiles;
    p.sched.dp_tiles = pl.dp_tiles;
    p.sched.num_kb = p.num_kb;
    p.sched.clusters = clusters;
    p.sched.sk_base = pl.sk_blocks;
    p.sched.sk_extra = pl.sk_extra;
    p.partials = pl.sk_tiles > 0 ? reinterpret_cast<float*>(static_cast<uint8_t*>(work) + wl.off_part) : nullptr;
    p.flags = pl.sk_tiles > 0
                  ? reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(work) + wl.off_flags)
                  : nullptr;
    p.epoch = next_epoch();
    bool cleared_flags = false;
    if (p.flags) {
        // A graph replays this launch with the same epoch, so flags left by
        // the previous replay would already read as published: a captured
        // launch clears its flags first (an eager launch's epoch is new).
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cleared_flags = true;   // conservatively: a memset may sit between the copy and the GEMM
        if ((e = cudaStreamIsCapturing(stream, &cs)) != cudaSuccess ||
            (cs == cudaStreamCaptureStatusActive &&
             (e = cudaMemsetAsync(p.flags, 0, static_cast<size_t>(flag_bytes(pl)), stream)) != cudaSuccess)) {
            if (work && work != scratch) cudaFreeAsync(work, stream);
            return cuda_fail(e, "stream-K flags");
        }
    }
    p.inject = g_inject.load(std::memory_order_relaxed);
    p.trace = g_trace.load(std::memory_order_relaxed);
    // right after an operand copy on the same stream (no flag clearing in
    // between), the GEMM launches as its programmatic dependent: its launch
    // and set-up overlap the copy's tail
    p.pdl = ((pl.repack_a || pl.repack_b) && !cleared_flags) ? 1 : 0;
    if ((e = hg::status_word_ptr(&p.status)) != cudaSuccess) {
        if (work && work != scratch) cudaFreeAsync(work, stream);
        return cuda_fail(e, "status word");
    }

    const int ew = pl.epi_warps == 16 ? 16 : 8;
    e = dtype == HGEMM_BF16   ? hg::launch_tc_bf16(cg, bn, mc, ew, ta, tb, tc, tc32, tb2, p, clusters, stream)
        : dtype == HGEMM_TF32 ? hg::launch_tc_tf32(cg, bn, mc, ew, ta, tb, tc, tc32, tb2, p, clusters, stream)
        : is_fp8(dtype)       ? hg::launch_tc_fp8(static_cast<int>(dtype), cg, bn, mc, ew, ta, tb, tc, tc32, tb2, p,
                                                  clusters, stream)
                            : hg::launch_tc_f16(cg, bn, mc, ew, ta, tb, tc, tc32, tb2, p, clusters, stream);
    if (work && work != scratch) cudaFreeAsync(work, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return HGEMM_OK;
}

}  // namespace

namespace hg {

hgemm_status_t gemm_in_scratch(const void* A, const void* B, void* C, int64_t M, int64_t N,
                               int64_t K, hgemm_dtype_t dtype, const hgemm_config_t* config,
                               cudaStream_t stream, void* scratch, size_t scratch_bytes) {
    return run(A, B, C, M, N, K, dtype, config, stream, scratch, scratch_bytes);
}

hgemm_status_t set_last_error(const char* what, cudaError_t e) {
    return cuda_fail(e, what);
}

}  // namespace hg

extern "C" {

hgemm_status_t hgemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                     hgemm_dtype_t dtype, void* stream) {
    return run(A, B, C, M, N, K, dtype, nullptr, static_cast<cudaStream_t>(stream));
}

hgemm_status_t hgemm_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                        hgemm_dtype_t dtype, const hgemm_config_t* cfg, void* stream) {
    return run(A, B, C, M, N, K, dtype, cfg, static_cast<cudaStream_t>(stream));
}

hgemm_status_t hgemm_fp8(const void* A, const void* B, void* C, const float* a_scale, const float* b_scale,
                         int64_t M, int64_t N, int64_t K, hgemm_dtype_t dtype, void* stream) {
    if (!is_fp8(dtype)) {
        t_last_error = "hgemm_fp8 takes HGEMM_E4M3 or HGEMM_E5M2";
        return HGEMM_ERR_INVALID_ARG;
    }
    return run(A, B, C, M, N, K, dtype, nullptr, static_cast<cudaStream_t>(stream), nullptr, 0, a_scale, b_scale);
}

hgemm_status_t hgemm_fp8_ex(const void* A, const void* B, void* C, const float* a_scale, const float* b_scale,
                            int64_t M, int64_t N, int64_t K, hgemm_dtype_t dtype, const hgemm_config_t* cfg,
                            void* stream) {
    if (!is_fp8(dtype)) {
        t_last_error = "hgemm_fp8_ex takes HGEMM_E4M3 or HGEMM_E5M2";
        return HGEMM_ERR_INVALID_ARG;
    }
    return run(A, B, C, M, N, K, dtype, cfg, static_cast<cudaStream_t>(stream), nullptr, 0, a_scale, b_scale);
}

hgemm_status_t hgemm_fp8_blockscaled_ex(const void* A, const void* B, void* C, const float* a_scale,
                                        const float* b_scale, int64_t M, int64_t N, int64_t K, int32_t block,
                                        hgemm_dtype_t dtype, const hgemm_config_t* cfg, void* stream) {
    t_last_error.clear();
    if (!is_fp8(dtype)) {
        t_last_error = "hgemm_fp8_blockscaled takes HGEMM_E4M3 or HGEMM_E5M2";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (block != 32 && block != 64) {
        t_last_error = "the scale block is 32 or 64";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (cfg && ((cfg->block_n != 0 && cfg->block_n != 128) || cfg->split_k > 1 || cfg->stream_k > 1 ||
                cfg->store_mode != 0 || cfg->cta_group < 0 || cfg->cta_group > 2)) {
        t_last_error = "the block-scaled fp8 GEMM takes cta_group 1 or 2, block_n 128, whole tiles and its "
                       "own stores";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (M > 0 && N > 0 && K > 0 &&
        (!a_scale || !b_scale || (reinterpret_cast<uintptr_t>(a_scale) & 3u) || (reinterpret_cast<uintptr_t>(b_scale) & 3u))) {
        t_last_error = "a_scale and b_scale must be 4-byte aligned device arrays";
        return HGEMM_ERR_INVALID_ARG;
    }
    return run(A, B, C, M, N, K, dtype, cfg, static_cast<cudaStream_t>(stream), nullptr, 0, a_scale, b_scale, 0,
               nullptr, block);
}

hgemm_status_t hgemm_fp8_blockscaled(const void* A, const void* B, void* C, const float* a_scale,
                                     const float* b_scale, int64_t M, int64_t N, int64_t K, int32_t block,
                                     hgemm_dtype_t dtype, void* stream) {
    return hgemm_fp8_blockscaled_ex(A, B, C, a_scale, b_scale, M, N, K, block, dtype, nullptr, stream);
}

hgemm_status_t hgemm_conv2d(const void* x, const void* w, void* y, int32_t N, int32_t H, int32_t W, int32_t C,
                            int32_t K, int32_t R, int32_t S, int32_t stride, int32_t pad, hgemm_dtype_t dtype,
                            void* stream) {
    t_last_error.clear();
    if (N < 0 || H < 1 || W < 1 || C < 1 || K < 1 || R < 1 || S < 1 || stride < 1 || pad < 0) {
        t_last_error = "conv2d needs N >= 0, H, W, C, K, R, S, stride >= 1 and pad >= 0";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (dtype != HGEMM_F16 && dtype != HGEMM_BF16 && dtype != HGEMM_TF32) {
        t_last_error = "conv2d takes HGEMM_F16, HGEMM_BF16 or HGEMM_TF32";
        return HGEMM_ERR_INVALID_ARG;
    }
    const int64_t Pl = (static_cast<int64_t>(H) + 2 * pad - R) / stride + 1;
    const int64_t Ql = (static_cast<int64_t>(W) + 2 * pad - S) / stride + 1;
    if (static_cast<int64_t>(H) + 2 * pad < R || static_cast<int64_t>(W) + 2 * pad < S || N == 0) return HGEMM_OK;
    const int es = esize_of(dtype);
    const int64_t M = static_cast<int64_t>(N) * Pl * Ql;
    const int64_t Kg = static_cast<int64_t>(R) * S * C;
    if (M > 2147483647LL || Kg > 2147483647LL || Pl > 2147483647LL || Ql > 2147483647LL) {
        t_last_error = "conv2d shape too large";
        return HGEMM_ERR_INVALID_ARG;
    }
    if (!x || !w || !y) {
        t_last_error = "null pointer for a non-empty operand";
        return HGEMM_ERR_INVALID_ARG;
    }
    const uintptr_t amask = static_cast<uintptr_t>(es - 1);
    if ((reinterpret_cast<uintptr_t>(x) & amask) || (reinterpret_cast<uintptr_t>(w) & amask) ||
        (reinterpret_cast<uintptr_t>(y) & amask)) {
        t_last_error = "operands must be aligned to their element size";
        return HGEMM_ERR_INVALID_ARG;
    }
    const int64_t xbytes = static_cast<int64_t>(es) * N * H * W * C;
    const int64_t wbytes = static_cast<int64_t>(es) * Kg * K;
    const int64_t ybytes = static_cast<int64_t>(es) * M * K;
    if (overlaps(y, ybytes, x, xbytes) || overlaps(y, ybytes, w, wbytes)) {
        t_last_error = "y overlaps x or w";
        return HGEMM_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // A pointwise, stride-1, unpadded convolution is the GEMM itself: x is
    // already the (N*H*W) x C matrix.
    if (R == 1 && S == 1 && stride == 1 && pad == 0) return run(x, w, y, M, K, Kg, dtype, nullptr, s);
    hg::ConvShape cs{N, H, W, C, K, R, S, stride, pad, static_cast<int32_t>(Pl), static_cast<int32_t>(Ql)};
    // Implicit GEMM: activations whose channels come in whole 128-byte blocks
    // (64 fp16/bf16 or 32 fp32 values) are read straight from x by TMA im2col
    // copies; the im2col corners and offsets are 8-bit, the traversal stride
    // at most 8.
    const bool implicit = C % bk_of(dtype) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 && pad <= 127 &&
                          R <= 128 && S <= 128 && stride <= 8 && g_conv_implicit.load(std::memory_order_relaxed);
    if (implicit) return run(x, w, y, M, K, Kg, dtype, nullptr, s, nullptr, 0, nullptr, nullptr, 0, &cs);
    int dev = 0;
    DeviceInfo info;
    hgemm_status_t st = device_info(&dev, &info);
    if (st != HGEMM_OK) return st;
    // the im2col matrix: M rows of Kg elements, padded to a 128-byte pitch
    const int64_t lda = pitch128(Kg, es);
    cudaMemPool_t pool;
    if ((st = pool_for_device(dev, &pool)) != HGEMM_OK) return st;
    void* A = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&A, static_cast<size_t>(align256(es * M * lda)), pool, s);
    if (e != cudaSuccess) {
        cuda_fail(e, "cudaMallocFromPoolAsync (im2col matrix)");
        return HGEMM_ERR_ALLOC;
    }
    if ((e = hg::launch_im2col(x, cs, es, A, lda, s)) != cudaSuccess) {
        cudaFreeAsync(A, s);
        return cuda_fail(e, "im2col");
    }
    st = run(A, w, y, M, K, Kg, dtype, nullptr, s, nullptr, 0, nullptr, nullptr, lda);
    cudaFreeAsync(A, s);
    return st;
}

namespace {

// Internal streams of hgemm_host, one set per device, created on first use and
// kept for the process: copies in (B, then the bands of A), the band GEMMs,
// and copies out (the bands of C).
struct HostStreams {
    cudaStream_t in = nullptr, compute = nullptr, out = nullptr;
};

hgemm_status_t host_streams(HostStreams* hs) {
    static std::mutex mu;
    static HostStreams cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return HGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(mu);
    HostStreams& c = cache[dev];
    if (!c.in) {
        HostStreams n;
        if ((e = cudaStreamCreateWithFlags(&n.in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&n.compute, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&n.out, cudaStreamNonBlocking)) != cudaSuccess) {
            if (n.in) cudaStreamDestroy(n.in);
            if (n.compute) cudaStreamDestroy(n.compute);
            if (n.out) cudaStreamDestroy(n.out);
            return cuda_fail(e, "cudaStreamCreateWithFlags");
        }
        c = n;
    }
    *hs = c;
    return HGEMM_OK;
}

}  // namespace

hgemm_status_t hgemm_host(const void* hA, const void* hB, void* hC, int64_t M, int64_t N,
                          int64_t K, hgemm_dtype_t dtype, void* dA, void* dB, void* dC,
                          void* stream) {
    t_last_error.clear();
    hgemm_status_t st = check_args(dA, dB, dC, M, N, K, dtype);
    if (st != HGEMM_OK) return st;
    if (M == 0 || N == 0) return HGEMM_OK;
    if (!hC || (K > 0 && (!hA || !hB))) {
        t_last_error = "null host pointer for a non-empty operand";
        return HGEMM_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    const int64_t es = esize_of(dtype), ces = c_esize_of(dtype);
    // Row bands of A and C: band i's copy in, GEMM and copy out run on three
    // streams, so copies of later bands overlap earlier bands' GEMMs and the
    // copies out overlap the copies in (the two directions of the host link,
    // about 190 and 180 GB/s on GB300, whatever the number of streams). The
    // copies in set the pace; what is left after them is the last band's GEMM
    // and copy out. Four bands, multiples of 256 rows and at least 512
    // (4096^3: 1 band 0.594 ms, 2 bands 0.494, 4 bands 0.462, 8 bands 0.474).
    // Small problems take one band.
    int64_t bands = (M >= 1024 && K > 0) ? 4 : 1;
    int64_t band_rows = (M + bands - 1) / bands;
    band_rows = (band_rows + 255) / 256 * 256;
    if (band_rows < 512) band_rows = bands > 1 ? 512 : M;
    if (band_rows > M) band_rows = M;
    bands = (M + band_rows - 1) / band_rows;
    HostStreams hs;
    if ((st = host_streams(&hs)) != HGEMM_OK) return st;
    cudaEvent_t ev[2 * 8 + 2];
    const int n_ev = static_cast<int>(2 * bands + 2);
    for (int i = 0; i < n_ev; ++i) {
        if ((e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming)) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
            return cuda_fail(e, "cudaEventCreateWithFlags");
        }
    }
    // On an error part of the pipeline may be enqueued: let it finish before
    // the events go and the caller reuses its buffers.
    auto drain = [&]() {
        cudaStreamSynchronize(hs.in);
        cudaStreamSynchronize(hs.compute);
        cudaStreamSynchronize(hs.out);
        for (int j = 0; j < n_ev; ++j) cudaEventDestroy(ev[j]);
    };
    auto fail = [&](cudaError_t err, const char* what) {
        drain();
        return cuda_fail(err, what);
    };
    // everything starts after the work already on `stream`
    cudaEvent_t ev_start = ev[2 * bands], ev_end_out = ev[2 * bands + 1];
    if ((e = cudaEventRecord(ev_start, s)) != cudaSuccess) return fail(e, "cudaEventRecord");
    if ((e = cudaStreamWaitEvent(hs.in, ev_start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hs.compute, ev_start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hs.out, ev_start, 0)) != cudaSuccess)
        return fail(e, "cudaStreamWaitEvent");
    if (K > 0 &&
        (e = cudaMemcpyAsync(dB, hB, static_cast<size_t>(es * K * N), cudaMemcpyHostToDevice, hs.in)) != cudaSuccess)
        return fail(e, "copy B to device");
    for (int64_t i = 0; i < bands; ++i) {
        const int64_t r0 = i * band_rows, rows = (r0 + band_rows <= M) ? band_rows : M - r0;
        cudaEvent_t ev_in = ev[2 * i], ev_done = ev[2 * i + 1];
        if (K > 0 && (e = cudaMemcpyAsync(static_cast<uint8_t*>(dA) + es * r0 * K,
                                          static_cast<const uint8_t*>(hA) + es * r0 * K,
                                          static_cast<size_t>(es * rows * K), cudaMemcpyHostToDevice, hs.in)) !=
                         cudaSuccess)
            return fail(e, "copy A to device");
        if ((e = cudaEventRecord(ev_in, hs.in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(hs.compute, ev_in, 0)) != cudaSuccess)
            return fail(e, "band event");
        if ((st = run(static_cast<const uint8_t*>(dA) + es * r0 * K, dB, static_cast<uint8_t*>(dC) + ces * r0 * N,
                      rows, N, K, dtype, nullptr, hs.compute)) != HGEMM_OK) {
            drain();  // keeps run()'s error message
            return st;
        }
        if ((e = cudaEventRecord(ev_done, hs.compute)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(hs.out, ev_done, 0)) != cudaSuccess)
            return fail(e, "band event");
        if ((e = cudaMemcpyAsync(static_cast<uint8_t*>(hC) + ces * r0 * N,
                                 static_cast<const uint8_t*>(dC) + ces * r0 * N,
                                 static_cast<size_t>(ces * rows * N), cudaMemcpyDeviceToHost, hs.out)) != cudaSuccess)
            return fail(e, "copy C to host");
    }
    // `stream` resumes after the last copy out (which follows every band)
    if ((e = cudaEventRecord(ev_end_out, hs.out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, ev_end_out, 0)) != cudaSuccess)
        return fail(e, "join");
    e = cudaStreamSynchronize(s);
    for (int j = 0; j < n_ev; ++j) cudaEventDestroy(ev[j]);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    return HGEMM_OK;
}

hgemm_status_t hgemm_plan(int64_t M, int64_t N, int64_t K, hgemm_dtype_t dtype,
                          const hgemm_config_t* cfg, int32_t sm_count, hgemm_plan_t* out) {
    t_last_error.clear();
    if (!out) return HGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || M > 2147483647LL || N > 2147483647LL || K > 2147483647LL ||
        !valid_dtype(dtype))
        return HGEMM_ERR_INVALID_ARG;
    int sms = sm_count;
    if (sms <= 0) {
        int dev = 0;
        DeviceInfo info;
        hgemm_status_t st = device_info(&dev, &info);
        if (st != HGEMM_OK) return st;
        sms = info.sms;
    }
    const int64_t es = esize_of(dtype), ces = c_esize_of(dtype);
    const bool a_bad = ((K * es) & 15) != 0, b_bad = ((N * es) & 15) != 0, c_bad = ((N * ces) & 15) != 0;
    hgemm_status_t st = make_plan(M, N, K, dtype, cfg, sms, a_bad, b_bad, c_bad, out);
    if (st != HGEMM_OK || sm_count > 0) return st;
    // planning for the current device: the K split the launch would keep
    int resident = 0;
    return fit_split_to_device(M, N, K, dtype, cfg, sms, a_bad, b_bad, c_bad, out, &resident);
}

int32_t hgemm_work_unit(const hgemm_plan_t* plan, int32_t cluster, int32_t i, int32_t* tile,
                        int32_t* kb0, int32_t* kb1, int32_t* kind) {
    const int32_t csize = plan ? static_cast<int32_t>(cluster_ctas(*plan)) : 1;
    if (!plan || plan->cta_group < 1 || cluster < 0 || cluster >= plan->grid_ctas / csize || i < 0 ||
        plan->num_kb < 1)
        return 0;
    hg::Schedule sc{};
    sc.num_tiles = plan->num_tiles;
    sc.dp_tiles = plan->dp_tiles;
    sc.num_kb = plan->num_kb;
    sc.clusters = plan->grid_ctas / csize;
    sc.sk_base = plan->sk_blocks;
    sc.sk_extra = plan->sk_extra;
    hg::WorkUnit w;
    if (!hg::next_unit(sc, cluster, i, w)) return 0;
    if (tile) *tile = w.tile;
    if (kb0) *kb0 = w.kb0;
    if (kb1) *kb1 = w.kb1;
    if (kind) *kind = w.kind;
    return 1;
}

void hgemm_tile_coord(int32_t t, int32_t tiles_m, int32_t tiles_n, int32_t group_m, int32_t* tm,
                      int32_t* tn) {
    int32_t a = 0, b = 0;
    if (tiles_m > 0 && tiles_n > 0 && group_m > 0) hg::tile_coord(t, tiles_m, tiles_n, group_m, a, b);
    if (tm) *tm = a;
    if (tn) *tn = b;
}

void hgemm_split_share(int32_t kb0, int32_t kb1, int32_t rank, int32_t parts, int32_t* lo, int32_t* hi) {
    if (!lo || !hi || parts < 1 || rank < 0 || rank >= parts || kb0 > kb1) return;
    int32_t a, b;
    hg::split_share(kb0, kb1, static_cast<uint32_t>(rank), parts, a, b);
    *lo = a;
    *hi = b;
}

hgemm_status_t hgemm_get_device_status(int32_t device, int32_t reset, uint32_t* info) {
    t_last_error.clear();
    int prev = 0;
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (device != prev && (e = cudaSetDevice(device)) != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    unsigned long long* ptr = nullptr;
    unsigned long long word = 0;
    hgemm_status_t st = HGEMM_OK;
    if ((e = hg::status_word_ptr(&ptr)) != cudaSuccess ||
        (e = cudaMemcpy(&word, ptr, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess) {
        st = cuda_fail(e, "read status word");
    } else {
        if (info) *info = static_cast<uint32_t>(word >> 32);
        st = static_cast<hgemm_status_t>(word & 0xFFFFFFFFull);
        if (reset && word != 0) {
            const unsigned long long zero = 0;
            if ((e = cudaMemcpy(ptr, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
                st = cuda_fail(e, "reset status word");
        }
    }
    if (device != prev) cudaSetDevice(prev);
    return st;
}

void hgemm_set_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1, std::memory_order_relaxed); }

#ifdef HG_TRACE
// Traced builds only: device buffer for the kernels' timeline records
// (grid_ctas x kTraceUnits x kTraceFields u64), or null.
void hgemm_trace_set(void* buf) { g_trace.store(static_cast<unsigned long long*>(buf)); }
#endif

void hgemm_conv2d_set_mode(int32_t mode) { g_conv_implicit.store(mode == 0, std::memory_order_relaxed); }

void hgemm_test_inject(int32_t kind) {
    g_inject.store(kind == 1 || kind == 2 ? kind : 0, std::memory_order_relaxed);
}

const char* hgemm_status_string(hgemm_status_t s) {
    switch (s) {
        case HGEMM_OK: return "HGEMM_OK";
        case HGEMM_ERR_INVALID_ARG: return "HGEMM_ERR_INVALID_ARG: invalid argument";
        case HGEMM_ERR_UNSUPPORTED_DEVICE: return "HGEMM_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 GPU";
        case HGEMM_ERR_CUDA: return "HGEMM_ERR_CUDA: a CUDA call failed";
        case HGEMM_ERR_ALLOC: return "HGEMM_ERR_ALLOC: workspace allocation failed";
        case HGEMM_ERR_TIMEOUT: return "HGEMM_ERR_TIMEOUT: a bounded wait in the kernel ran out";
    }
    return "unknown hgemm status";
}

const char* hgemm_last_error(void) { return t_last_error.c_str(); }

int32_t hgemm_version(void) { return 200; }

}  // extern "C"
