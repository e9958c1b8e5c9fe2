// hgemm_aux.cu - small kernels around the GEMM: the 128-byte-pitch repack of
// an operand whose rows TMA cannot address, the K = 0 zero fill, and the
// device status word that bounded waits report into.
#include <mutex>

#include "launch.h"

namespace hg {

__device__ unsigned long long g_status_word;

// Copy `rows` rows of `row_bytes` bytes (row r at src + r row_bytes: any
// alignment) into rows `dst_pitch` bytes apart (dst and dst_pitch multiples
// of 16), for up to two matrices in one launch (a RepackJob each). A warp
// copies one pass of a row at a time: lane l writes the pass's 16-byte
// segments l, l + 32, ..., kRepackBatch of them (8: 64 registers of data,
// three 256-thread blocks per SM; 16 was 2-3 us slower on every copied shape
// tried). A segment's bytes start at
// offset `off` inside an aligned 16-byte source block and run into the next
// block: every source block is read once, with an aligned 16-byte load, by
// the lane whose segment starts in it, and the next block comes from the
// neighbouring lane by shuffle (lane 31 loads the block after the pass
// itself). Blocks at or past the end of the source read as zero: a block
// that starts inside the buffer holds at least one of its bytes, so the load
// stays in mapped memory whatever the buffer's alignment. The last segment's
// bytes past row_bytes land in the destination row's padding, which the
// GEMM's tensor maps never reach. Measured against a thread-per-segment copy
// that loaded both blocks itself: 1000 x 4095 x 4104 bf16 (B copied) 57.0 ->
// 50.5 us end to end; L2 eviction hints (source evict-first, copy
// evict-last) changed nothing.
constexpr int kRepackBatch = 8;
constexpr int kRepackBlocksPerSm = 3;   // 256-thread blocks resident per SM (register bound)

__device__ __forceinline__ uint4 load_block(const uint8_t* b, const uint8_t* end) {
    return b < end ? __ldg(reinterpret_cast<const uint4*>(b)) : make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ uint4 shfl_down_u4(const uint4& v, uint32_t d) {
    return make_uint4(__shfl_down_sync(0xffffffffu, v.x, d), __shfl_down_sync(0xffffffffu, v.y, d),
                      __shfl_down_sync(0xffffffffu, v.z, d), __shfl_down_sync(0xffffffffu, v.w, d));
}

__device__ __forceinline__ uint4 shfl_u4(const uint4& v, int src) {
    return make_uint4(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src),
                      __shfl_sync(0xffffffffu, v.z, src), __shfl_sync(0xffffffffu, v.w, src));
}

// Work unit: one pass (32 x kRepackBatch segments, 4 KB) of one row; the
// units of job a's rows, then job b's, are spread over the warps in turn, so
// a launch ends at most one short unit after its last full round.
__global__ void __launch_bounds__(256, kRepackBlocksPerSm) repack_rows_kernel(RepackJob a, RepackJob b) {
    // the GEMM that reads the copies may start its set-up now
    grid_launch_dependents();
    const uint32_t lane = threadIdx.x & 31u;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    constexpr int64_t kPassSegs = 32 * kRepackBatch;
    const int64_t passes_a = (a.row_bytes + 16 * kPassSegs - 1) / (16 * kPassSegs);
    const int64_t passes_b = (b.row_bytes + 16 * kPassSegs - 1) / (16 * kPassSegs);
    const int64_t units_a = a.rows * passes_a;
    const int64_t units = units_a + b.rows * passes_b;
    for (int64_t u = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; u < units; u += nw) {
        const bool in_a = u < units_a;                      // warp-uniform
        const RepackJob& j = in_a ? a : b;
        const int64_t passes = in_a ? passes_a : passes_b;
        const int64_t ui = in_a ? u : u - units_a;
        const int64_t r = ui / passes;
        const int64_t t0 = (ui - r * passes) * kPassSegs;
        const uint8_t* const end = j.src + j.rows * j.row_bytes;
        const int64_t nseg = (j.row_bytes + 15) / 16;
        const uint8_t* const row = j.src + r * j.row_bytes;
        const uint32_t off = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row) & 15u);
        const uint8_t* const base = row - off;
        uint8_t* const d = j.dst + r * j.dst_pitch;
        uint4 v[kRepackBatch];
#pragma unroll
        for (int q = 0; q < kRepackBatch; ++q) {
            const int64_t t = t0 + 32 * q + lane;
            v[q] = t <= nseg ? load_block(base + 16 * t, end) : make_uint4(0u, 0u, 0u, 0u);
        }
        const int64_t tx = t0 + kPassSegs;
        const uint4 x = (lane == 31u && off != 0u && tx <= nseg) ? load_block(base + 16 * tx, end)
                                                                  : make_uint4(0u, 0u, 0u, 0u);
        if (off == 0u) {
#pragma unroll
            for (int q = 0; q < kRepackBatch; ++q) {
                const int64_t t = t0 + 32 * q + lane;
                if (t < nseg) *reinterpret_cast<uint4*>(d + 16 * t) = v[q];
            }
        } else {
#pragma unroll
            for (int q = 0; q < kRepackBatch; ++q) {
                uint4 hi = shfl_down_u4(v[q], 1);
                const uint4 nx = shfl_u4(v[q + 1 < kRepackBatch ? q + 1 : q], 0);
                if (lane == 31u) hi = q + 1 < kRepackBatch ? nx : x;
                const int64_t t = t0 + 32 * q + lane;
                if (t < nseg) *reinterpret_cast<uint4*>(d + 16 * t) = bytes_from(v[q], hi, off);
            }
        }
    }
}

// im2col for channels-last convolution: row m = (n, p, q) of A holds the
// receptive field of output pixel (n, p, q) in (r, s, c) order, c fastest:
//   A[m][(r*S + s)*C + c] = x[n][p*stride - pad + r][q*stride - pad + s][c]
// (0 outside the image), and columns [R*S*C, lda) are 0.
//
// Vector form (C a multiple of 16 bytes, x 16-byte aligned): one warp per
// (row, tap) segment copies that tap's C channels in 16-byte pieces, so the
// index arithmetic is done once per segment; the padding columns are one
// more segment per row. Element form otherwise: one thread per 16 bytes of a
// row, element by element.
template <typename T>
__global__ void im2col_vec_kernel(const T* __restrict__ x, ConvShape cs, T* __restrict__ A, int64_t lda) {
    constexpr int kPer = 16 / sizeof(T);
    const int lane = threadIdx.x & 31;
    const int64_t rows = static_cast<int64_t>(cs.N) * cs.P * cs.Q;
    const int taps = cs.R * cs.S;
    const int64_t taps_cols = static_cast<int64_t>(taps) * cs.C;
    const int segs = taps + (lda > taps_cols ? 1 : 0);
    const int cpieces = cs.C / kPer;
    // narrow taps (fewer than 32 pieces): a warp takes several segments at
    // once, lane = (segment within the group, piece)
    const int group = cpieces >= 32 ? 1 : 32 / cpieces;
    const int sub = cpieces >= 32 ? 0 : lane / cpieces;
    const int sl = cpieces >= 32 ? lane : lane - sub * cpieces;
    const int step = cpieces >= 32 ? 32 : cpieces;
    const int64_t total = rows * segs;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t g0 = (static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * group;
         g0 < total; g0 += warps * group) {
        const int64_t g = g0 + sub;
        if (sub >= group || g >= total) continue;
        const int64_t m = g / segs;
        const int seg = static_cast<int>(g - m * segs);
        T* dst = A + m * lda;
        if (seg == taps) {
            for (int64_t k = taps_cols + static_cast<int64_t>(sl) * kPer; k < lda; k += static_cast<int64_t>(step) * kPer)
                *reinterpret_cast<uint4*>(dst + k) = make_uint4(0, 0, 0, 0);
            continue;
        }
        const int q = static_cast<int>(m % cs.Q);
        const int64_t np = m / cs.Q;
        const int p = static_cast<int>(np % cs.P);
        const int n = static_cast<int>(np / cs.P);
        const int r = seg / cs.S, sx = seg - (seg / cs.S) * cs.S;
        const int h = p * cs.stride - cs.pad + r, w = q * cs.stride - cs.pad + sx;
        const bool inside = h >= 0 && h < cs.H && w >= 0 && w < cs.W;
        const T* src = x + ((static_cast<int64_t>(n) * cs.H + h) * cs.W + w) * cs.C;
        T* d = dst + static_cast<int64_t>(seg) * cs.C;
        for (int j = sl; j < cpieces; j += step)
            *reinterpret_cast<uint4*>(d + j * kPer) =
                inside ? *reinterpret_cast<const uint4*>(src + j * kPer) : make_uint4(0, 0, 0, 0);
    }
}

template <typename T>
__global__ void im2col_kernel(const T* __restrict__ x, ConvShape cs, T* __restrict__ A, int64_t lda) {
    constexpr int kPer = 16 / sizeof(T);
    const int64_t chunks = lda / kPer;
    const int64_t rows = static_cast<int64_t>(cs.N) * cs.P * cs.Q;
    const int64_t taps = static_cast<int64_t>(cs.R) * cs.S * cs.C;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < rows * chunks;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / chunks, k0 = (i - m * chunks) * kPer;
        const int q = static_cast<int>(m % cs.Q);
        const int64_t np = m / cs.Q;
        const int p = static_cast<int>(np % cs.P);
        const int n = static_cast<int>(np / cs.P);
        union {
            T v[kPer];
            uint4 u;
        } out;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int64_t kk = k0 + j;
            T v = T(0);
            if (kk < taps) {
                const int c = static_cast<int>(kk % cs.C);
                const int64_t rs = kk / cs.C;
                const int r = static_cast<int>(rs / cs.S), s = static_cast<int>(rs % cs.S);
                const int h = p * cs.stride - cs.pad + r, w = q * cs.stride - cs.pad + s;
                if (h >= 0 && h < cs.H && w >= 0 && w < cs.W)
                    v = x[((static_cast<int64_t>(n) * cs.H + h) * cs.W + w) * cs.C + c];
            }
            out.v[j] = v;
        }
        *reinterpret_cast<uint4*>(A + m * lda + k0) = out.u;
    }
}

cudaError_t launch_im2col(const void* x, const ConvShape& cs, int esize, void* A, int64_t lda,
                          cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(cs.N) * cs.P * cs.Q;
    if (rows <= 0) return cudaSuccess;
    if ((esize != 2 && esize != 4) || (lda * esize) % 16 != 0 || (reinterpret_cast<uintptr_t>(A) & 15) != 0)
        return cudaErrorInvalidValue;
    const bool vec = (static_cast<int64_t>(cs.C) * esize) % 16 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    int64_t blocks;
    if (vec) {
        const int64_t cpieces = static_cast<int64_t>(cs.C) * esize / 16;
        const int64_t group = cpieces >= 32 ? 1 : 32 / cpieces;
        const int64_t segs = rows * (static_cast<int64_t>(cs.R) * cs.S + 1);
        blocks = (segs / group + 7) / 8 + 1;  // 8 warps per block, `group` segments per warp
    } else {
        blocks = (rows * (lda * esize / 16) + 255) / 256;
    }
    if (blocks > 152 * 64) blocks = 152 * 64;
    const unsigned b = static_cast<unsigned>(blocks);
    if (esize == 2) {
        if (vec)
            im2col_vec_kernel<uint16_t><<<b, 256, 0, stream>>>(static_cast<const uint16_t*>(x), cs,
                                                                static_cast<uint16_t*>(A), lda);
        else
            im2col_kernel<uint16_t><<<b, 256, 0, stream>>>(static_cast<const uint16_t*>(x), cs,
                                                            static_cast<uint16_t*>(A), lda);
    } else {
        if (vec)
            im2col_vec_kernel<uint32_t><<<b, 256, 0, stream>>>(static_cast<const uint32_t*>(x), cs,
                                                                static_cast<uint32_t*>(A), lda);
        else
            im2col_kernel<uint32_t><<<b, 256, 0, stream>>>(static_cast<const uint32_t*>(x), cs,
                                                            static_cast<uint32_t*>(A), lda);
    }
    return cudaGetLastError();
}

__global__ void zero_kernel(uint16_t* __restrict__ dst, int64_t count) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        dst[i] = 0;
}

cudaError_t launch_repack(const RepackJob& a, const RepackJob& b, cudaStream_t stream) {
    RepackJob ja = a, jb = b;
    if (ja.rows < 0) ja.rows = 0;
    if (jb.rows < 0) jb.rows = 0;
    constexpr int64_t kPassBytes = 16 * 32 * kRepackBatch;
    const int64_t units = ja.rows * ((ja.row_bytes + kPassBytes - 1) / kPassBytes) +
                          jb.rows * ((jb.row_bytes + kPassBytes - 1) / kPassBytes);
    if (units == 0) return cudaSuccess;
    // one unit per warp at a time, on the blocks that fit at once
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        sms = 152;
    int64_t blocks = (units + 7) / 8;
    const int64_t resident = static_cast<int64_t>(sms) * kRepackBlocksPerSm;
    if (blocks > resident) blocks = resident;
    repack_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(ja, jb);
    return cudaGetLastError();
}

cudaError_t launch_zero(uint16_t* dst, int64_t count, cudaStream_t stream) {
    if (count <= 0) return cudaSuccess;
    int64_t blocks = (count + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    zero_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(dst, count);
    return cudaGetLastError();
}

cudaError_t status_word_ptr(unsigned long long** out) {
    static std::mutex mu;
    static unsigned long long* cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return e;
        cache[dev] = static_cast<unsigned long long*>(p);
    }
    *out = cache[dev];
    return cudaSuccess;
}

// Stage counts and shared-memory bytes per (cta_group, block_n, operand
// bytes, K split): a B swizzle atom is 128 bytes of columns, so the stage
// size of a narrow tile depends on the operand size; a K split has no
// epilogue staging boxes.
#define HG_CFG_SWITCH(FIELD)                                                                   \
    if (esize == 2 && split > 1) {                                                             \
        if (cta_group == 1 && block_n == 128) return TcCfg<1, 128, 2, 2>::FIELD;               \
        if (cta_group == 1 && block_n == 256) return TcCfg<1, 256, 2, 2>::FIELD;               \
    } else if (esize == 2) {                                                                   \
        if (cta_group == 1 && block_n == 64) return TcCfg<1, 64, 2>::FIELD;                    \
        if (cta_group == 1 && block_n == 128) return TcCfg<1, 128, 2>::FIELD;                  \
        if (cta_group == 1 && block_n == 256) return TcCfg<1, 256, 2>::FIELD;                  \
        if (cta_group == 2 && block_n == 128) return TcCfg<2, 128, 2>::FIELD;                  \
        if (cta_group == 2 && block_n == 224) return TcCfg<2, 224, 2>::FIELD;                  \
        if (cta_group == 2 && block_n == 256) return TcCfg<2, 256, 2>::FIELD;                  \
    } else if (esize == 4 || esize == 1) {                                                     \
        if (cta_group == 1 && block_n == 64) return esize == 4 ? TcCfg<1, 64, 4>::FIELD : TcCfg<1, 64, 1>::FIELD;     \
        if (cta_group == 1 && block_n == 128) return esize == 4 ? TcCfg<1, 128, 4>::FIELD : TcCfg<1, 128, 1>::FIELD;  \
        if (cta_group == 1 && block_n == 256) return esize == 4 ? TcCfg<1, 256, 4>::FIELD : TcCfg<1, 256, 1>::FIELD;  \
        if (cta_group == 2 && block_n == 128) return esize == 4 ? TcCfg<2, 128, 4>::FIELD : TcCfg<2, 128, 1>::FIELD;  \
        if (cta_group == 2 && block_n == 224) return esize == 4 ? TcCfg<2, 224, 4>::FIELD : TcCfg<2, 224, 1>::FIELD;  \
        if (cta_group == 2 && block_n == 256) return esize == 4 ? TcCfg<2, 256, 4>::FIELD : TcCfg<2, 256, 1>::FIELD;  \
    }                                                                                          \
    return 0;

int tc_stages(int cta_group, int block_n, int esize, int split) { HG_CFG_SWITCH(kStages) }

int tc_tmem_cols(int cta_group, int block_n) {
    if (cta_group == 1 && block_n == 64) return TcCfg<1, 64>::kTmemCols;
    if (cta_group == 1 && block_n == 128) return TcCfg<1, 128>::kTmemCols;
    if (cta_group == 1 && block_n == 256) return TcCfg<1, 256>::kTmemCols;
    if (cta_group == 2 && block_n == 128) return TcCfg<2, 128>::kTmemCols;
    if (cta_group == 2 && block_n == 224) return TcCfg<2, 224>::kTmemCols;
    if (cta_group == 2 && block_n == 256) return TcCfg<2, 256>::kTmemCols;
    return 0;
}

int tc_smem_bytes(int cta_group, int block_n, int esize, int split) { HG_CFG_SWITCH(kSmemBytes) }

}  // namespace hg
