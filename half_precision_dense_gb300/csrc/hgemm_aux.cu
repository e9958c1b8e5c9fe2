// hgemm_aux.cu - small kernels around the GEMM: the 16-byte-pitch repack of
// an operand whose rows TMA cannot address, the K = 0 zero fill, and the
// device status word that bounded waits report into.
#include <mutex>

#include "launch.h"

namespace hg {

__device__ unsigned long long g_status_word;

// Copy a rows x cols matrix of 16-bit values with row pitch `cols` (any base
// alignment of 2 bytes) into `dst` with row pitch `dst_ld` (a multiple of 8
// elements, 16-byte aligned base). Each thread moves 8 consecutive elements
// of one row: 2-byte loads (the source rows are not 16-byte aligned), one
// 16-byte store. Elements past `cols` in the destination row are not written.
__global__ void repack_rows_kernel(const uint16_t* __restrict__ src, int64_t rows, int64_t cols,
                                   uint16_t* __restrict__ dst, int64_t dst_ld) {
    const int64_t chunks = (cols + 7) / 8;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const uint16_t* s = src + r * cols;
        uint16_t* d = dst + r * dst_ld;
        for (int64_t ch = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; ch < chunks;
             ch += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const int64_t c0 = ch * 8;
            if (c0 + 8 <= cols) {
                uint16_t v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = s[c0 + i];
                uint4 packed;
                packed.x = v[0] | (static_cast<uint32_t>(v[1]) << 16);
                packed.y = v[2] | (static_cast<uint32_t>(v[3]) << 16);
                packed.z = v[4] | (static_cast<uint32_t>(v[5]) << 16);
                packed.w = v[6] | (static_cast<uint32_t>(v[7]) << 16);
                *reinterpret_cast<uint4*>(d + c0) = packed;
            } else {
                for (int64_t c = c0; c < cols; ++c) d[c] = s[c];
            }
        }
    }
}

__global__ void zero_kernel(uint16_t* __restrict__ dst, int64_t count) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        dst[i] = 0;
}

cudaError_t launch_repack(const uint16_t* src, int64_t rows, int64_t cols, uint16_t* dst,
                          int64_t dst_ld, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const int64_t chunks = (cols + 7) / 8;
    const int threads = 128;
    int64_t gx = (chunks + threads - 1) / threads;
    if (gx > 1024) gx = 1024;
    int64_t gy = rows < 32768 ? rows : 32768;
    repack_rows_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), threads, 0,
                         stream>>>(src, rows, cols, dst, dst_ld);
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

int tc_stages(int cta_group, int block_n) {
    if (cta_group == 1 && block_n == 64) return TcCfg<1, 64>::kStages;
    if (cta_group == 1 && block_n == 128) return TcCfg<1, 128>::kStages;
    if (cta_group == 1 && block_n == 256) return TcCfg<1, 256>::kStages;
    if (cta_group == 2 && block_n == 128) return TcCfg<2, 128>::kStages;
    if (cta_group == 2 && block_n == 224) return TcCfg<2, 224>::kStages;
    if (cta_group == 2 && block_n == 256) return TcCfg<2, 256>::kStages;
    return 0;
}

int tc_tmem_cols(int cta_group, int block_n) {
    if (cta_group == 1 && block_n == 64) return TcCfg<1, 64>::kTmemCols;
    if (cta_group == 1 && block_n == 128) return TcCfg<1, 128>::kTmemCols;
    if (cta_group == 1 && block_n == 256) return TcCfg<1, 256>::kTmemCols;
    if (cta_group == 2 && block_n == 128) return TcCfg<2, 128>::kTmemCols;
    if (cta_group == 2 && block_n == 224) return TcCfg<2, 224>::kTmemCols;
    if (cta_group == 2 && block_n == 256) return TcCfg<2, 256>::kTmemCols;
    return 0;
}

int tc_smem_bytes(int cta_group, int block_n) {
    if (cta_group == 1 && block_n == 64) return TcCfg<1, 64>::kSmemBytes;
    if (cta_group == 1 && block_n == 128) return TcCfg<1, 128>::kSmemBytes;
    if (cta_group == 1 && block_n == 256) return TcCfg<1, 256>::kSmemBytes;
    if (cta_group == 2 && block_n == 128) return TcCfg<2, 128>::kSmemBytes;
    if (cta_group == 2 && block_n == 224) return TcCfg<2, 224>::kSmemBytes;
    if (cta_group == 2 && block_n == 256) return TcCfg<2, 256>::kSmemBytes;
    return 0;
}

}  // namespace hg
