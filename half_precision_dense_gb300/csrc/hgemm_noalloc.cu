// hgemm_noalloc.cu - hgemm for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) on the GEMM path:
// code running while a CUDA graph is being captured with allocation
// disallowed, real-time or embedded pipelines that fix their memory at start
// and treat any later allocation as a fault, and hosts whose device memory is
// owned by another runtime's pool. For them, hgemm_noalloc() takes the
// workspace the GEMM may need - the 128-byte-pitch copy of an operand whose
// rows TMA cannot address, and the fp32 partial sums of a stream-K schedule
// (hgemm_noalloc_ex with a config) - from a fixed array compiled into this
// library instead of from the stream-ordered allocator.
#include <mutex>

#include "hgemm.h"
#include "launch.h"

namespace {

// 64 MiB of scratch: holds the repacked copy of any operand up to 32 Mi
// half-precision elements (e.g. B of the 4104 x 4095 tail workload, 33.6 MB).
// Every GPU that loads this library holds the array until the process exits.
constexpr size_t kScratchBytes = size_t{64} << 20;

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

// Device address of the scratch array on the current device, looked up once
// per device. In host code `g_noalloc_scratch` is only a host-side stand-in
// for the symbol, never a device address: it must not be handed to a kernel.
hgemm_status_t scratch_ptr(void** out) {
    static std::mutex mu;
    static void* cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return hg::set_last_error("hgemm_noalloc: cudaGetDevice", e);
    if (dev < 0 || dev >= 64) return HGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return hg::set_last_error("hgemm_noalloc: cudaGetSymbolAddress(scratch)", e);
        cache[dev] = p;
    }
    *out = cache[dev];
    return HGEMM_OK;
}

}  // namespace

extern "C" hgemm_status_t hgemm_noalloc_ex(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                           int64_t K, hgemm_dtype_t dtype, const hgemm_config_t* config,
                                           void* stream) {
    void* scratch = nullptr;
    hgemm_status_t st = scratch_ptr(&scratch);
    if (st != HGEMM_OK) return st;
    return hg::gemm_in_scratch(A, B, C, M, N, K, dtype, config, static_cast<cudaStream_t>(stream), scratch,
                               kScratchBytes);
}

extern "C" hgemm_status_t hgemm_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                        int64_t K, hgemm_dtype_t dtype, void* stream) {
    return hgemm_noalloc_ex(A, B, C, M, N, K, dtype, nullptr, stream);
}

extern "C" uint64_t hgemm_noalloc_scratch_bytes(void) { return kScratchBytes; }
