// launch.h - internal interface between the C-ABI front end (hgemm_api.cu)
// and the translation units that hold the kernel instantiations.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hgemm.h"
#include "hgemm_fp8bs.cuh"
#include "hgemm_tc.cuh"

namespace hg {

// Launch the tcgen05 kernel for (cta_group, block_n, mc, epi) with `clusters`
// CTA clusters (of cta_group * mc CTAs) on `stream`; `epi` is the number of
// epilogue warps (8, or 16 for a 16-bit C on 224- and 256-wide tiles). Returns
// cudaErrorInvalidValue for a combination that is not instantiated.
// `c` stores 64-column chunks of C; `c32` the 32-column last chunk of tiles
// whose width is an odd multiple of 32; `b2` loads the part-full last B
// atom of a CTA (its box is that atom's used columns; unused otherwise).
cudaError_t launch_tc_bf16(int cta_group, int block_n, int mc, int epi, const CUtensorMap& a, const CUtensorMap& b,
                           const CUtensorMap& c, const CUtensorMap& c32, const CUtensorMap& b2, const TcParams& p,
                           int clusters, cudaStream_t stream);
cudaError_t launch_tc_f16(int cta_group, int block_n, int mc, int epi, const CUtensorMap& a, const CUtensorMap& b,
                          const CUtensorMap& c, const CUtensorMap& c32, const CUtensorMap& b2, const TcParams& p,
                          int clusters, cudaStream_t stream);
// tf32: fp32 A, B and C; (cta_group, block_n) in (1, 64|128|256), (2, 128|256); mc 1.
cudaError_t launch_tc_tf32(int cta_group, int block_n, int mc, int epi, const CUtensorMap& a, const CUtensorMap& b,
                           const CUtensorMap& c, const CUtensorMap& c32, const CUtensorMap& b2, const TcParams& p,
                           int clusters, cudaStream_t stream);

// Most CTA clusters of the (cta_group, block_n) kernel that can be resident at
// once on the current device (0 on error).
int max_active_clusters_bf16(int cta_group, int block_n, int mc, int epi);
int max_active_clusters_f16(int cta_group, int block_n, int mc, int epi);
int max_active_clusters_tf32(int cta_group, int block_n, int mc, int epi);
// fp8: kind 3 = E4M3, 4 = E5M2 operands (B row-major, read MN-major), bf16 C;
// the tf32 tile shapes.
cudaError_t launch_tc_fp8(int kind, int cta_group, int block_n, int mc, int epi, const CUtensorMap& a,
                          const CUtensorMap& b, const CUtensorMap& c, const CUtensorMap& c32, const CUtensorMap& b2,
                          const TcParams& p, int clusters, cudaStream_t stream);
int max_active_clusters_fp8(int kind, int cta_group, int block_n, int mc, int epi);

// Whether the kernel instance for (cta_group, block_n, mc, epi) is compiled
// (host only, no device needed): the planner refuses a plan without one.
bool tc_instance_exists_bf16(int cta_group, int block_n, int mc, int epi);
bool tc_instance_exists_f16(int cta_group, int block_n, int mc, int epi);
bool tc_instance_exists_tf32(int cta_group, int block_n, int mc, int epi);
bool tc_instance_exists_fp8(int kind, int cta_group, int block_n, int mc, int epi);

// The block-scaled fp8 kernel (hgemm_fp8bs.cuh): kind 3 = E4M3, 4 = E5M2;
// cta_group 1 (128 x 128 tiles) or 2 (256 x 128); gs = 32 or 64 (scale block).
// B is read in place (MN-major); `b2` loads a pair CTA's 64-column half atom.
cudaError_t launch_fp8bs(int kind, int cta_group, int gs, const CUtensorMap& a, const CUtensorMap& b,
                         const CUtensorMap& b2, const Fp8bsParams& p, int clusters, cudaStream_t stream);
int max_active_clusters_fp8bs(int kind, int cta_group, int gs);
int fp8bs_stages(int cta_group);
int fp8bs_smem_bytes(int cta_group);
int fp8bs_tmem_cols();

// Shared-memory ring depth and bytes of an instantiation (host constants) for
// operands of `esize` bytes (2: fp16/bf16, 4: tf32, 1: fp8).
int tc_stages(int cta_group, int block_n, int esize, int split);
int tc_smem_bytes(int cta_group, int block_n, int esize, int split);
int tc_tmem_cols(int cta_group, int block_n);

// Auxiliary kernels (hgemm_aux.cu). The repack copies `rows` rows of
// `row_bytes` bytes (any alignment, row r at src + r row_bytes) into rows
// `dst_pitch` bytes apart (dst and dst_pitch multiples of 16); one launch
// takes up to two matrices (rows = 0: none).
struct RepackJob {
    const uint8_t* src;
    int64_t rows, row_bytes;
    uint8_t* dst;
    int64_t dst_pitch;
};
cudaError_t launch_repack(const RepackJob& a, const RepackJob& b, cudaStream_t stream);
cudaError_t launch_zero(uint16_t* dst, int64_t count, cudaStream_t stream);
// Convolution geometry (channels-last): x N x H x W x C, filters R x S x C x K,
// output N x P x Q x K.
struct ConvShape {
    int32_t N, H, W, C, K, R, S, stride, pad, P, Q;
};
// A (N*P*Q rows of `lda` elements of `esize` = 2 or 4 bytes; lda * esize a
// multiple of 16, A 16-byte aligned) = the im2col matrix of x.
cudaError_t launch_im2col(const void* x, const ConvShape& cs, int esize, void* A, int64_t lda,
                          cudaStream_t stream);
// Device address of the status word on the current device (cached per device).
cudaError_t status_word_ptr(unsigned long long** out);

// The GEMM of hgemm_ex() (config may be null), with the workspace taken from
// `scratch` (`scratch_bytes` long) instead of the stream-ordered allocator
// (hgemm_api.cu). Shapes needing more workspace give HGEMM_ERR_INVALID_ARG.
hgemm_status_t gemm_in_scratch(const void* A, const void* B, void* C, int64_t M, int64_t N,
                               int64_t K, hgemm_dtype_t dtype, const hgemm_config_t* config,
                               cudaStream_t stream, void* scratch, size_t scratch_bytes);
// Record a failed CUDA call as this thread's last error; returns HGEMM_ERR_CUDA.
hgemm_status_t set_last_error(const char* what, cudaError_t e);

}  // namespace hg
