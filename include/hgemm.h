/*
 * hgemm.h - C ABI of the GB300 (sm_103a) dense half-precision GEMM library.
 *
 * The operation ("[CUDA 优化实战] hgemm - 超越 cuBLAS", section 1, the kernel
 * signature hgemm_*_kernel(T *a, T *b, T *c, int m, int n, int k)):
 *
 *     C[i][j] = round_to_nearest_even( sum_k A[i][k] * B[k][j] )
 *
 *   A  M x K, row-major (element (i, k) at A[i*K + k])     fp16 or bf16
 *   B  K x N, row-major (element (k, j) at B[k*N + j])     same dtype as A
 *   C  M x N, row-major (element (i, j) at C[i*N + j])     same dtype as A
 *
 * Products are accumulated in fp32 (in tensor memory) and each C element is
 * rounded once to the input dtype, as the page's mma.sync ... .f32 accumulate
 * and __float22half2_rn / __float22bfloat162_rn write-back do. The order of the
 * fp32 additions is unspecified, so results agree with an exact sum within the
 * rounding of fp32 accumulation, not bit for bit.
 *
 * TF32 variant (dtype HGEMM_TF32; the series' earlier kernel multiplied tf32
 * operands with the m16n8k8 tensor-core shape, same page, section 1): A, B
 * and C are fp32 arrays with the same layouts. Each operand enters the
 * product as its tf32 part - the sign, the 8 exponent bits and the top 10
 * fraction bits, the low 13 fraction bits ignored - the products (exact in
 * fp32) are accumulated in fp32, and C receives that fp32 accumulator.
 *
 * FP8 variant (dtypes HGEMM_E4M3 / HGEMM_E5M2; "深度学习加速核心：GEMM优化从分块到
 * TensorCore的实战解析", sections 2.3 and 4.3: E4M3 and E5M2 operands used with
 * per-layer or per-channel scale factors): A and B hold 8-bit OCP floats of
 * one format (E4M3: bias 7, no infinities, S.1111.111 NaN; E5M2: bias 15,
 * IEEE infinities and NaNs) in the same layouts; C is bfloat16:
 *
 *     C[i][j] = round_to_nearest_even_bf16( a_scale[i] * b_scale[j] * sum_k A[i][k] * B[k][j] )
 *
 * with the products (exact) accumulated in fp32 and the two fp32 scales
 * applied to the fp32 sum (hgemm_fp8; hgemm() with an fp8 dtype uses 1).
 *
 * Edge shapes ("CUDA GEMM 优化实践笔记", the register-tiled kernel's
 * bounds-checked tile loads fill out-of-range elements with zero): any M, N, K
 * >= 0 is accepted; elements outside the matrices contribute nothing and no
 * element outside C is written. M == 0 or N == 0 does nothing; K == 0 writes
 * zeros to C.
 *
 * Conventions for every entry point:
 *   - Pointers named A, B, C are DEVICE pointers on the calling thread's
 *     current CUDA device, dense and contiguous as above, owned by the caller.
 *     The library never frees or retains them past the call's stream work.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Work is enqueued asynchronously; no entry point synchronises
 *     the stream unless its comment says so.
 *   - C must not overlap A or B (checked; HGEMM_ERR_INVALID_ARG).
 *   - Return values are hgemm_status_t. On HGEMM_ERR_CUDA the CUDA error text
 *     is available from hgemm_last_error() on the same thread.
 *   - There is no CPU fallback: a device that is not compute capability 10.3
 *     gives HGEMM_ERR_UNSUPPORTED_DEVICE.
 *   - Per device, the library keeps state for the life of the process: the
 *     device addresses of its status word and of hgemm_noalloc's array, its
 *     memory pool, hgemm_host's streams and the kernels' shared-memory
 *     settings. It looks them up on first use and never again, so it must
 *     not be called on a device after cudaDeviceReset() on that device in
 *     the same process (the cached addresses would belong to the destroyed
 *     context).
 */
#ifndef HGEMM_H_
#define HGEMM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HGEMM_F16 = 0,  /* IEEE binary16 A, B and C */
    HGEMM_BF16 = 1, /* bfloat16 A, B and C */
    HGEMM_TF32 = 2, /* fp32 A, B and C, multiplied as tf32 (see above) */
    HGEMM_E4M3 = 3, /* 8-bit E4M3 A and B, bfloat16 C (see hgemm_fp8) */
    HGEMM_E5M2 = 4  /* 8-bit E5M2 A and B, bfloat16 C (see hgemm_fp8) */
} hgemm_dtype_t;

typedef enum {
    HGEMM_OK = 0,
    HGEMM_ERR_INVALID_ARG = 1,        /* null pointer with a non-empty shape, negative or too large
                                         dimension, unknown dtype, C overlapping A or B, bad config */
    HGEMM_ERR_UNSUPPORTED_DEVICE = 2, /* no CUDA device, or not compute capability 10.3 */
    HGEMM_ERR_CUDA = 3,               /* a CUDA runtime/driver call failed (see hgemm_last_error) */
    HGEMM_ERR_ALLOC = 4,              /* the stream-ordered workspace could not be allocated */
    HGEMM_ERR_TIMEOUT = 5             /* reported by hgemm_get_device_status: a bounded wait in the
                                         kernel ran out and the kernel returned early */
} hgemm_status_t;

/*
 * hgemm - C = A.B as described above, enqueued on `stream`.
 *
 * A, B: device pointers to the operands (read only). C: device pointer to the
 * result (written). M, N, K: dimensions, each in [0, 2^31 - 1]. dtype:
 * HGEMM_F16, HGEMM_BF16 or HGEMM_TF32 (A, B and C share the element type;
 * pointers aligned to it).
 *
 * Workspace: operands whose row pitch (K or N elements) or base address is
 * not a multiple of 16 bytes are first copied into a workspace whose rows
 * start on 128-byte boundaries by one copy kernel, and the GEMM launches as
 * its programmatic dependent (its set-up overlaps the copy's tail). A whose
 * rows are an odd multiple of 16 bytes apart is copied too when the plan
 * takes 224-wide pair tiles and N >= 3584 (its loads run 10-20 % slower in
 * place; hgemm_plan's repack_a tells); such a C is written with
 * realigned 16-byte and element stores (store_mode 5 below), and when
 * tiles are shared by stream-K ranges the parts' fp32 partial sums go through
 * the workspace too. It comes from a stream-ordered memory pool owned
 * by the library (one per device, cudaMallocFromPoolAsync / cudaFreeAsync on
 * `stream`; the pool keeps up to 256 MiB cached between calls). Calls that need
 * no workspace allocate nothing; hgemm_plan reports the bytes.
 *
 * CUDA graphs: the call may be recorded by stream capture (the pool
 * allocation becomes a graph allocation node). The capture holds the
 * pointers, so replays read the operands' current values. Stream-K parts
 * mark their partial sums with a number unique to each launch, which a graph
 * replays unchanged, so a captured call with a stream-K phase first clears
 * its marks (one small memset node in the graph).
 */
hgemm_status_t hgemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                     hgemm_dtype_t dtype, void* stream);

/*
 * hgemm_conv2d - 2-D convolution as one GEMM through im2col
 * ("深度学习加速核心：GEMM优化从分块到TensorCore的实战解析", section 1.1: the
 * input feature map rearranged by the kernel's receptive fields into one large
 * matrix turns the convolution into a GEMM).
 *
 *   x  N x H x W x C  (channels last), device
 *   w  R x S x C x K  (read as an (R*S*C) x K row-major matrix), device
 *   y  N x P x Q x K  (written), device, P = (H + 2 pad - R) / stride + 1,
 *                      Q = (W + 2 pad - S) / stride + 1
 *
 *   y[n][p][q][k] = round( sum_{r,s,c} x[n][p*stride-pad+r][q*stride-pad+s][c] * w[r][s][c][k] )
 *
 * (cross-correlation; x is zero outside the image; fp32 accumulation; the
 * rounding and element types are those of hgemm() for dtype HGEMM_F16,
 * HGEMM_BF16 or HGEMM_TF32). The im2col matrix (N*P*Q rows of R*S*C elements,
 * padded to a 16-byte pitch) lives in the library's stream-ordered pool for
 * the duration of the call's stream work; then hgemm's path computes
 * y = A . w. A 1 x 1 filter with stride 1 and no padding needs no im2col (x
 * is the (N*H*W) x C matrix) and goes straight to the GEMM. When C is a
 * multiple of 64 (fp16/bf16) or 32 (tf32), x is 16-byte aligned, stride <= 8
 * and pad <= 127, the matrix is never built: the GEMM's producer reads each
 * 128-pixel x 128-byte tile of it straight from x with TMA im2col-mode copies
 * (implicit GEMM).
 * N == 0 or an output with no pixels does nothing. Errors as for
 * hgemm(); a negative or zero size (other than N), stride < 1 or pad < 0 is
 * HGEMM_ERR_INVALID_ARG.
 */
hgemm_status_t hgemm_conv2d(const void* x, const void* w, void* y, int32_t N, int32_t H, int32_t W, int32_t C,
                            int32_t K, int32_t R, int32_t S, int32_t stride, int32_t pad, hgemm_dtype_t dtype,
                            void* stream);

/*
 * hgemm_conv2d_set_mode - 0 (default): hgemm_conv2d takes the implicit GEMM
 * where the shape allows it; 1: always the explicit im2col matrix (the same
 * results; for comparisons and tests). Process-wide.
 */
void hgemm_conv2d_set_mode(int32_t mode);

/*
 * hgemm_noalloc - hgemm for callers that must not allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc on the GEMM path: work recorded into a CUDA
 * graph whose capture forbids allocation, real-time or embedded pipelines
 * that reserve all memory up front, and hosts whose device memory belongs to
 * another runtime's pool.
 *
 * Same operation and arguments as hgemm(), and the same results. The only
 * workspace the GEMM can need (the 128-byte-pitch copy of A or B when a row
 * pitch or base address is not 16-byte aligned, and the fp32 partial sums of
 * the stream-K phase) comes from a fixed 64 MiB array inside the library
 * (hgemm_noalloc_scratch_bytes()); the call makes no cudaMalloc,
 * cudaMallocAsync, cudaFree or other allocating call.
 *   - A shape whose workspace would exceed the array returns
 *     HGEMM_ERR_INVALID_ARG (hgemm_last_error() gives the sizes) and enqueues
 *     nothing; a copy of A made only for speed is left out instead when it
 *     would not fit (A is then read in place). The stream-K partial sums need at most one 128 x 256 fp32
 *     block per CTA (under 20 MiB), so the limit only bites on unaligned
 *     operands (their 128-byte-pitch copies).
 *   - Every call on a device shares that device's array, which keeps the last
 *     call's contents (nothing in it needs to start at zero: stream-K parts
 *     mark their partial sums with a number unique to each launch, so stale
 *     marks are never mistaken for fresh ones; a captured call clears its
 *     marks first, as for hgemm()). Calls whose GPU
 *     work overlaps - on different streams, or from different host threads -
 *     race on the array: serialise them (one stream, or events).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture begins.
 *   - Every GPU that loads the library holds the array until the process exits.
 */
hgemm_status_t hgemm_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                             int64_t K, hgemm_dtype_t dtype, void* stream);

/* Size in bytes of hgemm_noalloc's fixed scratch array. */
uint64_t hgemm_noalloc_scratch_bytes(void);

/*
 * Launch configuration, for tuning sweeps and tests. Zero in any field means
 * "let the planner choose". A configuration whose fields are each valid but
 * whose combination has no compiled kernel is HGEMM_ERR_INVALID_ARG (from
 * hgemm_plan as from the GEMM calls; hgemm_last_error names it).
 *   cta_group:     1 = one CTA per 128-row tile; 2 = a CTA pair (cluster of 2)
 *                  sharing a 256-row tile through tcgen05 cta_group::2.
 *   block_n:       columns of C per tile: 64, 128 or 256 with cta_group 1;
 *                  128, 224 or 256 with cta_group 2.
 *   group_m:       tile rows per raster group (L2 reuse), >= 1.
 *   max_clusters:  cap on resident CTA clusters (forces more tiles per CTA).
 *   store_mode:    1 = TMA tensor stores of C (through a swizzled smem box),
 *                  2 = plain per-element stores, 3 = 16-byte vector stores
 *                  straight from registers, 4 = 16-byte vector stores of whole
 *                  rows read back from the swizzled smem box (1, 3 and 4 need
 *                  a 16-byte aligned C whose row pitch is a multiple of 16
 *                  bytes), 5 = the staged rows written as the aligned 16-byte
 *                  segments they cover, shifted into place, with element
 *                  stores at each row's ragged ends (16-bit C of any pitch).
 *                  The planner takes 4 for an aligned C (1 when the K loop
 *                  has at most 8 blocks: the epilogue then sets the pace, and
 *                  TMA stores are faster); for any other C, 5 (16-bit C) or 2
 *                  (fp32 C).
 *   stream_k:      how the tiles past the last whole wave are shared:
 *                  0 = planner's choice; 1 = never (whole tiles only, spread
 *                  over as few clusters as keep the wave count); 2 = stream-K
 *                  over the leftover tiles plus one full wave (or all tiles
 *                  when there are fewer than clusters): their 64-deep K blocks
 *                  are cut into equal contiguous ranges, one per cluster;
 *                  3 = stream-K over every tile; 4 = stream-K over the
 *                  leftover tiles of the partial last wave only.
 *   multicast:     reserved, 0 or 1 (any other value is
 *                  HGEMM_ERR_INVALID_ARG). No operand tile is multicast
 *                  across the CTAs of a cluster: every TMA load lands in the
 *                  shared memory of the CTA that issues it.
 *   split_k:       CTAs per cluster that split each tile's K loop: 0 =
 *                  planner's choice, 1 = none, 2, 4 or 8 = a cluster of that
 *                  many single CTAs (cta_group 1, block_n 128 or 256, at least
 *                  32 columns per CTA; 16-bit dtypes; no stream-K) per tile. CTA r multiplies K blocks
 *                  [r n / s, (r + 1) n / s) of the tile's n; the fp32 partial
 *                  sums meet through distributed shared memory and each CTA
 *                  adds all of them, in rank order, for 1/s of the tile's
 *                  columns. Needs a cluster per tile (HGEMM_ERR_INVALID_ARG
 *                  otherwise).
 *   epi_warps:     epilogue warps per CTA: 0 = planner's choice, 8 (each
 *                  reads 64-column chunks of the accumulator), or 16 (32-column
 *                  chunks, twice the chunks in flight; a 16-bit C, i.e. fp16,
 *                  bf16 or fp8 with its bf16 C, on cta_group 1 with block_n
 *                  256 or cta_group 2 with block_n 224 or 256; no K split, no
 *                  stream-K). The planner takes 16 wherever those limits
 *                  allow, else 8. Any other value, or 16 outside those
 *                  limits, is HGEMM_ERR_INVALID_ARG.
 */
typedef struct {
    int32_t cta_group;
    int32_t block_n;
    int32_t group_m;
    int32_t max_clusters;
    int32_t store_mode;
    int32_t stream_k;
    int32_t multicast;
    int32_t split_k;
    int32_t epi_warps;
} hgemm_config_t;

/* hgemm with an explicit configuration (cfg may be NULL = all zero). */
hgemm_status_t hgemm_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                        hgemm_dtype_t dtype, const hgemm_config_t* cfg, void* stream);

/*
 * hgemm_noalloc_ex - hgemm_noalloc with a launch configuration (cfg may be
 * NULL, as for hgemm_ex). A stream-K schedule (cfg->stream_k 2-4) keeps its
 * fp32 partial sums and their marks in the fixed scratch array as well; the
 * planner itself never picks stream-K.
 */
hgemm_status_t hgemm_noalloc_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                                hgemm_dtype_t dtype, const hgemm_config_t* cfg, void* stream);

/*
 * hgemm_fp8 - the FP8 variant: C (bf16, M x N) = per-channel-scaled A.B.
 *
 * A (M x K) and B (K x N) are row-major 8-bit E4M3 or E5M2 patterns (dtype
 * HGEMM_E4M3 or HGEMM_E5M2, both operands the same format), C row-major
 * bfloat16. a_scale: device array of M fp32 factors, one per row of A;
 * b_scale: device array of N fp32 factors, one per column of B; either may be
 * NULL (all ones). Scale arrays are read only and need 4-byte alignment.
 * B is read in place, MN-major (a copy into the library's workspace only
 * when N is not a multiple of 16, the row pitch TMA needs);
 * tiles are (1, 64 | 128 | 256) or (2, 128 | 224 | 256). Errors as for hgemm();
 * a dtype other than HGEMM_E4M3 / HGEMM_E5M2 is HGEMM_ERR_INVALID_ARG.
 */
hgemm_status_t hgemm_fp8(const void* A, const void* B, void* C, const float* a_scale, const float* b_scale,
                         int64_t M, int64_t N, int64_t K, hgemm_dtype_t dtype, void* stream);

/* hgemm_fp8 with a forced launch configuration (see hgemm_config_t). */
hgemm_status_t hgemm_fp8_ex(const void* A, const void* B, void* C, const float* a_scale, const float* b_scale,
                            int64_t M, int64_t N, int64_t K, hgemm_dtype_t dtype, const hgemm_config_t* cfg,
                            void* stream);

/*
 * hgemm_fp8_blockscaled - the FP8 GEMM with one fp32 scale per sub-block
 * ("深度学习加速核心：GEMM优化从分块到TensorCore的实战解析", section 4.3: FP8
 * data is scaled block-wise, one factor per 32 x 32 or 64 x 64 sub-block;
 * section 5.2, the third mishap: the factors must be 32-bit, a 16-bit one
 * overflowed to infinity):
 *
 *     C[i][j] = round_to_nearest_even_bf16( sum_k A64[i][k] * B64[k][j] )
 *     A64[i][k] = A[i][k] * a_scale[i / block][k / block]
 *     B64[k][j] = B[k][j] * b_scale[k / block][j / block]
 *
 * A (M x K) and B (K x N): row-major 8-bit E4M3 or E5M2 patterns (dtype
 * HGEMM_E4M3 or HGEMM_E5M2, one format for both), device. C: row-major
 * bfloat16 (M x N), device, written. block: 32 or 64. a_scale: device fp32
 * array of ceil(M / block) x ceil(K / block) factors, row-major (factor of A's
 * sub-block (i / block, k / block)); b_scale: device fp32 array of
 * ceil(K / block) x ceil(N / block) factors, row-major. Both are read only,
 * 4-byte aligned, owned by the caller; a partial last block of a dimension
 * has one factor like the others.
 *
 * Each block's products are summed in fp32 by the tensor cores, multiplied
 * by its factor a_scale * b_scale (formed in fp32) and added into an fp32
 * accumulator; C is that accumulator rounded once. Tiles are 128 x 128 (one
 * CTA) or 256 x 128 (a CTA pair). A or B whose row pitch is not a multiple
 * of 16 bytes (K or N not a multiple of 16) is copied into the library's
 * stream-ordered workspace first, as for hgemm(). Errors as for hgemm(); a
 * dtype other than HGEMM_E4M3 / HGEMM_E5M2, a block other than 32 or 64, or
 * a NULL or misaligned scale array (with M, N, K > 0) is
 * HGEMM_ERR_INVALID_ARG. K == 0 writes zeros to C.
 */
hgemm_status_t hgemm_fp8_blockscaled(const void* A, const void* B, void* C, const float* a_scale,
                                     const float* b_scale, int64_t M, int64_t N, int64_t K, int32_t block,
                                     hgemm_dtype_t dtype, void* stream);

/*
 * hgemm_fp8_blockscaled with a forced configuration: cta_group (1 or 2),
 * group_m and max_clusters are honoured; block_n must be 0 or 128, split_k
 * and stream_k 0 or 1, store_mode 0 (HGEMM_ERR_INVALID_ARG otherwise).
 */
hgemm_status_t hgemm_fp8_blockscaled_ex(const void* A, const void* B, void* C, const float* a_scale,
                                        const float* b_scale, int64_t M, int64_t N, int64_t K, int32_t block,
                                        hgemm_dtype_t dtype, const hgemm_config_t* cfg, void* stream);

/*
 * hgemm_host - the same product for operands in HOST memory.
 *
 * hA, hB: host operands; hC: host result. dA, dB, dC: caller-owned device
 * buffers of at least M*K, K*N and M*N elements of the operand / result
 * type. After the work already enqueued on `stream`, it copies hB->dB and then,
 * in row bands (up to 4 of at least 512 rows, for M >= 1024), copies each band
 * of hA into dA,
 * multiplies it (hgemm on that band) and copies the band of dC back to hC:
 * band copies in, band GEMMs and band copies out run on three internal streams
 * (created once per device), so they overlap. It then makes `stream` wait for
 * the last copy out and synchronises it, so hC holds the result when it
 * returns HGEMM_OK. Host buffers should be page-locked for the copies to run
 * asynchronously. Concurrent calls share the internal streams.
 */
hgemm_status_t hgemm_host(const void* hA, const void* hB, void* hC, int64_t M, int64_t N,
                          int64_t K, hgemm_dtype_t dtype, void* dA, void* dB, void* dC,
                          void* stream);

/*
 * Planner output for a problem (host-only; needs no GPU unless sm_count is 0,
 * in which case the current device is queried).
 */
typedef struct {
    int32_t cta_group;     /* 1 or 2 */
    int32_t block_m;       /* rows of C per tile: 128 * cta_group */
    int32_t block_n;       /* columns of C per tile */
    int32_t block_k;       /* K per pipeline stage (64) */
    int32_t stages;        /* depth of the shared-memory ring */
    int32_t group_m;       /* raster group height in tiles */
    int32_t tiles_m;       /* ceil(M / block_m) */
    int32_t tiles_n;       /* ceil(N / block_n) */
    int32_t num_tiles;     /* tiles_m * tiles_n */
    int32_t grid_ctas;     /* CTAs launched (a multiple of cta_group * split_k) */
    int32_t smem_bytes;    /* dynamic shared memory per CTA */
    int32_t tmem_cols;     /* tensor-memory columns allocated per CTA */
    int32_t repack_a;      /* 1 if A goes through the workspace (rows padded to 128 bytes) */
    int32_t repack_b;      /* 1 if B does (B is otherwise read in place, MN-major, for every dtype) */
    int32_t store_mode;    /* 1 = TMA, 2 = plain, 3 = vector, 4 = staged vector, 5 = realigned staged stores */
    int32_t dp_tiles;      /* tiles computed whole, round-robin (the first dp_tiles in raster order) */
    int32_t sk_tiles;      /* tiles after them shared by stream-K ranges (0 = none) */
    int32_t sk_blocks;     /* K blocks per cluster in the stream-K phase (the first
                              sk_extra clusters take one more) */
    int32_t sk_extra;
    int32_t num_kb;        /* 64-deep K blocks per tile: ceil(K / 64) */
    int32_t multicast;     /* always 1 (reserved; no operand multicast) */
    int32_t split_k;       /* CTAs per cluster splitting a tile's K loop (1 = none). A
                              planner-chosen split needs one resident cluster per tile; where
                              fewer fit on the device, the launch takes half the split on the
                              same tiles, then whole tiles (see hgemm_plan) */
    int64_t workspace_bytes; /* stream-ordered workspace: repacked operands + fp32 partials */
    int32_t epi_warps;     /* epilogue warps per CTA (8 or 16) */
} hgemm_plan_t;

/* Fill *out with the plan hgemm_ex would use (pointers are assumed 16-byte
 * aligned). sm_count <= 0 plans for the current device, after the K-split
 * fallback above (the split the launch keeps). sm_count > 0 plans for that
 * many SMs without touching a device and assumes a cluster per tile fits. */
hgemm_status_t hgemm_plan(int64_t M, int64_t N, int64_t K, hgemm_dtype_t dtype,
                          const hgemm_config_t* cfg, int32_t sm_count, hgemm_plan_t* out);

/*
 * The i-th work unit of cluster `cluster` under `plan` (host copy of the
 * device schedule): K blocks [*kb0, *kb1) of tile *tile; *kind 0 = whole tile,
 * 1 = stream-K part owning the tile (holds K block 0; adds the partners'
 * partial sums), 2 = other stream-K part. Returns 0 when the cluster has no
 * i-th unit (then the outputs are untouched), 1 otherwise.
 */
int32_t hgemm_work_unit(const hgemm_plan_t* plan, int32_t cluster, int32_t i, int32_t* tile,
                        int32_t* kb0, int32_t* kb1, int32_t* kind);

/*
 * Tile raster used by every CTA role (host copy of the device function).
 * Tile index t in [0, tiles_m*tiles_n) maps to tile row *tm and column *tn:
 * tiles are taken in groups of group_m tile rows; inside a group the row index
 * varies fastest ("[CUDA 优化实战] hgemm - 超越 cuBLAS", section 1, grid
 * swizzling with SWIZZLE_W: neighbouring CTAs share operand panels in L2).
 */
void hgemm_tile_coord(int32_t t, int32_t tiles_m, int32_t tiles_n, int32_t group_m,
                      int32_t* tm, int32_t* tn);

/*
 * The K blocks [*lo, *hi) of a tile's range [kb0, kb1) that rank `rank` of a
 * K-split cluster of `parts` CTAs multiplies (host copy of the device
 * function; see hgemm_config_t.split_k): contiguous shares in rank order,
 * equal to within one block. Leaves *lo and *hi untouched unless
 * 0 <= rank < parts and kb0 <= kb1.
 */
void hgemm_split_share(int32_t kb0, int32_t kb1, int32_t rank, int32_t parts, int32_t* lo, int32_t* hi);

/*
 * Device-side status word of `device`, set by a kernel whose bounded wait ran
 * out (HGEMM_ERR_TIMEOUT) and left unchanged otherwise. Call after the stream
 * that ran the GEMM has been synchronised. *info (may be NULL) receives the
 * role and barrier that timed out. reset != 0 clears the word. Synchronous.
 */
hgemm_status_t hgemm_get_device_status(int32_t device, int32_t reset, uint32_t* info);

/* Upper bound, in nanoseconds, on any single wait inside the kernels
 * (default 2e9). Applies to launches made after the call, from any thread. */
void hgemm_set_timeout_ns(uint64_t ns);

/*
 * Test hook for the failure path (not for production use; affects launches
 * made after the call, from any thread, until reset with 0).
 * kind 1: in each launch with a stream-K phase, the CTAs owning a tile shared
 * across clusters wait for partial sums that are never published. Each such
 * wait runs out after the timeout set by hgemm_set_timeout_ns; the kernel
 * records HGEMM_ERR_TIMEOUT in the device status word, writes those tiles
 * without the missing parts, and returns normally. An owner's unit is the last
 * of its CTA, so the waiting CTAs have no copies or MMAs in flight, and
 * nothing traps or hangs.
 * kind 2: in each launch with a K split within clusters (split_k > 1), the
 * first CTA of every cluster withholds its "ring free" arrival, so its peers'
 * bounded waits run out. Each CTA records HGEMM_ERR_TIMEOUT, skips the rest
 * of the reduction (C is left partly unwritten) and returns normally. By
 * then every CTA's MMAs have completed, so nothing is in flight.
 */
void hgemm_test_inject(int32_t kind);

/* Static text for a status code. */
const char* hgemm_status_string(hgemm_status_t s);

/* Text of the last CUDA error seen by an entry point on this thread ("" if none). */
const char* hgemm_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t hgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HGEMM_H_ */
