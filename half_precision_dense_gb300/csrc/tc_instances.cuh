// tc_instances.cuh - host launch helpers for the kernel instantiations of one
// dtype. Included once by hgemm_tc_bf16.cu and once by hgemm_tc_f16.cu so the
// two dtypes compile in parallel.
#pragma once

#include <mutex>

#include "launch.h"

namespace hg {

// Launch bookkeeping of one persistent cluster kernel: the dynamic
// shared-memory opt-in (per device, set once), the launch configuration
// (one cluster of kCluster CTAs per work slot) and the resident clusters
// (queried once per device).
template <auto kKernel, int kCluster, int kSmemBytes, int kBlockThreads = kThreads>
struct ClusterKernel {
    static cudaError_t prepare() {
        static std::mutex mu;
        static uint64_t done_mask = 0;
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        std::lock_guard<std::mutex> lk(mu);
        const uint64_t bit = 1ull << (dev & 63);
        if (done_mask & bit) return cudaSuccess;
        e = cudaFuncSetAttribute(kKernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e == cudaSuccess) done_mask |= bit;
        return e;
    }

    // `pdl`: programmatic dependent launch, the kernel may start before the
    // preceding kernel on the stream ends (it waits with griddepcontrol.wait
    // before reading global memory).
    static void fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int clusters,
                            cudaStream_t stream, bool pdl = false) {
        cfg = cudaLaunchConfig_t{};
        cfg.gridDim = dim3(static_cast<unsigned>(clusters * kCluster), 1, 1);
        cfg.blockDim = dim3(kBlockThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = stream;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kCluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 2 : 1;
    }

    template <typename... Args>
    static cudaError_t launch(int clusters, cudaStream_t stream, bool pdl, const Args&... args) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[2];
        fill_config(cfg, attr, clusters, stream, pdl);
        return cudaLaunchKernelEx(&cfg, kKernel, args...);
    }

    static int max_clusters() {
        static std::mutex mu;
        static int cache[64] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
        {
            std::lock_guard<std::mutex> lk(mu);
            if (cache[dev] > 0) return cache[dev];
        }
        if (prepare() != cudaSuccess) return 0;
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[2];
        fill_config(cfg, attr, 1, nullptr);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kKernel, &cfg) != cudaSuccess) return 0;
        std::lock_guard<std::mutex> lk(mu);
        cache[dev] = n;
        return n;
    }
};

template <int CG, int BN, int kDt, int MC = 1, int EW = kEpiWarps>
struct TcInstance {
    // The kernel's own configuration (its operand size sets the stage bytes
    // and the ring depth), so the launch reserves the shared memory it uses.
    using Cfg = TcCfg<CG, BN, elem_bytes(kDt), (CG == 1 && MC > 1) ? MC : 1>;
    using K = ClusterKernel<&hgemm_tc_kernel<CG, BN, kDt, MC, EW>, CG * MC, Cfg::kSmemBytes, 32 * (EW + 3)>;

    static cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                              const CUtensorMap& c32, const CUtensorMap& b2, const TcParams& p, int clusters,
                              cudaStream_t stream) {
        return K::launch(clusters, stream, p.pdl != 0, a, b, c, c32, b2, p);
    }

    static int max_clusters() { return K::max_clusters(); }
    static bool exists() { return true; }   // host-only: the instance is compiled
};

// Every tile shape of the 16-bit kinds (KDT 0 = fp16, 1 = bf16), the K split
// across 2, 4 or 8 single CTAs (mc with cta_group 1), and the single 256-wide
// and pair 224- and 256-wide tiles with 16 epilogue warps (epi == 16).
#define HG_TC_DISPATCH(KDT, CALL)                                                          \
    if (epi == 16 && mc == 1 && cta_group == 1 && block_n == 256)                          \
        return TcInstance<1, 256, KDT, 1, 16>::CALL;                                       \
    if (epi == 16 && mc == 1 && cta_group == 2 && block_n == 224)                          \
        return TcInstance<2, 224, KDT, 1, 16>::CALL;                                       \
    if (epi == 16 && mc == 1 && cta_group == 2 && block_n == 256)                          \
        return TcInstance<2, 256, KDT, 1, 16>::CALL;                                       \
    if (epi == 8 && mc == 1 && cta_group == 1 && block_n == 64) return TcInstance<1, 64, KDT>::CALL; \
    if (epi == 8 && mc == 1 && cta_group == 1 && block_n == 128) return TcInstance<1, 128, KDT>::CALL; \
    if (epi == 8 && mc == 1 && cta_group == 1 && block_n == 256) return TcInstance<1, 256, KDT>::CALL; \
    if (epi == 8 && mc == 1 && cta_group == 2 && block_n == 128) return TcInstance<2, 128, KDT>::CALL; \
    if (epi == 8 && mc == 1 && cta_group == 2 && block_n == 224) return TcInstance<2, 224, KDT>::CALL; \
    if (epi == 8 && mc == 1 && cta_group == 2 && block_n == 256) return TcInstance<2, 256, KDT>::CALL; \
    if (epi == 8 && mc == 2 && cta_group == 1 && block_n == 128) return TcInstance<1, 128, KDT, 2>::CALL; \
    if (epi == 8 && mc == 4 && cta_group == 1 && block_n == 128) return TcInstance<1, 128, KDT, 4>::CALL; \
    if (epi == 8 && mc == 2 && cta_group == 1 && block_n == 256) return TcInstance<1, 256, KDT, 2>::CALL; \
    if (epi == 8 && mc == 4 && cta_group == 1 && block_n == 256) return TcInstance<1, 256, KDT, 4>::CALL; \
    if (epi == 8 && mc == 8 && cta_group == 1 && block_n == 256) return TcInstance<1, 256, KDT, 8>::CALL;

// The tf32 (KDT 2) and fp8 (KDT 3 = E4M3, 4 = E5M2) tile shapes: no K split,
// 8 epilogue warps (and 16 for fp8, below).
#define HG_TC_DISPATCH_K(KDT, CALL)                                                        \
    if (epi == 8 && mc == 1 && cta_group == 1 && block_n == 64) return TcInstance<1, 64, KDT>::CALL;   \
    if (epi == 8 && mc == 1 && cta_group == 1 && block_n == 128) return TcInstance<1, 128, KDT>::CALL; \
    if (epi == 8 && mc == 1 && cta_group == 1 && block_n == 256) return TcInstance<1, 256, KDT>::CALL; \
    if (epi == 8 && mc == 1 && cta_group == 2 && block_n == 128) return TcInstance<2, 128, KDT>::CALL; \
    if (epi == 8 && mc == 1 && cta_group == 2 && block_n == 256) return TcInstance<2, 256, KDT>::CALL;
// tf32 and fp8 also take the 224-wide pair tile.
#define HG_TC_DISPATCH_W(KDT, CALL)                                                       \
    HG_TC_DISPATCH_K(KDT, CALL)                                                            \
    if (epi == 8 && mc == 1 && cta_group == 2 && block_n == 224) return TcInstance<2, 224, KDT>::CALL;
#define HG_TC_DISPATCH_TF32(CALL) HG_TC_DISPATCH_W(2, CALL)
// fp8 writes a bf16 C: 16 epilogue warps on the single 256-wide and pair
// 224- and 256-wide tiles, as for the 16-bit kinds.
#define HG_TC_DISPATCH_F8(KDT, CALL)                                                      \
    HG_TC_DISPATCH_W(KDT, CALL)                                                            \
    if (epi == 16 && mc == 1 && cta_group == 1 && block_n == 256)                          \
        return TcInstance<1, 256, KDT, 1, 16>::CALL;                                       \
    if (epi == 16 && mc == 1 && cta_group == 2 && block_n == 224)                          \
        return TcInstance<2, 224, KDT, 1, 16>::CALL;                                       \
    if (epi == 16 && mc == 1 && cta_group == 2 && block_n == 256)                          \
        return TcInstance<2, 256, KDT, 1, 16>::CALL;

}  // namespace hg
