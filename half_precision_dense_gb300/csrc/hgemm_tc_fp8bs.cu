// Instantiations of the block-scaled FP8 GEMM kernel (hgemm_fp8bs.cuh):
// E4M3 or E5M2 operands, scale blocks of 32 or 64, single CTAs or CTA pairs.
#include "hgemm_fp8bs.cuh"
#include "tc_instances.cuh"

namespace hg {

template <int CG, int kGs, int kDt>
using Fp8bsInstance = ClusterKernel<&hgemm_fp8bs_kernel<CG, kGs, kDt>, CG, Fp8bsCfg<CG>::kSmemBytes, kBsThreads>;

#define HG_FP8BS_DISPATCH(CALL)                                                               \
    if (kind == 3 && cta_group == 1 && gs == 32) return Fp8bsInstance<1, 32, 3>::CALL;        \
    if (kind == 3 && cta_group == 1 && gs == 64) return Fp8bsInstance<1, 64, 3>::CALL;        \
    if (kind == 3 && cta_group == 2 && gs == 32) return Fp8bsInstance<2, 32, 3>::CALL;        \
    if (kind == 3 && cta_group == 2 && gs == 64) return Fp8bsInstance<2, 64, 3>::CALL;        \
    if (kind == 4 && cta_group == 1 && gs == 32) return Fp8bsInstance<1, 32, 4>::CALL;        \
    if (kind == 4 && cta_group == 1 && gs == 64) return Fp8bsInstance<1, 64, 4>::CALL;        \
    if (kind == 4 && cta_group == 2 && gs == 32) return Fp8bsInstance<2, 32, 4>::CALL;        \
    if (kind == 4 && cta_group == 2 && gs == 64) return Fp8bsInstance<2, 64, 4>::CALL;

cudaError_t launch_fp8bs(int kind, int cta_group, int gs, const CUtensorMap& a, const CUtensorMap& b,
                         const CUtensorMap& b2, const Fp8bsParams& p, int clusters, cudaStream_t stream) {
    HG_FP8BS_DISPATCH(launch(clusters, stream, p.pdl != 0, a, b, b2, p))
    return cudaErrorInvalidValue;
}

int max_active_clusters_fp8bs(int kind, int cta_group, int gs) {
    HG_FP8BS_DISPATCH(max_clusters())
    return 0;
}

int fp8bs_stages(int cta_group) {
    return cta_group == 2 ? Fp8bsCfg<2>::kStages : Fp8bsCfg<1>::kStages;
}

int fp8bs_smem_bytes(int cta_group) {
    return cta_group == 2 ? Fp8bsCfg<2>::kSmemBytes : Fp8bsCfg<1>::kSmemBytes;
}

int fp8bs_tmem_cols() { return Fp8bsCfg<1>::kTmemCols; }

}  // namespace hg
