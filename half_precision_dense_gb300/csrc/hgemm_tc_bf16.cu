// bf16 instantiations of the tcgen05 GEMM kernel.
#include "tc_instances.cuh"

namespace hg {

cudaError_t launch_tc_bf16(int cta_group, int block_n, int mc, int epi, const CUtensorMap& a, const CUtensorMap& b,
                           const CUtensorMap& c, const CUtensorMap& c32, const CUtensorMap& b2, const TcParams& p, int clusters,
                           cudaStream_t stream) {
    HG_TC_DISPATCH(1, launch(a, b, c, c32, b2, p, clusters, stream))
    return cudaErrorInvalidValue;
}

int max_active_clusters_bf16(int cta_group, int block_n, int mc, int epi) {
    HG_TC_DISPATCH(1, max_clusters())
    return 0;
}

bool tc_instance_exists_bf16(int cta_group, int block_n, int mc, int epi) {
    HG_TC_DISPATCH(1, exists())
    return false;
}

}  // namespace hg
