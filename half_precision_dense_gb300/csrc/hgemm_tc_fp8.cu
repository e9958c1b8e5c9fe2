// fp8 instantiations of the tcgen05 GEMM kernel (E4M3 or E5M2 operands, bf16 C).
#include "tc_instances.cuh"

namespace hg {

cudaError_t launch_tc_fp8(int kind, int cta_group, int block_n, int mc, int epi, const CUtensorMap& a,
                          const CUtensorMap& b, const CUtensorMap& c, const CUtensorMap& c32, const CUtensorMap& b2,
                          const TcParams& p, int clusters, cudaStream_t stream) {
    if (kind == 3) {
        HG_TC_DISPATCH_F8(3, launch(a, b, c, c32, b2, p, clusters, stream))
    } else if (kind == 4) {
        HG_TC_DISPATCH_F8(4, launch(a, b, c, c32, b2, p, clusters, stream))
    }
    return cudaErrorInvalidValue;
}

int max_active_clusters_fp8(int kind, int cta_group, int block_n, int mc, int epi) {
    if (kind == 3) {
        HG_TC_DISPATCH_F8(3, max_clusters())
    } else if (kind == 4) {
        HG_TC_DISPATCH_F8(4, max_clusters())
    }
    return 0;
}

bool tc_instance_exists_fp8(int kind, int cta_group, int block_n, int mc, int epi) {
    if (kind == 3) {
        HG_TC_DISPATCH_F8(3, exists())
    } else if (kind == 4) {
        HG_TC_DISPATCH_F8(4, exists())
    }
    return false;
}

}  // namespace hg
