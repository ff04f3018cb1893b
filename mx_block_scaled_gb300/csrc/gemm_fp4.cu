// gemm_fp4.cu -- MXFP4 (E2M1 packed, kind::mxf4nvf4, scale_vec::2X) instantiations of
// the persistent block-scaled GEMM kernels.
#include "launch_impl.cuh"

namespace mxg {

using L = Launchers<K_MXFP4>;

cudaError_t prepare_gemm_fp4() { return L::prepare(); }

cudaError_t launch_gemm_fp4(int bn, bool lean, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                             int grid, cudaStream_t s)
{
    return L::launch_single(bn, lean, p, ma, mb, grid, s);
}

cudaError_t launch_gemm_grouped_fp4(int bn, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                    int grid, cudaStream_t s)
{
    return L::launch_grouped(bn, p, ma, mb, grid, s);
}

cudaError_t launch_gemm_pair_fp4(int bn, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                 const CUtensorMap &msa, const CUtensorMap &msb, const CUtensorMap &msarm, int clusters, cudaStream_t s)
{
    return L::launch_pair(bn, p, ma, mb, msa, msb, msarm, clusters, s);
}

int gemm_pair_max_clusters_fp4(int bn) { return L::max_clusters(bn); }

cudaError_t launch_gemm_grouped_pair_fp4(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                         const CUtensorMap &msa, const CUtensorMap &msb, int clusters, cudaStream_t s)
{
    return L::grouped_pair(p, ma, mb, msa, msb, clusters, s);
}

int gemm_grouped_pair_max_clusters_fp4() { return L::pair_max_clusters<256, true>(); }

KernelInfo gemm_grouped_pair_info_fp4()
{
    using C = CfgPair<K_MXFP4, 256, true>;
    return KernelInfo{C::kStages, C::kAccStages, C::kSmemBytes};
}

KernelInfo gemm_pair_info_fp4(int bn) { return L::pair_info(bn); }

KernelInfo gemm_info_fp4(int bn, bool lean) { return L::info(bn, lean); }

}  // namespace mxg
