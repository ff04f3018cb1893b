// gemm_bf16.cu -- BF16 (kind::f16, FP32 accumulation, no scales) instantiations
// of the persistent GEMM kernels: the same TMA ring, TMEM accumulator, warp
// roles and epilogue as the MX GEMM, with 64 BF16 values of K per 128-byte
// stage row and four K = 16 MMAs per stage.
#include "launch_impl.cuh"

namespace mxg {

using L = Launchers<K_BF16>;

cudaError_t prepare_gemm_bf16() { return L::prepare(); }

cudaError_t launch_gemm_bf16(int bn, bool lean, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                             int grid, cudaStream_t s)
{
    return L::launch_single(bn, lean, p, ma, mb, grid, s);
}

cudaError_t launch_gemm_pair_bf16(int bn, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                  const CUtensorMap &msa, const CUtensorMap &msb, const CUtensorMap &msarm, int clusters, cudaStream_t s)
{
    return L::launch_pair(bn, p, ma, mb, msa, msb, msarm, clusters, s);
}

int gemm_pair_max_clusters_bf16(int bn) { return L::max_clusters(bn); }

KernelInfo gemm_pair_info_bf16(int bn) { return L::pair_info(bn); }

KernelInfo gemm_info_bf16(int bn, bool lean) { return L::info(bn, lean); }

}  // namespace mxg
