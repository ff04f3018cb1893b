// gemm_bf16.cu -- BF16 (kind::f16, FP32 accumulation, no scales) instantiations
// of the persistent GEMM kernels: the same TMA ring, TMEM accumulator, warp
// roles and epilogue as the MX GEMM, with 64 BF16 values of K per 128-byte
// stage row and four K = 16 MMAs per stage.
#include "gemm_kernel_pair.cuh"
#include "launch.h"

namespace mxg {

namespace {
template <int BN>
cudaError_t launch(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, int grid, cudaStream_t s)
{
    using C = Cfg<K_BF16, BN>;
    if constexpr (BN == 256) {
        if (p.sk_ctas > 0) {  // stream-K plans: the instantiation with fixup warps
            mx_gemm_kernel<K_BF16, BN, false, true><<<grid, kThreadsSk, C::kSmemBytes, s>>>(p, ma, mb);
            return cudaGetLastError();
        }
    }
    mx_gemm_kernel<K_BF16, BN><<<grid, kThreads, C::kSmemBytes, s>>>(p, ma, mb);
    return cudaGetLastError();
}

cudaLaunchConfig_t cluster2_config(int clusters, int smem, cudaStream_t s, cudaLaunchAttribute *attr,
                                   int threads)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int BN>
cudaError_t launch_pair(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &msa,
                        const CUtensorMap &msb, int clusters, cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    if constexpr (BN == 256) {
        if (p.sk_ctas > 0) {  // stream-K plans: the instantiation with fixup warps
            auto kern = mx_gemm_pair_kernel<K_BF16, BN, true>;
            cudaLaunchConfig_t cfg = cluster2_config(clusters, CfgPair<K_BF16, BN>::kSmemBytes, s, attr, kThreadsSk);
            return cudaLaunchKernelEx(&cfg, kern, p, ma, mb, msa, msb);
        }
    }
    auto kern = mx_gemm_pair_kernel<K_BF16, BN>;
    cudaLaunchConfig_t cfg = cluster2_config(clusters, CfgPair<K_BF16, BN>::kSmemBytes, s, attr, kThreads);
    return cudaLaunchKernelEx(&cfg, kern, p, ma, mb, msa, msb);
}

template <int BN>
int pair_max_clusters()
{
    auto kern = mx_gemm_pair_kernel<K_BF16, BN>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CfgPair<K_BF16, BN>::kSmemBytes) !=
        cudaSuccess)
        return 0;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster2_config(1, CfgPair<K_BF16, BN>::kSmemBytes, nullptr, attr, kThreads);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess)
        return 0;
    return n;
}

template <int BN>
KernelInfo pair_info()
{
    using C = CfgPair<K_BF16, BN>;
    return KernelInfo{C::kStages, C::kAccStages, C::kSmemBytes};
}

template <int BN>
KernelInfo info()
{
    using C = Cfg<K_BF16, BN>;
    return KernelInfo{C::kStages, C::kAccStages, C::kSmemBytes};
}
}  // namespace

cudaError_t prepare_gemm_bf16()
{
    const void *k[8] = {(const void *)mx_gemm_kernel<K_BF16, 32>,
                        (const void *)mx_gemm_kernel<K_BF16, 64>,
                        (const void *)mx_gemm_kernel<K_BF16, 128>,
                        (const void *)mx_gemm_kernel<K_BF16, 256>,
                        (const void *)mx_gemm_kernel<K_BF16, 256, false, true>,
                        (const void *)mx_gemm_pair_kernel<K_BF16, 128>,
                        (const void *)mx_gemm_pair_kernel<K_BF16, 256>,
                        (const void *)mx_gemm_pair_kernel<K_BF16, 256, true>};
    const int smem[8] = {Cfg<K_BF16, 32>::kSmemBytes,      Cfg<K_BF16, 64>::kSmemBytes,      Cfg<K_BF16, 128>::kSmemBytes,
                         Cfg<K_BF16, 256>::kSmemBytes,     Cfg<K_BF16, 256>::kSmemBytes,     CfgPair<K_BF16, 128>::kSmemBytes,
                         CfgPair<K_BF16, 256>::kSmemBytes, CfgPair<K_BF16, 256>::kSmemBytes};
    for (int i = 0; i < 8; ++i) {
        cudaError_t e = cudaFuncSetAttribute(k[i], cudaFuncAttributeMaxDynamicSharedMemorySize, smem[i]);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemm_bf16(int bn, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, int grid,
                             cudaStream_t s)
{
    switch (bn) {
    case 32: return launch<32>(p, ma, mb, grid, s);
    case 64: return launch<64>(p, ma, mb, grid, s);
    case 128: return launch<128>(p, ma, mb, grid, s);
    case 256: return launch<256>(p, ma, mb, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm_pair_bf16(int bn, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                  const CUtensorMap &msa, const CUtensorMap &msb, int clusters, cudaStream_t s)
{
    switch (bn) {
    case 128: return launch_pair<128>(p, ma, mb, msa, msb, clusters, s);
    case 256: return launch_pair<256>(p, ma, mb, msa, msb, clusters, s);
    default: return cudaErrorInvalidValue;
    }
}

int gemm_pair_max_clusters_bf16(int bn) { return bn == 128 ? pair_max_clusters<128>() : pair_max_clusters<256>(); }

KernelInfo gemm_pair_info_bf16(int bn) { return bn == 128 ? pair_info<128>() : pair_info<256>(); }

KernelInfo gemm_info_bf16(int bn)
{
    switch (bn) {
    case 32: return info<32>();
    case 64: return info<64>();
    case 128: return info<128>();
    default: return info<256>();
    }
}

}  // namespace mxg
