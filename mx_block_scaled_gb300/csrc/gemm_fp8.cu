// gemm_fp8.cu -- MXFP8 (E4M3, kind::mxf8f6f4, scale_vec::1X) instantiations of
// the persistent block-scaled GEMM kernel.
#include "gemm_kernel_pair.cuh"
#include "launch.h"

namespace mxg {

namespace {
template <int BN>
cudaError_t launch(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, int grid, cudaStream_t s)
{
    using C = Cfg<K_MXFP8, BN>;
    if constexpr (BN == 256) {
        if (p.sk_ctas > 0) {  // stream-K plans: the instantiation with fixup warps
            mx_gemm_kernel<K_MXFP8, BN, false, true><<<grid, kThreadsSk, C::kSmemBytes, s>>>(p, ma, mb);
            return cudaGetLastError();
        }
    }
    mx_gemm_kernel<K_MXFP8, BN><<<grid, kThreads, C::kSmemBytes, s>>>(p, ma, mb);
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
            auto kern = mx_gemm_pair_kernel<K_MXFP8, BN, true>;
            cudaLaunchConfig_t cfg = cluster2_config(clusters, CfgPair<K_MXFP8, BN>::kSmemBytes, s, attr, kThreadsSk);
            return cudaLaunchKernelEx(&cfg, kern, p, ma, mb, msa, msb);
        }
    }
    auto kern = mx_gemm_pair_kernel<K_MXFP8, BN>;
    cudaLaunchConfig_t cfg = cluster2_config(clusters, CfgPair<K_MXFP8, BN>::kSmemBytes, s, attr, kThreads);
    return cudaLaunchKernelEx(&cfg, kern, p, ma, mb, msa, msb);
}

template <int BN>
int pair_max_clusters()
{
    auto kern = mx_gemm_pair_kernel<K_MXFP8, BN>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CfgPair<K_MXFP8, BN>::kSmemBytes) !=
        cudaSuccess)
        return 0;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster2_config(1, CfgPair<K_MXFP8, BN>::kSmemBytes, nullptr, attr, kThreads);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess)
        return 0;
    return n;
}

template <int BN>
cudaError_t launch_grouped(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, int grid, cudaStream_t s)
{
    using C = Cfg<K_MXFP8, BN>;
    mx_gemm_kernel<K_MXFP8, BN, true><<<grid, kThreads, C::kSmemBytes, s>>>(p, ma, mb);
    return cudaGetLastError();
}

template <int BN>
KernelInfo pair_info()
{
    using C = CfgPair<K_MXFP8, BN>;
    return KernelInfo{C::kStages, C::kAccStages, C::kSmemBytes};
}

template <int BN>
KernelInfo info()
{
    using C = Cfg<K_MXFP8, BN>;
    return KernelInfo{C::kStages, C::kAccStages, C::kSmemBytes};
}
}  // namespace

// Opt every instantiation into its shared-memory size (once per device; called
// when a plan is created, never on the launch path).
cudaError_t prepare_gemm_fp8()
{
    const void *single[5] = {(const void *)mx_gemm_kernel<K_MXFP8, 32>, (const void *)mx_gemm_kernel<K_MXFP8, 64>,
                             (const void *)mx_gemm_kernel<K_MXFP8, 128>, (const void *)mx_gemm_kernel<K_MXFP8, 256>,
                             (const void *)mx_gemm_kernel<K_MXFP8, 256, false, true>};
    const int single_smem[5] = {Cfg<K_MXFP8, 32>::kSmemBytes, Cfg<K_MXFP8, 64>::kSmemBytes, Cfg<K_MXFP8, 128>::kSmemBytes,
                                Cfg<K_MXFP8, 256>::kSmemBytes, Cfg<K_MXFP8, 256>::kSmemBytes};
    for (int i = 0; i < 5; ++i) {
        cudaError_t e = cudaFuncSetAttribute(single[i], cudaFuncAttributeMaxDynamicSharedMemorySize, single_smem[i]);
        if (e != cudaSuccess)
            return e;
    }
    const void *cl[3] = {(const void *)mx_gemm_pair_kernel<K_MXFP8, 128>, (const void *)mx_gemm_pair_kernel<K_MXFP8, 256>,
                         (const void *)mx_gemm_pair_kernel<K_MXFP8, 256, true>};
    const int cl_smem[3] = {CfgPair<K_MXFP8, 128>::kSmemBytes, CfgPair<K_MXFP8, 256>::kSmemBytes,
                            CfgPair<K_MXFP8, 256>::kSmemBytes};
    for (int i = 0; i < 3; ++i) {
        cudaError_t e = cudaFuncSetAttribute(cl[i], cudaFuncAttributeMaxDynamicSharedMemorySize, cl_smem[i]);
        if (e != cudaSuccess)
            return e;
    }
    const void *gr[3] = {(const void *)mx_gemm_kernel<K_MXFP8, 64, true>,
                         (const void *)mx_gemm_kernel<K_MXFP8, 128, true>,
                         (const void *)mx_gemm_kernel<K_MXFP8, 256, true>};
    const int gr_smem[3] = {Cfg<K_MXFP8, 64>::kSmemBytes, Cfg<K_MXFP8, 128>::kSmemBytes, Cfg<K_MXFP8, 256>::kSmemBytes};
    for (int i = 0; i < 3; ++i) {
        cudaError_t e = cudaFuncSetAttribute(gr[i], cudaFuncAttributeMaxDynamicSharedMemorySize, gr_smem[i]);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemm_fp8(int bn, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, int grid,
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

cudaError_t launch_gemm_grouped_fp8(int bn, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                    int grid, cudaStream_t s)
{
    switch (bn) {
    case 64: return launch_grouped<64>(p, ma, mb, grid, s);
    case 128: return launch_grouped<128>(p, ma, mb, grid, s);
    case 256: return launch_grouped<256>(p, ma, mb, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm_pair_fp8(int bn, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                 const CUtensorMap &msa, const CUtensorMap &msb, int clusters, cudaStream_t s)
{
    switch (bn) {
    case 128: return launch_pair<128>(p, ma, mb, msa, msb, clusters, s);
    case 256: return launch_pair<256>(p, ma, mb, msa, msb, clusters, s);
    default: return cudaErrorInvalidValue;
    }
}

int gemm_pair_max_clusters_fp8(int bn) { return bn == 128 ? pair_max_clusters<128>() : pair_max_clusters<256>(); }

KernelInfo gemm_pair_info_fp8(int bn) { return bn == 128 ? pair_info<128>() : pair_info<256>(); }

KernelInfo gemm_info_fp8(int bn)
{
    switch (bn) {
    case 32: return info<32>();
    case 64: return info<64>();
    case 128: return info<128>();
    default: return info<256>();
    }
}

}  // namespace mxg
