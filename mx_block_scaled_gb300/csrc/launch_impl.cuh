// launch_impl.cuh -- the launchers of every GEMM instantiation of one element
// kind (MXFP8, MXFP4 or BF16), shared by gemm_fp8.cu, gemm_fp4.cu and
// gemm_bf16.cu.  Every GEMM launch allows programmatic dependent launch: its
// CTAs may become resident while the preceding kernel in the stream (the scale
// relayout, the quantiser, a previous GEMM) finishes, run their prologue
// (barriers, TMEM allocation, descriptor prefetch) and then wait in
// griddep_wait() before touching global memory.
#pragma once

#include <cuda_runtime.h>

#include "gemm_kernel_pair.cuh"
#include "launch.h"

namespace mxg {

template <int KIND>
struct Launchers {
    // Single-CTA 128 x BN tiles; plans with stream-K segments run the
    // instantiation with the two fixup warps, which add the segments of 128-
    // and 256-wide tiles (narrower tiles and the lean form add them in their
    // epilogue warps).
    template <int BN, bool LEAN = false>
    static cudaError_t single(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, int grid, cudaStream_t s)
    {
        cudaLaunchAttribute attr[2];
        constexpr int kSmem = Cfg<KIND, BN, LEAN>::kSmemBytes;
        if (p.sk_ctas > 0) {
            cudaLaunchConfig_t cfg = launch_config(grid, LEAN ? kLeanThreads : kThreadsSk, kSmem, s, attr, 1);
            return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<KIND, BN, false, true, LEAN>, p, ma, mb);
        }
        cudaLaunchConfig_t cfg = launch_config(grid, LEAN ? kLeanThreads : kThreads, kSmem, s, attr, 1);
        return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<KIND, BN, false, false, LEAN>, p, ma, mb);
    }

    template <int BN>
    static cudaError_t grouped(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, int grid,
                               cudaStream_t s)
    {
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = launch_config(grid, kThreads, Cfg<KIND, BN>::kSmemBytes, s, attr, 1);
        return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<KIND, BN, true>, p, ma, mb);
    }

    // 256 x BN tiles on CTA pairs (clusters of two).
    template <int BN>
    static cudaError_t pair(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &msa,
                            const CUtensorMap &msb, const CUtensorMap &msarm, int clusters, cudaStream_t s)
    {
        cudaLaunchAttribute attr[2];
        if constexpr (BN == 256) {
            if (p.sk_ctas > 0) {
                cudaLaunchConfig_t cfg =
                    launch_config(2 * clusters, kThreads, CfgPair<KIND, BN>::kSmemBytes, s, attr, 2);
                return cudaLaunchKernelEx(&cfg, mx_gemm_pair_kernel<KIND, BN, true>, p, ma, mb, msa, msb, msarm);
            }
        }
        cudaLaunchConfig_t cfg = launch_config(2 * clusters, kThreads, CfgPair<KIND, BN>::kSmemBytes, s, attr, 2);
        return cudaLaunchKernelEx(&cfg, mx_gemm_pair_kernel<KIND, BN>, p, ma, mb, msa, msb, msarm);
    }

    // Grouped (mixture-of-experts) GEMM on 256 x 256 CTA-pair tiles (the
    // tokens' 256-row tiles inside each group), on `clusters` clusters.
    static cudaError_t grouped_pair(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                    const CUtensorMap &msa, const CUtensorMap &msb, int clusters, cudaStream_t s)
    {
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg =
            launch_config(2 * clusters, kThreads, CfgPair<KIND, 256, true>::kSmemBytes, s, attr, 2);
        return cudaLaunchKernelEx(&cfg, mx_gemm_pair_kernel<KIND, 256, false, true>, p, ma, mb, msa, msb, msa);
    }

    // Co-resident clusters of two of the pair kernel (its work slots).
    template <int BN, bool GROUPED = false>
    static int pair_max_clusters()
    {
        auto kern = mx_gemm_pair_kernel<KIND, BN, false, GROUPED>;
        constexpr int kSmem = CfgPair<KIND, BN, GROUPED>::kSmemBytes;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
            return 0;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = launch_config(2, kThreads, kSmem, nullptr, attr, 2, false);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess)
            return 0;
        return n;
    }

    template <typename K>
    static cudaError_t opt_in(K kern, int smem)
    {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    }

    // Opt every instantiation into its shared-memory size (once per device;
    // called when a plan is created, never on the launch path).
    static cudaError_t prepare()
    {
        cudaError_t e = cudaSuccess;
        auto chk = [&](cudaError_t r) {
            if (e == cudaSuccess)
                e = r;
        };
        chk(opt_in(mx_gemm_kernel<KIND, 32>, Cfg<KIND, 32>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 64>, Cfg<KIND, 64>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 128>, Cfg<KIND, 128>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 256>, Cfg<KIND, 256>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 32, false, true>, Cfg<KIND, 32>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 64, false, true>, Cfg<KIND, 64>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 128, false, true>, Cfg<KIND, 128>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 256, false, true>, Cfg<KIND, 256>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 32, false, false, true>, Cfg<KIND, 32, true>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 64, false, false, true>, Cfg<KIND, 64, true>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 32, false, true, true>, Cfg<KIND, 32, true>::kSmemBytes));
        chk(opt_in(mx_gemm_kernel<KIND, 64, false, true, true>, Cfg<KIND, 64, true>::kSmemBytes));
        chk(opt_in(mx_gemm_pair_kernel<KIND, 128>, CfgPair<KIND, 128>::kSmemBytes));
        chk(opt_in(mx_gemm_pair_kernel<KIND, 192>, CfgPair<KIND, 192>::kSmemBytes));
        chk(opt_in(mx_gemm_pair_kernel<KIND, 256>, CfgPair<KIND, 256>::kSmemBytes));
        chk(opt_in(mx_gemm_pair_kernel<KIND, 256, true>, CfgPair<KIND, 256>::kSmemBytes));
        if constexpr (KIND != K_BF16) {
            chk(opt_in(mx_gemm_pair_kernel<KIND, 256, false, true>, CfgPair<KIND, 256, true>::kSmemBytes));
            chk(opt_in(mx_gemm_kernel<KIND, 64, true>, Cfg<KIND, 64>::kSmemBytes));
            chk(opt_in(mx_gemm_kernel<KIND, 128, true>, Cfg<KIND, 128>::kSmemBytes));
            chk(opt_in(mx_gemm_kernel<KIND, 256, true>, Cfg<KIND, 256>::kSmemBytes));
        }
        return e;
    }

    static cudaError_t launch_single(int bn, bool lean, const GemmParams &p, const CUtensorMap &ma,
                                     const CUtensorMap &mb, int grid, cudaStream_t s)
    {
        if (lean) {
            switch (bn) {
            case 32: return single<32, true>(p, ma, mb, grid, s);
            case 64: return single<64, true>(p, ma, mb, grid, s);
            default: return cudaErrorInvalidValue;
            }
        }
        switch (bn) {
        case 32: return single<32>(p, ma, mb, grid, s);
        case 64: return single<64>(p, ma, mb, grid, s);
        case 128: return single<128>(p, ma, mb, grid, s);
        case 256: return single<256>(p, ma, mb, grid, s);
        default: return cudaErrorInvalidValue;
        }
    }

    static cudaError_t launch_grouped(int bn, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                      int grid, cudaStream_t s)
    {
        switch (bn) {
        case 64: return grouped<64>(p, ma, mb, grid, s);
        case 128: return grouped<128>(p, ma, mb, grid, s);
        case 256: return grouped<256>(p, ma, mb, grid, s);
        default: return cudaErrorInvalidValue;
        }
    }

    static cudaError_t launch_pair(int bn, const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                   const CUtensorMap &msa, const CUtensorMap &msb, const CUtensorMap &msarm, int clusters,
                                   cudaStream_t s)
    {
        switch (bn) {
        case 128: return pair<128>(p, ma, mb, msa, msb, msarm, clusters, s);
        case 192: return pair<192>(p, ma, mb, msa, msb, msarm, clusters, s);
        case 256: return pair<256>(p, ma, mb, msa, msb, msarm, clusters, s);
        default: return cudaErrorInvalidValue;
        }
    }

    static int max_clusters(int bn)
    {
        return bn == 128 ? pair_max_clusters<128>() : bn == 192 ? pair_max_clusters<192>() : pair_max_clusters<256>();
    }

    template <int BN, bool LEAN = false>
    static KernelInfo single_info()
    {
        using C = Cfg<KIND, BN, LEAN>;
        return KernelInfo{C::kStages, C::kAccStages, C::kSmemBytes};
    }

    static KernelInfo info(int bn, bool lean)
    {
        if (lean)
            return bn == 32 ? single_info<32, true>() : single_info<64, true>();
        switch (bn) {
        case 32: return single_info<32>();
        case 64: return single_info<64>();
        case 128: return single_info<128>();
        default: return single_info<256>();
        }
    }

    template <int BN>
    static KernelInfo pair_info_of()
    {
        return KernelInfo{CfgPair<KIND, BN>::kStages, CfgPair<KIND, BN>::kAccStages, CfgPair<KIND, BN>::kSmemBytes};
    }

    static KernelInfo pair_info(int bn)
    {
        return bn == 128 ? pair_info_of<128>() : bn == 192 ? pair_info_of<192>() : pair_info_of<256>();
    }
};

}  // namespace mxg
