// launch.h -- internal interface between the host API (mxgemm.cu) and the
// translation units that instantiate the GEMM kernel (gemm_fp8.cu, gemm_fp4.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace mxg {

// Launch configuration: `grid` CTAs of `threads`, programmatic stream
// serialization allowed, and clusters of `cluster` CTAs when cluster > 1.
inline cudaLaunchConfig_t launch_config(int grid, int threads, int smem, cudaStream_t s, cudaLaunchAttribute (&attr)[2],
                                        int cluster, bool pdl = true)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cfg;
}

// Set the shared-memory opt-in of every GEMM instantiation on the current
// device.  Must run (once per device) before any launch below.
cudaError_t prepare_gemm_fp8();
cudaError_t prepare_gemm_fp4();
cudaError_t prepare_gemm_bf16();

// Launch the persistent GEMM kernel for tile width `bn` (32, 64, 128, 256) on
// `grid` CTAs; `lean` selects the lean decode form (bn 32 or 64).  Returns
// cudaErrorInvalidValue for an unsupported bn.
cudaError_t launch_gemm_fp8(int bn, bool lean, const GemmParams &p, const CUtensorMap &map_a,
                            const CUtensorMap &map_b, int grid, cudaStream_t stream);
cudaError_t launch_gemm_fp4(int bn, bool lean, const GemmParams &p, const CUtensorMap &map_a,
                            const CUtensorMap &map_b, int grid, cudaStream_t stream);

// Grouped (mixture-of-experts) form of the single-CTA kernel, bn = 64, 128 or
// 256 (p.grouped = 1), on `grid` CTAs.
cudaError_t launch_gemm_grouped_fp8(int bn, const GemmParams &p, const CUtensorMap &map_a, const CUtensorMap &map_b,
                                    int grid, cudaStream_t stream);
cudaError_t launch_gemm_grouped_fp4(int bn, const GemmParams &p, const CUtensorMap &map_a, const CUtensorMap &map_b,
                                    int grid, cudaStream_t stream);

// CTA-pair kernel (cluster of 2, cta_group::2), pair tile 256 x bn (bn = 128 or
// 256), on `clusters` clusters; it also takes 3-D maps of the two tile-layout
// scale tensors and, for p.sa_fused, a 2-D map of the row-major A-role scales.
// And the largest co-resident cluster count.
cudaError_t launch_gemm_pair_fp8(int bn, const GemmParams &p, const CUtensorMap &map_a, const CUtensorMap &map_b,
                                 const CUtensorMap &map_sfa, const CUtensorMap &map_sfb, const CUtensorMap &map_sarm, int clusters,
                                 cudaStream_t stream);
cudaError_t launch_gemm_pair_fp4(int bn, const GemmParams &p, const CUtensorMap &map_a, const CUtensorMap &map_b,
                                 const CUtensorMap &map_sfa, const CUtensorMap &map_sfb, const CUtensorMap &map_sarm, int clusters,
                                 cudaStream_t stream);
int gemm_pair_max_clusters_fp8(int bn);
int gemm_pair_max_clusters_fp4(int bn);

// Grouped GEMM on 256 x 256 CTA-pair tiles (p.grouped = 1, tokens in the A
// role), on `clusters` clusters; its co-resident cluster count and pipeline facts.
cudaError_t launch_gemm_grouped_pair_fp8(const GemmParams &p, const CUtensorMap &map_a, const CUtensorMap &map_b,
                                         const CUtensorMap &map_sfa, const CUtensorMap &map_sfb, int clusters,
                                         cudaStream_t stream);
cudaError_t launch_gemm_grouped_pair_fp4(const GemmParams &p, const CUtensorMap &map_a, const CUtensorMap &map_b,
                                         const CUtensorMap &map_sfa, const CUtensorMap &map_sfb, int clusters,
                                         cudaStream_t stream);
int gemm_grouped_pair_max_clusters_fp8();
int gemm_grouped_pair_max_clusters_fp4();

// BF16 (kind::f16, no scales) GEMM: single-CTA tiles (bn 32..256) and CTA-pair
// tiles (bn 128, 256; the scale maps are not read).
cudaError_t launch_gemm_bf16(int bn, bool lean, const GemmParams &p, const CUtensorMap &map_a,
                             const CUtensorMap &map_b, int grid, cudaStream_t stream);
cudaError_t launch_gemm_pair_bf16(int bn, const GemmParams &p, const CUtensorMap &map_a, const CUtensorMap &map_b,
                                  const CUtensorMap &map_sfa, const CUtensorMap &map_sfb, const CUtensorMap &map_sarm, int clusters,
                                  cudaStream_t stream);
int gemm_pair_max_clusters_bf16(int bn);

// Pipeline facts of one instantiation, for plan descriptions.
struct KernelInfo {
    int stages;
    int acc_stages;
    int smem_bytes;
};
KernelInfo gemm_info_fp8(int bn, bool lean = false);
KernelInfo gemm_info_fp4(int bn, bool lean = false);
KernelInfo gemm_pair_info_fp8(int bn);
KernelInfo gemm_pair_info_fp4(int bn);
KernelInfo gemm_info_bf16(int bn, bool lean = false);
KernelInfo gemm_grouped_pair_info_fp8();
KernelInfo gemm_grouped_pair_info_fp4();
KernelInfo gemm_pair_info_bf16(int bn);

}  // namespace mxg
