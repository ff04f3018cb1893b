// launch.h -- internal interface between the host API (mxgemm.cu) and the
// translation units that instantiate the GEMM kernel (gemm_fp8.cu, gemm_fp4.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace mxg {

// Launch the persistent GEMM kernel for tile width `bn` (32, 64, 128, 256) on
// `grid` CTAs.  Returns cudaErrorInvalidValue for an unsupported bn.
cudaError_t launch_gemm_fp8(int bn, const GemmParams &p, const CUtensorMap &map_a, const CUtensorMap &map_b,
                            int grid, cudaStream_t stream);
cudaError_t launch_gemm_fp4(int bn, const GemmParams &p, const CUtensorMap &map_a, const CUtensorMap &map_b,
                            int grid, cudaStream_t stream);

// Pipeline facts of one instantiation, for plan descriptions.
struct KernelInfo {
    int stages;
    int acc_stages;
    int smem_bytes;
};
KernelInfo gemm_info_fp8(int bn);
KernelInfo gemm_info_fp4(int bn);

}  // namespace mxg
