// gemm_fp8.cu -- MXFP8 (E4M3, kind::mxf8f6f4, scale_vec::1X) instantiations of
// the persistent block-scaled GEMM kernel.
#include "launch.h"

namespace mxg {

namespace {
template <int BN>
cudaError_t launch(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, int grid, cudaStream_t s)
{
    using C = Cfg<false, BN>;
    auto kern = mx_gemm_kernel<false, BN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess)
        return e;
    kern<<<grid, kThreads, C::kSmemBytes, s>>>(p, ma, mb);
    return cudaGetLastError();
}

template <int BN>
KernelInfo info()
{
    using C = Cfg<false, BN>;
    return KernelInfo{C::kStages, C::kAccStages, C::kSmemBytes};
}
}  // namespace

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
