// probe.cu -- the tensor pipe's own rate: every SM (or CTA pair) issues
// back-to-back tcgen05.mma from operands resident in shared memory (no loads),
// optionally with the scale copies (tcgen05.cp) a GEMM k-stage issues, and
// times them.  It gives the ceiling the GEMM kernels are compared with: the
// cycles one MMA of each kind takes per M = 128 (or 256 on a pair) x N tile.
#include <cstdint>
#include <mutex>

#include "launch.h"
#include "ptx.cuh"
#include "../../include/mxgemm.h"

namespace {

using namespace mxg;

constexpr int kProbeSlots = 4;       // operand sets cycled through
constexpr int kProbeMaxUnits = 256;  // CTAs (or pairs) reporting
constexpr uint64_t kProbeWaitNs = 2000000000ull;

__device__ unsigned long long g_probe_out[4 * kProbeMaxUnits];  // per unit: cycles, ns, start, end
__device__ int g_probe_err;

template <int KIND, int CG, int N>
struct ProbeCfg {
    static constexpr bool kFp4 = KIND == K_MXFP4;
    static constexpr bool kScaled = KIND != K_BF16;
    static constexpr int kBRows = CG == 2 ? N / 2 : N;  // B rows held by this CTA
    static constexpr int kABytes = kBM * kRowBytes;
    static constexpr int kBBytes = kBRows * kRowBytes;
    static constexpr int kKt = kFp4 ? 2 : 1;  // scale K-tiles per k-stage
    static constexpr int kChunksB = N / 128;
    static constexpr int kSfaBytes = kScaled ? kKt * kSfChunk : 0;
    static constexpr int kSfbBytes = kScaled ? kKt * kChunksB * kSfChunk : 0;
    static constexpr int kSet = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static constexpr int kSmemRaw = 1024 + kProbeSlots * kSet;
    // at least 120 KB, so that one CTA holds an SM (and its TMEM) alone
    static constexpr int kSmem = kSmemRaw < 120 * 1024 ? 120 * 1024 : kSmemRaw;
    static constexpr int kSfaCols = kScaled ? 4 * kKt : 0;
    static constexpr int kSetCols = kSfaCols + (kScaled ? 4 * kKt * kChunksB : 0);
    static constexpr int kM = CG == 2 ? 2 * kBM : kBM;
    static constexpr uint32_t kIdesc = kScaled ? idesc_block_scaled(kFp4 ? 1u : 0u, kM, N) : idesc_bf16(kM, N);
    static constexpr int kMmasPerStage = kFp4 ? 4 : 4;  // MXFP8 / BF16: 4 per 128-byte K-slice; MXFP4: 2 per K-tile
    static_assert(N == 128 || N == 256, "probe tiles are 128 or 256 wide");
};

template <int KIND, int CG, int N, bool CP>
__global__ void __launch_bounds__(128, 1) tensor_rate_probe(int stages)
{
    using C = ProbeCfg<KIND, CG, N>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_holder;
    __shared__ uint64_t done;
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *g = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    // Finite operand bytes of each kind (the values do not matter to the rate)
    // and scale code 127 (x1).
    for (int i = threadIdx.x; i < kProbeSlots * C::kSet; i += blockDim.x) {
        uint8_t v;
        if (i >= kProbeSlots * (C::kABytes + C::kBBytes))
            v = 127;
        else if (KIND == K_MXFP8)
            v = static_cast<uint8_t>((i * 37u) & 0x37u);  // E4M3 below 1, never NaN
        else if (KIND == K_MXFP4)
            v = static_cast<uint8_t>(i * 29u);  // any E2M1 pair is finite
        else
            v = (i & 1) ? 0x3Fu : static_cast<uint8_t>(i * 13u);  // BF16 in [0.5, 2)
        g[i] = v;
    }
    fence_proxy_async_smem();
    const uint32_t done_bar = smem_addr(&done);
    if (threadIdx.x == 0) {
        mbar_init(done_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        if constexpr (CG == 2) {
            tmem_alloc_pair(smem_addr(&tmem_holder), 512);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_addr(&tmem_holder), 512);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2)
        cluster_sync();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;
    unsigned long long c0 = 0, t0 = 0;
    if (warp == 0 && leader) {
        c0 = clock64();
        t0 = global_timer_ns();
        const uint32_t sA = base;
        const uint32_t sB = sA + kProbeSlots * C::kABytes;
        const uint32_t sSfa = sB + kProbeSlots * C::kBBytes;
        const uint32_t sSfb = sSfa + kProbeSlots * C::kSfaBytes;
        for (int it = 0; it < stages; ++it) {
            const int s = it % kProbeSlots;
            const uint32_t sfa_col = tmem + 256 + s * C::kSetCols;
            const uint32_t sfb_col = sfa_col + C::kSfaCols;
            if (elect_one()) {
                if constexpr (CP && C::kScaled) {
#pragma unroll
                    for (int t = 0; t < C::kKt; ++t) {
                        const uint64_t da = sdesc_sf_chunk(sSfa + s * C::kSfaBytes + t * kSfChunk);
                        if constexpr (CG == 2)
                            tc_cp_pair_32x128b_warpx4(sfa_col + 4 * t, da);
                        else
                            tc_cp_32x128b_warpx4(sfa_col + 4 * t, da);
#pragma unroll
                        for (int c = 0; c < C::kChunksB; ++c) {
                            const uint64_t db = sdesc_sf_chunk(sSfb + s * C::kSfbBytes + (c * C::kKt + t) * kSfChunk);
                            if constexpr (CG == 2)
                                tc_cp_pair_32x128b_warpx4(sfb_col + 4 * (t * C::kChunksB + c), db);
                            else
                                tc_cp_32x128b_warpx4(sfb_col + 4 * (t * C::kChunksB + c), db);
                        }
                    }
                }
                const uint64_t adesc = sdesc_kmajor_sw128(sA + s * C::kABytes);
                const uint64_t bdesc = sdesc_kmajor_sw128(sB + s * C::kBBytes);
#pragma unroll
                for (int m = 0; m < C::kMmasPerStage; ++m) {
                    const int t = C::kFp4 ? m / 2 : 0;
                    const uint32_t sf_id = C::kFp4 ? static_cast<uint32_t>((m % 2) * 2) : static_cast<uint32_t>(m);
                    const uint32_t idesc = C::kScaled ? idesc_with_sf_ids(C::kIdesc, sf_id, sf_id) : C::kIdesc;
                    const uint64_t koff = static_cast<uint64_t>((m * 32) >> 4);
                    const uint32_t acc = (it > 0 || m > 0) ? 1u : 0u;
                    const uint32_t sfa_t = sfa_col + 4 * t, sfb_t = sfb_col + 4 * t * C::kChunksB;
                    if constexpr (KIND == K_BF16) {
                        if constexpr (CG == 2)
                            mma_pair_bf16(tmem, adesc + koff, bdesc + koff, idesc, acc);
                        else
                            mma_bf16(tmem, adesc + koff, bdesc + koff, idesc, acc);
                    } else if constexpr (KIND == K_MXFP4) {
                        if constexpr (CG == 2)
                            mma_pair_mxf4(tmem, adesc + koff, bdesc + koff, idesc, sfa_t, sfb_t, acc);
                        else
                            mma_mxf4(tmem, adesc + koff, bdesc + koff, idesc, sfa_t, sfb_t, acc);
                    } else {
                        if constexpr (CG == 2)
                            mma_pair_mxf8f6f4(tmem, adesc + koff, bdesc + koff, idesc, sfa_t, sfb_t, acc);
                        else
                            mma_mxf8f6f4(tmem, adesc + koff, bdesc + koff, idesc, sfa_t, sfb_t, acc);
                    }
                }
            }
            __syncwarp();
        }
        if (elect_one()) {
            if constexpr (CG == 2)
                tc_commit_pair(done_bar, 0x3);
            else
                tc_commit(done_bar);
        }
        __syncwarp();
    }
    unsigned long long c1 = 0, t1 = 0;
    if (warp == 0) {
        const volatile int never = 0;
        const bool ok = warp_wait(done_bar, 0, &never, kProbeWaitNs);
        if (!ok && (threadIdx.x & 31) == 0)
            atomicExch(&g_probe_err, 1);
        c1 = clock64();
        t1 = global_timer_ns();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2)
        cluster_sync();
    if (warp == 0) {
        tc_fence_after();
        if constexpr (CG == 2)
            tmem_dealloc_pair(tmem, 512);
        else
            tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && leader) {
        const int u = CG == 2 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
        if (u < kProbeMaxUnits) {
            g_probe_out[4 * u + 0] = c1 - c0;
            g_probe_out[4 * u + 1] = t1 - t0;
            g_probe_out[4 * u + 2] = t0;
            g_probe_out[4 * u + 3] = t1;
        }
    }
}

template <int KIND, int CG, int N, bool CP>
int run_probe(int stages, double *result, cudaStream_t s)
{
    using C = ProbeCfg<KIND, CG, N>;
    auto kernel = tensor_rate_probe<KIND, CG, N, CP>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config(CG == 2 ? 2 : 1, 128, C::kSmem, s, attr, CG, false);
    int units = sms;
    if (CG == 2 && cudaOccupancyMaxActiveClusters(&units, kernel, &cfg) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    units = units < kProbeMaxUnits ? units : kProbeMaxUnits;
    if (units < 1)
        return MXGEMM_ERR_CUDA;
    cfg.gridDim = dim3(CG * units, 1, 1);
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_probe_err, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    // a short warm-up launch, then the measured one
    if (cudaLaunchKernelEx(&cfg, kernel, 64) != cudaSuccess || cudaLaunchKernelEx(&cfg, kernel, stages) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    unsigned long long h[4 * kProbeMaxUnits];
    int err = 0;
    if (cudaMemcpyFromSymbolAsync(h, g_probe_out, sizeof(unsigned long long) * 4 * units, 0, cudaMemcpyDeviceToHost,
                                  s) != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&err, g_probe_err, sizeof err, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    if (err)
        return MXGEMM_ERR_DEVICE_TIMEOUT;
    double cycles = 0.0, ns = 0.0;
    unsigned long long tmin = ~0ull, tmax = 0ull;
    for (int u = 0; u < units; ++u) {
        cycles += static_cast<double>(h[4 * u]);
        ns += static_cast<double>(h[4 * u + 1]);
        tmin = h[4 * u + 2] < tmin ? h[4 * u + 2] : tmin;
        tmax = h[4 * u + 3] > tmax ? h[4 * u + 3] : tmax;
    }
    const double mmas = static_cast<double>(stages) * C::kMmasPerStage;
    const double k_per_mma = KIND == K_BF16 ? 16.0 : KIND == K_MXFP4 ? 64.0 : 32.0;
    const double flops = 2.0 * C::kM * N * k_per_mma * mmas * units;
    result[0] = cycles / units / mmas;                                    // cycles per MMA
    result[1] = cycles / ns;                                              // SM clock, GHz
    result[2] = tmax > tmin ? flops / static_cast<double>(tmax - tmin) / 1e6 : 0.0;  // PFLOP/s, whole GPU
    result[3] = units;
    return MXGEMM_OK;
}

template <int KIND, int CG, int N>
int run_probe_cp(int scale_copies, int stages, double *result, cudaStream_t s)
{
    return scale_copies ? run_probe<KIND, CG, N, true>(stages, result, s)
                        : run_probe<KIND, CG, N, false>(stages, result, s);
}

template <int KIND>
int run_probe_kind(int cta_group, int n, int scale_copies, int stages, double *result, cudaStream_t s)
{
    if (cta_group == 1)
        return n == 128 ? run_probe_cp<KIND, 1, 128>(scale_copies, stages, result, s)
                        : run_probe_cp<KIND, 1, 256>(scale_copies, stages, result, s);
    return n == 128 ? run_probe_cp<KIND, 2, 128>(scale_copies, stages, result, s)
                    : run_probe_cp<KIND, 2, 256>(scale_copies, stages, result, s);
}

}  // namespace

extern "C" MXGEMM_API int mxgemm_probe_tensor_rate(int fmt, int cta_group, int n, int scale_copies, int stages,
                                                   double *result, void *stream)
{
    if (!result || (cta_group != 1 && cta_group != 2) || (n != 128 && n != 256) ||
        (scale_copies != 0 && scale_copies != 1) || stages < 16 || stages > (1 << 22))
        return MXGEMM_ERR_ARG;
    if (fmt != MXGEMM_FMT_MXFP8_E4M3 && fmt != MXGEMM_FMT_MXFP4_E2M1 && fmt != MXGEMM_FMT_BF16)
        return MXGEMM_ERR_ARG;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    if (major != 10 || minor != 3)
        return MXGEMM_ERR_ARCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fmt == MXGEMM_FMT_MXFP8_E4M3)
        return run_probe_kind<K_MXFP8>(cta_group, n, scale_copies, stages, result, s);
    if (fmt == MXGEMM_FMT_MXFP4_E2M1)
        return run_probe_kind<K_MXFP4>(cta_group, n, scale_copies, stages, result, s);
    return run_probe_kind<K_BF16>(cta_group, n, 0, stages, result, s);
}
