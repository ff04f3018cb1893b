// quantize.cu -- MX quantiser: BF16 or FP32 activations [rows, K] -> E4M3 /
// E2M1 codes and E8M0 scales, the scales written either row-major or straight
// into the 512-byte tile layout the GEMM's tensor cores read (so the GEMM can
// skip its scale relayout for that operand).
//
// The FlyDSL page (English digest, "Performance numbers need their baselines")
// leaves quantisation outside the timed GEMM and "API compatibility is not
// universal input coverage" notes that incompatible scale layouts cost extra
// copies; producing the tile layout here is the copy-free form of that step.
// Recipe (per row and 32-value block along K; no formula is printed on the
// pages, this is the reading the oracle states too):
//   s = max(floor(log2 amax) - e_max, -127), e_max = 8 (E4M3) / 2 (E2M1),
//   an all-zero block s = 0, scale code s + 127; element = x * 2^-s rounded to
//   nearest-even on the element grid, saturating at 448 / 6; a block holding a
//   NaN or an infinity gets scale code 0xFF and zero codes.
//
// The work is a pure stream (read 2 or 4 bytes, write 1 or 1/2 byte + 1/32
// byte per element), so the kernel is built for HBM bandwidth:
//   * one warp handles a unit of G chunks of 512 consecutive elements of one
//     row; each lane owns 16 consecutive elements of a chunk (one 32-byte load
//     for BF16, two for FP32), so a warp's loads cover 1 or 2 KB contiguously
//     and all G chunks' loads are in flight before any arithmetic;
//   * amax is an unsigned max over the absolute-value bit patterns (monotone
//     for finite values; any pattern >= the infinity pattern marks a NaN or an
//     infinity), reduced over the two lanes of a block with one shuffle;
//   * 2^-s is built from its exponent bits, x * 2^-s is exact, and the
//     rounding is the hardware conversion cvt.rn.satfinite to e4m3x2 / e2m1x2;
//   * the four scale bytes of one 128-wide K-tile are gathered with shuffles
//     into one 32-bit word, which is exactly one row's 4-byte slot of a
//     512-byte scale tile (row r = 32q + p, K-block c at byte p*16 + q*4 + c);
//   * the grid is persistent (SM count x resident blocks), warps stride over
//     units; in tile layout the padding rows up to a multiple of 128 are
//     filled with code 127 by the same launch.
#include <cstdint>

#include <cuda_runtime.h>

#include "quantize.h"

namespace mxg {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kLaneElts = 16;
constexpr int kChunk = 32 * kLaneElts;  // elements per warp per chunk

// 32 bytes per lane, read-only path, not kept in L1 (each byte is read once).
__device__ __forceinline__ void ld_stream_32B(const void *p, uint32_t (&r)[8])
{
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "l"(p));
}

// Two FP32 values -> two E4M3 codes (lo in the low byte), nearest-even,
// saturating to +-448.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi)
{
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// Eight FP32 values -> eight E2M1 codes in one word (element i in nibble i),
// nearest-even, saturating to +-6.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&v)[8])
{
    uint32_t d;
    asm("{\n\t"
        ".reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t"
        "}"
        : "=r"(d)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return d;
}

// Byte offset of the 4-byte slot of (row, k-tile) in the tile layout.
__device__ __forceinline__ int64_t tile_slot(int64_t row, int64_t kt, int64_t num_kt)
{
    return ((row >> 7) * num_kt + kt) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

template <int FMT, int IN>
struct QTraits {
    static constexpr int kEMax = FMT == kQuantFmtMxfp8 ? 8 : 2;
    static constexpr int kG = IN == kQuantInBf16 ? 4 : 2;        // chunks per unit
    static constexpr int kLoads = IN == kQuantInBf16 ? 1 : 2;    // 32-B loads per lane per chunk
    static constexpr int kInBytes = IN == kQuantInBf16 ? 2 : 4;
};

template <int FMT, int IN>
__global__ void __launch_bounds__(kThreads) mx_quantize_kernel(QuantParams p)
{
    using T = QTraits<FMT, IN>;
    constexpr int G = T::kG;
    // a GEMM launched after this kernel (programmatic dependent launch) may run
    // its prologue now; it waits for this grid to complete before reading
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t K = p.K;
    const int64_t units_per_row = (K + kChunk * G - 1) / (kChunk * G);
    const int64_t units = p.rows * units_per_row;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int64_t num_kt = K >> 7;  // valid when tiled (K % 128 == 0)
    const int64_t sf_row_bytes = K >> 5;
    const char *x = static_cast<const char *>(p.x);
    uint8_t *codes = static_cast<uint8_t *>(p.codes);

    for (int64_t u = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); u < units; u += nwarps) {
        const int64_t row = u / units_per_row;
        const int64_t k0 = (u - row * units_per_row) * (kChunk * G);
        const char *xrow = x + row * K * T::kInBytes;

        uint32_t raw[G][T::kLoads][8];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t k = k0 + g * kChunk + lane * kLaneElts;
#pragma unroll
            for (int l = 0; l < T::kLoads; ++l) {
                if (k < K) {
                    ld_stream_32B(xrow + k * T::kInBytes + l * 32, raw[g][l]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        raw[g][l][i] = 0;
                }
            }
        }

#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t kc = k0 + g * kChunk;            // first element of the chunk
            const int64_t k = kc + lane * kLaneElts;       // this lane's first element
            float v[kLaneElts];
            uint32_t amax;
            if (IN == kQuantInBf16) {
                uint32_t m = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t w = raw[g][0][i];
                    m = __vmaxu2(m, w & 0x7FFF7FFFu);
                    v[2 * i] = __uint_as_float(w << 16);
                    v[2 * i + 1] = __uint_as_float(w & 0xFFFF0000u);
                }
                amax = max(m & 0xFFFFu, m >> 16) << 16;  // as the FP32 pattern
            } else {
                uint32_t m = 0;
#pragma unroll
                for (int l = 0; l < 2; ++l)
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t w = raw[g][l][i];
                        m = max(m, w & 0x7FFFFFFFu);
                        v[8 * l + i] = __uint_as_float(w);
                    }
                amax = m;
            }
            amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));  // the block's two lanes

            const bool nonfinite = amax >= 0x7F800000u;
            const int e = static_cast<int>(amax >> 23);                 // biased exponent of amax
            int scode = amax == 0 ? 127 : max(e - T::kEMax, 0);         // s + 127
            const float mul = __uint_as_float(static_cast<uint32_t>(254 - scode) << 23);  // 2^-s
            if (nonfinite)
                scode = 255;

            // codes
            if (FMT == kQuantFmtMxfp8) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t a = cvt_e4m3x2(v[4 * i] * mul, v[4 * i + 1] * mul);
                    const uint32_t b = cvt_e4m3x2(v[4 * i + 2] * mul, v[4 * i + 3] * mul);
                    w[i] = nonfinite ? 0u : (a | (b << 16));
                }
                if (k < K)
                    *reinterpret_cast<uint4 *>(codes + row * K + k) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
                uint32_t w[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float t[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        t[i] = v[8 * h + i] * mul;
                    w[h] = nonfinite ? 0u : cvt_e2m1x8(t);
                }
                if (k < K)
                    *reinterpret_cast<uint2 *>(codes + row * (K >> 1) + (k >> 1)) = make_uint2(w[0], w[1]);
            }

            // scales: lanes 2b and 2b+1 hold block b of the chunk; lane 8q
            // gathers the four blocks of K-tile q
            const int base = lane & ~7;
            uint32_t word = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                word |= static_cast<uint32_t>(__shfl_sync(0xFFFFFFFFu, scode, base + 2 * c)) << (8 * c);
            if (p.tiled) {
                const int64_t kt = (kc >> 7) + (lane >> 3);
                if ((lane & 7) == 0 && kt < num_kt)
                    *reinterpret_cast<uint32_t *>(p.scales + tile_slot(row, kt, num_kt)) = word;
            } else if (p.sf_words) {
                const int64_t kt = (kc >> 7) + (lane >> 3);
                if ((lane & 7) == 0 && kt * 128 < K)
                    *reinterpret_cast<uint32_t *>(p.scales + row * sf_row_bytes + kt * 4) = word;
            } else {
                const int64_t j = (k >> 5);
                if ((lane & 1) == 0 && k < K)
                    p.scales[row * sf_row_bytes + j] = static_cast<uint8_t>(scode);
            }
        }
    }

    // tile layout: rows rows..ceil128(rows)-1 carry code 127 (x1.0)
    if (p.tiled) {
        const int64_t pad_rows = ((p.rows + 127) & ~int64_t(127)) - p.rows;
        const int64_t n = pad_rows * num_kt;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
             i += static_cast<int64_t>(gridDim.x) * kThreads) {
            const int64_t row = p.rows + i / num_kt, kt = i % num_kt;
            *reinterpret_cast<uint32_t *>(p.scales + tile_slot(row, kt, num_kt)) = 0x7F7F7F7Fu;
        }
    }
}

template <int FMT, int IN>
cudaError_t launch_one(const QuantParams &p, int num_sms, cudaStream_t s)
{
    static int occ = 0;  // resident blocks per SM (same for every sm_103 device)
    if (occ == 0) {
        int o = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, mx_quantize_kernel<FMT, IN>, kThreads, 0);
        if (e != cudaSuccess)
            return e;
        occ = o > 0 ? o : 1;
    }
    using T = QTraits<FMT, IN>;
    const int64_t units_per_row = (p.K + kChunk * T::kG - 1) / (kChunk * T::kG);
    const int64_t units = p.rows * units_per_row;
    int64_t blocks = (units + kWarps - 1) / kWarps;
    const int64_t cap = static_cast<int64_t>(num_sms) * occ;
    if (blocks > cap)
        blocks = cap;
    if (p.tiled && blocks < 1)
        blocks = 1;
    mx_quantize_kernel<FMT, IN><<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const QuantParams &p, int num_sms, cudaStream_t s)
{
    if (p.fmt == kQuantFmtMxfp8)
        return p.in_dtype == kQuantInBf16 ? launch_one<kQuantFmtMxfp8, kQuantInBf16>(p, num_sms, s)
                                          : launch_one<kQuantFmtMxfp8, kQuantInF32>(p, num_sms, s);
    return p.in_dtype == kQuantInBf16 ? launch_one<kQuantFmtMxfp4, kQuantInBf16>(p, num_sms, s)
                                      : launch_one<kQuantFmtMxfp4, kQuantInF32>(p, num_sms, s);
}

}  // namespace mxg
