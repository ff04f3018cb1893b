// placement.cu -- exhaustive scale-placement checker for MXFP4 dot products.
//
// "Deciding Scale Placement in MXFP4 Dot Products with Integer Arithmetic"
// (AI-compiler daily digest of 2026-10-22, item 2): when an MXFP4 dot product
// is lowered, the shared power-of-two scales can be applied to the elements
// before the products ("pre") or to the sum after it ("post"); in binary32 the
// two can round differently (overflow, NaN from inf - inf or inf * 0,
// subnormals), and the study bounds the scale exponents for which they agree
// under a fixed binary reduction tree.  This kernel decides it by enumeration:
// for each scale pair (sa, sb) it evaluates every tuple of k E2M1 elements per
// operand (16^(2k) tuples) in both placements and against the exact value
// rounded once, with every binary32 operation rounded to nearest even and no
// fused multiply-add:
//   f_a = 2^(sa-127), f_b = 2^(sb-127)   (exact binary32 values, also subnormal)
//   pre  = tree( (a_i f_a) (b_i f_b) ),  post = (tree( a_i b_i ) f_a) f_b,
//   rn   = binary32( sum a_i b_i * 2^(sa+sb-254) )  (exact in binary64, rounded once)
// tree(n terms) = tree(first ceil(n/2)) + tree(rest).  Two results agree when
// both are NaN or they are equal values.
#include <cstdint>

#include <cuda_runtime.h>

#include "placement.h"

namespace mxg {
namespace {

// 2^e as binary32, exactly, for e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int e)
{
    return e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(1 << (e + 149));
}

// 2^e as binary64, exactly, for e in [-1022, 1023].
__device__ __forceinline__ double pow2d(int e)
{
    return __longlong_as_double(static_cast<long long>(e + 1023) << 52);
}

// E2M1 value from its bit fields: sign bit 3, exponent bits 2..1 (bias 1),
// mantissa bit 0; exponent 0 is subnormal (m * 0.5).
__device__ __forceinline__ float e2m1(unsigned code)
{
    const unsigned e = (code >> 1) & 3u, m = code & 1u;
    const float mag = e ? (1.0f + 0.5f * m) * pow2f(static_cast<int>(e) - 1) : 0.5f * m;
    return (code & 8u) ? -mag : mag;
}

__device__ __forceinline__ float tree_sum(const float (&v)[4], int k)
{
    switch (k) {
    case 1: return v[0];
    case 2: return __fadd_rn(v[0], v[1]);
    case 3: return __fadd_rn(__fadd_rn(v[0], v[1]), v[2]);
    default: return __fadd_rn(__fadd_rn(v[0], v[1]), __fadd_rn(v[2], v[3]));
    }
}

__device__ __forceinline__ bool same(float x, float y)
{
    const bool nx = isnan(x), ny = isnan(y);
    return (nx || ny) ? (nx && ny) : x == y;
}

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    placement_scan_kernel(int k, const int *sa_list, const int *sb_list, int npairs, int chunks,
                          unsigned long long ntup, unsigned long long *counts, unsigned long long *first)
{
    const int pair = static_cast<int>(blockIdx.x) / chunks;
    const int chunk = static_cast<int>(blockIdx.x) % chunks;
    if (pair >= npairs)
        return;
    const int sa = sa_list[pair], sb = sb_list[pair];
    if (sa < 0 || sa > 254 || sb < 0 || sb > 254)
        return;  // reported by the finishing kernel
    const float fa = pow2f(sa - 127), fb = pow2f(sb - 127);
    const double fe = pow2d(sa + sb - 254);
    const unsigned long long per = (ntup + chunks - 1) / chunks;
    const unsigned long long t0 = per * chunk;
    const unsigned long long t1 = min(ntup, t0 + per);
    unsigned long long n_diff = 0, n_pre = 0, n_post = 0, first_local = ntup;
    for (unsigned long long t = t0 + threadIdx.x; t < t1; t += kThreads) {
        float pp[4] = {0.f, 0.f, 0.f, 0.f}, qq[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < k; ++i) {
            const float a = e2m1(static_cast<unsigned>(t >> (4 * i)) & 15u);
            const float b = e2m1(static_cast<unsigned>(t >> (4 * (k + i))) & 15u);
            pp[i] = __fmul_rn(__fmul_rn(a, fa), __fmul_rn(b, fb));
            qq[i] = __fmul_rn(a, b);  // exact: a multiple of 1/4, |.| <= 36
        }
        // Every partial sum of the unscaled products is a multiple of 1/4 below
        // 4 * 36 in magnitude, so the binary32 tree sum is the exact sum; the
        // scaled exact value is formed in binary64 (exact) and rounded once.
        const float unscaled = tree_sum(qq, k);
        const float pre = tree_sum(pp, k);
        const float post = __fmul_rn(__fmul_rn(unscaled, fa), fb);
        const float rn = __double2float_rn(static_cast<double>(unscaled) * fe);
        const bool d = !same(pre, post);
        n_diff += d;
        n_pre += same(pre, rn);
        n_post += same(post, rn);
        if (d && t < first_local)
            first_local = t;
    }
    // warp sums / minimum, then one atomic per warp
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        n_diff += __shfl_xor_sync(0xFFFFFFFFu, n_diff, o);
        n_pre += __shfl_xor_sync(0xFFFFFFFFu, n_pre, o);
        n_post += __shfl_xor_sync(0xFFFFFFFFu, n_post, o);
        first_local = min(first_local, __shfl_xor_sync(0xFFFFFFFFu, first_local, o));
    }
    if ((threadIdx.x & 31) == 0) {
        if (n_diff) atomicAdd(counts + 3 * pair, n_diff);
        if (n_pre) atomicAdd(counts + 3 * pair + 1, n_pre);
        if (n_post) atomicAdd(counts + 3 * pair + 2, n_post);
        if (first_local < ntup) atomicMin(first + pair, first_local);
    }
}

__global__ void placement_init_kernel(int npairs, unsigned long long ntup, unsigned long long *counts,
                                      unsigned long long *first)
{
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < npairs; p += gridDim.x * blockDim.x) {
        counts[3 * p] = counts[3 * p + 1] = counts[3 * p + 2] = 0;
        first[p] = ntup;
    }
}

// No counterexample -> -1; an invalid scale code -> counts and first of -1.
__global__ void placement_finish_kernel(const int *sa_list, const int *sb_list, int npairs, unsigned long long ntup,
                                        long long *counts, long long *first)
{
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < npairs; p += gridDim.x * blockDim.x) {
        const int sa = sa_list[p], sb = sb_list[p];
        if (sa < 0 || sa > 254 || sb < 0 || sb > 254) {
            counts[3 * p] = counts[3 * p + 1] = counts[3 * p + 2] = -1;
            first[p] = -1;
        } else if (static_cast<unsigned long long>(first[p]) >= ntup) {
            first[p] = -1;
        }
    }
}

}  // namespace

cudaError_t launch_placement_scan(int k, const int *sa, const int *sb, int npairs, long long *counts,
                                  long long *first_diff, int num_sms, cudaStream_t s)
{
    const unsigned long long ntup = 1ull << (8 * k);
    unsigned long long *c = reinterpret_cast<unsigned long long *>(counts);
    unsigned long long *f = reinterpret_cast<unsigned long long *>(first_diff);
    const int init_blocks = (npairs + 255) / 256;
    placement_init_kernel<<<init_blocks, 256, 0, s>>>(npairs, ntup, c, f);
    // enough blocks per pair to fill the GPU a few times over, each with >= 64 tuples per thread
    long long chunks = static_cast<long long>(num_sms) * 8 / npairs;
    const long long max_chunks = static_cast<long long>((ntup + kThreads * 64 - 1) / (kThreads * 64));
    chunks = chunks < 1 ? 1 : chunks;
    chunks = chunks > max_chunks ? max_chunks : chunks;
    const long long blocks = chunks * npairs;
    if (blocks > 0x7FFFFFFFll)
        return cudaErrorInvalidConfiguration;
    placement_scan_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(k, sa, sb, npairs, static_cast<int>(chunks),
                                                                            ntup, c, f);
    placement_finish_kernel<<<init_blocks, 256, 0, s>>>(sa, sb, npairs, ntup, counts, first_diff);
    return cudaGetLastError();
}

}  // namespace mxg
