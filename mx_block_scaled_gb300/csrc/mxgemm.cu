// mxgemm.cu -- host side of libmxgemm.so: argument validation, the per-shape
// plan (tile width, operand roles, split-K), TMA descriptor encoding, the scale
// relayout and split-K reduce kernels, and the C ABI of include/mxgemm.h.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "launch.h"
#include "mxgemm.h"
#include "placement.h"
#include "quantize.h"

namespace {

using mxg::GemmParams;

// Sticky device status word, written by kernels that give up on a wait.
__device__ int g_device_status;

// Stream-K arrival counters.  They live in the library rather than in the
// caller's workspace so that no launch needs a memset before it: the array is
// zero when the module loads, and every completed launch leaves its counters
// at zero (the last segment to arrive at a tile resets the tile's counter).
// Each plan owns a disjoint range (taken at plan creation, returned when the
// plan is destroyed), so plans running concurrently on different streams never
// share a counter.  A launch that gave up on a wait (device timeout) may leave
// counters nonzero; mxgemm_device_status(..., reset) then zeroes the array.
constexpr int kCounterPool = 1 << 16;
__device__ int g_sk_counters[kCounterPool];

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    bool kernels_prepared = false;
    bool is_sm103 = false;
    int num_sms = 0;
    int *status_ptr = nullptr;
    int *counters_ptr = nullptr;                  // device address of g_sk_counters
    std::vector<std::pair<int, int>> free_ranges; // unowned [offset, offset + length) of the counters
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

// First-fit range of n counters on device dev, or -1 (the plan then keeps its
// counters in the workspace, zeroed before each launch).
int counters_take(int dev, int n)
{
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    auto &fr = g_dev[dev].free_ranges;
    for (size_t i = 0; i < fr.size(); ++i) {
        if (fr[i].second >= n) {
            const int off = fr[i].first;
            fr[i].first += n;
            fr[i].second -= n;
            if (fr[i].second == 0)
                fr.erase(fr.begin() + static_cast<long>(i));
            return off;
        }
    }
    return -1;
}

void counters_give_back(int dev, int off, int n)
{
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    auto &fr = g_dev[dev].free_ranges;
    fr.emplace_back(off, n);
    std::sort(fr.begin(), fr.end());
    std::vector<std::pair<int, int>> merged;
    for (const auto &r : fr) {
        if (!merged.empty() && merged.back().first + merged.back().second == r.first)
            merged.back().second += r.second;
        else
            merged.push_back(r);
    }
    fr.swap(merged);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

int device_info(DeviceInfo **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return MXGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
            return MXGEMM_ERR_CUDA;
        d.is_sm103 = (prop.major == 10 && prop.minor == 3);
        d.num_sms = prop.multiProcessorCount;
        if (d.is_sm103) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess)
                return MXGEMM_ERR_CUDA;
            d.status_ptr = static_cast<int *>(p);
            if (cudaGetSymbolAddress(&p, g_sk_counters) != cudaSuccess)
                return MXGEMM_ERR_CUDA;
            d.counters_ptr = static_cast<int *>(p);
            d.free_ranges.assign(1, std::make_pair(0, kCounterPool));
        }
        if (!g_encode_tiled) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return MXGEMM_ERR_CUDA;
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        if (d.is_sm103) {
            if (mxg::prepare_gemm_fp8() != cudaSuccess || mxg::prepare_gemm_fp4() != cudaSuccess ||
                mxg::prepare_gemm_bf16() != cudaSuccess)
                return MXGEMM_ERR_CUDA;
            d.kernels_prepared = true;
        }
        d.ready = true;
    }
    *out = &d;
    return d.is_sm103 ? MXGEMM_OK : MXGEMM_ERR_ARCH;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Vector width of the epilogue's row stores: 2 = 32-byte stores (row pitch and
// base 32-byte aligned), 1 = 16-byte stores, 0 = element stores (transposed
// output, or rows not 16-byte aligned).
inline int vec_level(bool rows_contiguous, int64_t row_bytes, const void *base)
{
    if (!rows_contiguous || row_bytes % 16 != 0 || !aligned16(base))
        return 0;
    return (row_bytes % 32 == 0 && (reinterpret_cast<uintptr_t>(base) & 31u) == 0) ? 2 : 1;
}
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ----------------------------------------------------------- scale relayout --
// One block per (128-row block, up to 8 K-tiles): the 128 x (8 x 4) scale bytes
// are staged in shared memory as 32-bit words (4 K-blocks each; all four loads
// of a thread in flight at once), then written as 512-byte tiles, one 16-byte
// store per thread.  Inside a tile, row r = 32q + p and K-block c of the tile go
// to byte p*16 + q*4 + c: the layout the tensor cores read scale factors from
// when a 32-row x 16-byte chunk is copied into TMEM.
constexpr int kRelayoutKt = 8;  // K-tiles (of 4 K-blocks) per block

struct RelayoutJob {
    const uint8_t *src;
    uint8_t *dst;
    int rows;
    int num_kt;   // K / 128
    int blocks_x; // ceil(num_kt / kRelayoutKt)
    int blocks;   // ceil(rows / 128) * blocks_x
};

// zero / nzero: words the GEMM that follows needs zeroed (its stream-K arrival
// counters), cleared by block 0 so that no separate memset is launched.
__global__ void __launch_bounds__(256)
    relayout_scales_kernel(RelayoutJob j0, RelayoutJob j1, int *zero, int nzero)
{
    __shared__ uint32_t tile[128][kRelayoutKt + 1];
    mxg::griddep_launch_dependents();  // the GEMM that follows may start its prologue
    int b = blockIdx.x;
    if (b == 0)
        for (int i = threadIdx.x; i < nzero; i += 256)
            zero[i] = 0;
    const RelayoutJob &j = (b < j0.blocks) ? j0 : j1;
    if (b >= j0.blocks)
        b -= j0.blocks;
    const int rb = b / j.blocks_x;
    const int kt0 = (b % j.blocks_x) * kRelayoutKt;
    const uint32_t *src = reinterpret_cast<const uint32_t *>(j.src);  // num_kt words per row
    uint32_t v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + 256 * i;
        const int r = idx / kRelayoutKt, w = idx % kRelayoutKt;
        const int row = rb * 128 + r, kt = kt0 + w;
        v[i] = 0x7F7F7F7Fu;  // padding rows: scale code 127 (x1.0)
        if (row < j.rows && kt < j.num_kt)
            v[i] = __ldg(src + static_cast<size_t>(row) * j.num_kt + kt);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + 256 * i;
        tile[idx / kRelayoutKt][idx % kRelayoutKt] = v[i];
    }
    __syncthreads();
    const int w = threadIdx.x >> 5, p = threadIdx.x & 31;
    const int kt = kt0 + w;
    if (kt < j.num_kt) {
        uint4 o = make_uint4(tile[p][w], tile[32 + p][w], tile[64 + p][w], tile[96 + p][w]);
        reinterpret_cast<uint4 *>(j.dst + (static_cast<size_t>(rb) * j.num_kt + kt) * 512)[p] = o;
    }
}

RelayoutJob make_job(const uint8_t *src, int64_t rows, int64_t K, uint8_t *dst)
{
    RelayoutJob j;
    j.src = src;
    j.dst = dst;
    j.rows = static_cast<int>(rows);
    j.num_kt = static_cast<int>(K / 128);
    j.blocks_x = static_cast<int>(ceil_div(j.num_kt, kRelayoutKt));
    j.blocks = static_cast<int>(ceil_div(rows, 128)) * j.blocks_x;
    return j;
}

cudaError_t launch_relayout(const RelayoutJob &a, const RelayoutJob *b, cudaStream_t s, int *zero = nullptr,
                            int nzero = 0)
{
    RelayoutJob none{};
    none.blocks = 0;
    const RelayoutJob &j1 = b ? *b : none;
    const int blocks = a.blocks + j1.blocks;
    relayout_scales_kernel<<<blocks, 256, 0, s>>>(a, j1, zero, nzero);
    return cudaGetLastError();
}

// ------------------------------------------------- grouped scale relayout --
// Token scales of a grouped GEMM: the rows of group e (start and count
// sanitised exactly as the GEMM does it) go to their own run of 128-row tile
// blocks starting at block tok_rb[e], the last block padded with code 127, so
// that every 128-row token tile finds its scales in one 512-byte chunk per
// K-tile.  One block per (tile block, up to 8 K-tiles); blocks past the used
// (or available) ones exit at once.
__global__ void __launch_bounds__(256)
    grouped_relayout_kernel(const uint8_t *src, const long long *offsets, int groups, int total_rows, int num_kt,
                            int blocks_x, int cap_blocks, uint8_t *dst)
{
    __shared__ int tok_rb[mxg::kMaxGroups + 1];
    __shared__ int row0[mxg::kMaxGroups];
    __shared__ int rows[mxg::kMaxGroups];
    __shared__ uint32_t tile[128][kRelayoutKt + 1];
    mxg::griddep_launch_dependents();  // the grouped GEMM that follows may start its prologue
    if (threadIdx.x < 32)
        mxg::group_scan(offsets, groups, total_rows, 128, 1, static_cast<int>(threadIdx.x), nullptr, tok_rb, row0,
                        rows);
    __syncthreads();
    const int rb = static_cast<int>(blockIdx.x) / blocks_x;
    const int kt0 = (static_cast<int>(blockIdx.x) % blocks_x) * kRelayoutKt;
    if (rb >= tok_rb[groups] || rb >= cap_blocks)
        return;  // block-uniform
    int lo = 0, hi = groups - 1;  // the last group whose first block is <= rb (skips empty groups)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tok_rb[mid] <= rb)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int lb = rb - tok_rb[lo];
    const uint32_t *s32 = reinterpret_cast<const uint32_t *>(src);  // num_kt words per row
    uint32_t v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + 256 * i;
        const int r = idx / kRelayoutKt, w = idx % kRelayoutKt;
        const int local = lb * 128 + r, kt = kt0 + w;
        v[i] = 0x7F7F7F7Fu;
        if (local < rows[lo] && kt < num_kt)
            v[i] = __ldg(s32 + static_cast<size_t>(row0[lo] + local) * num_kt + kt);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + 256 * i;
        tile[idx / kRelayoutKt][idx % kRelayoutKt] = v[i];
    }
    __syncthreads();
    const int w = threadIdx.x >> 5, pr = threadIdx.x & 31;
    const int kt = kt0 + w;
    if (kt < num_kt) {
        uint4 o = make_uint4(tile[pr][w], tile[32 + pr][w], tile[64 + pr][w], tile[96 + pr][w]);
        reinterpret_cast<uint4 *>(dst + (static_cast<size_t>(rb) * num_kt + kt) * 512)[pr] = o;
    }
}

// -------------------------------------------------------- split-K reduce --
// C[e] = sum_s part[s][e], summed in split order (deterministic), then stored
// as FP32 or rounded to BF16.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ part, int splits,
                                                             long long n, long long slab, void *out,
                                                             int out_kind)
{
    mxg::griddep_wait();  // launched as a programmatic dependent of the GEMM that wrote `part`
    mxg::griddep_launch_dependents();
    const long long n4 = n / 4;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    for (long long i = tid; i < n4; i += stride) {
        float4 acc = __ldg(reinterpret_cast<const float4 *>(part) + i);
        for (int s = 1; s < splits; ++s) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(part + s * slab) + i);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        if (out_kind == mxg::OUT_BF16) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 w = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
            reinterpret_cast<uint2 *>(out)[i] = w;
        } else {
            reinterpret_cast<float4 *>(out)[i] = acc;
        }
    }
    if (tid < n - n4 * 4) {  // the last n % 4 elements
        const long long t = n4 * 4 + tid;
        float acc = part[t];
        for (int s = 1; s < splits; ++s)
            acc += part[s * slab + t];
        if (out_kind == mxg::OUT_BF16)
            static_cast<__nv_bfloat16 *>(out)[t] = __float2bfloat16_rn(acc);
        else
            static_cast<float *>(out)[t] = acc;
    }
}

}  // namespace

// ----------------------------------------------------------------- plan --
struct mxgemm_plan {
    int64_t M, N, K;
    int fmt, out;
    int swap;          // 1: compute C^T = B * A^T (B fills the MMA M dimension)
    int mode;          // 0: one CTA per 128-row tile; 1: 256-row tiles on CTA pairs with M = 256
                       // MMAs (cta_group::2)
    int bn;            // MMA N tile
    int splits;        // split-K factor
    int tiles_m, tiles_n;
    int kstages, kstages_per_split;
    int grid;
    int group_m;
    int num_sms;
    int dp_tiles;      // stream-K: tiles computed whole (first in raster order)
    int sk_tiles;      // stream-K: tiles whose k-stages are spread over sk_ctas CTAs
    int sk_ctas;       // 0: no stream-K (counts clusters in pair mode)
    int sk_halves;     // 128-row shares per tile (2 in pair mode): counters and slots per tile / unit
    int device;        // the device current when the plan was created; runs must use it
    size_t off_sfa, off_sfb, off_part, off_cnt, off_skp, ws_bytes;
    int sa_fuse;        // 1: row-major A scales are laid out inside the GEMM (pair tiles, K % 512 == 0)
    int lean;           // 1: the lean single-CTA form (weight-streaming decode tiles, two CTAs per SM)
    int cnt_pool = -1;  // stream-K counters: offset in the library's counter array (-1: in the workspace)
    int cnt_n = 0;      // counters of the plan (stream-K tiles x 128-row shares)
    // TMA descriptor cache (re-encoded when an operand pointer changes)
    const void *map_ptr_a = nullptr;
    const void *map_ptr_b = nullptr;
    const void *map_ptr_sfa = nullptr;
    const void *map_ptr_sfb = nullptr;
    const void *map_ptr_sarm = nullptr;
    CUtensorMap map_a, map_b, map_sfa, map_sfb, map_sarm;
};

struct mxgemm_grouped_plan {
    int64_t G, T, N, K;  // groups, token rows (of A and C), weight rows per group, K
    int fmt, out;
    int swap;            // 1: tokens are the MMA N (B) role, weights fill the 128-row M role
    int bn;              // MMA N tile
    int kstages;
    int num_sms;
    int device;
    int tok_sf_cap;      // 128-row blocks of the tokens' tile-layout scale region
    int mode = 0;        // 1: 256 x 256 CTA-pair tiles (tokens in the A role, 256-row tiles per group)
    int clusters = 0;    // pair mode: co-resident clusters of two (the grid)
    size_t off_tok_sf, off_w_sf, ws_bytes;
    const void *map_ptr_tok = nullptr;
    const void *map_ptr_w = nullptr;
    CUtensorMap map_tok, map_w;
    // pair mode: 3-D operand maps (two k-stages a box) and the scale maps
    const void *map_ptr_tok3 = nullptr, *map_ptr_w3 = nullptr, *map_ptr_sftok = nullptr, *map_ptr_sfw = nullptr;
    CUtensorMap map_tok3, map_w3, map_sftok, map_sfw;
};

namespace {

int encode_operand_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t row_bytes, int box_rows)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MXGEMM_OK : MXGEMM_ERR_CUDA;
}

// An operand (rows x row_bytes, row-major) as a 3-D tensor for the CTA-pair
// kernel: the 128-byte K-slices of a row, the rows, then the slice index (the
// innermost two dimensions make a k-stage tile, the third selects the stage).
// Box = box_rows rows x two consecutive k-stages, landing as two 128-byte
// swizzled tiles one after the other.  Needs row_bytes % 128 == 0, so that no
// slice reaches past the end of a row.
int encode_operand_map_2stage(CUtensorMap *map, const void *ptr, int64_t rows, int64_t row_bytes, int box_rows)
{
    cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(row_bytes / 128)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), 128u};
    cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(box_rows), 2u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MXGEMM_OK : MXGEMM_ERR_CUDA;
}

// Row-major scales (rows x K/32 bytes) as a 2-D tensor for the CTA-pair kernel's
// fused layout: box = one scale group (kSfGroup k-stages of kt_per_stage
// K-tiles: 4 bytes each) of a pair tile's 256 rows (rows past the end read as
// zero).  Needs (K/32) % 16 == 0 (row pitch) and group starts on 16-byte
// boundaries (the kernel aligns its groups to them).
int encode_rowmajor_sf_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int kt_per_stage)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 32), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 32)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(4 * kt_per_stage * mxg::kSfGroup), 256u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MXGEMM_OK : MXGEMM_ERR_CUDA;
}

// Tile-layout scales of `rows` operand rows as a 3-D tensor: rows of 256 bytes
// (a 512-byte chunk is two), 2 * (K/128) rows per 128-row block, then the row
// blocks.  Box = one scale group (kSfGroup k-stages of kt_per_stage K-tiles)
// of `blocks` consecutive 128-row blocks; a box reaching past the last K-tile
// or row block is zero-filled (and those chunks are never read).
int encode_sf_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int kt_per_stage, int blocks)
{
    const int64_t num_kt = K / 128;
    cuuint64_t dims[3] = {256u, static_cast<cuuint64_t>(2 * num_kt), static_cast<cuuint64_t>(ceil_div(rows, 128))};
    cuuint64_t strides[2] = {256u, static_cast<cuuint64_t>(num_kt * 512)};
    cuuint32_t box[3] = {256u, static_cast<cuuint32_t>(2 * kt_per_stage * mxg::kSfGroup),
                         static_cast<cuuint32_t>(blocks)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MXGEMM_OK : MXGEMM_ERR_CUDA;
}

// N tile for a B role of rows_b rows.  BN = 32 only when the whole B role fits
// in one tile, so a 32-row tile always starts on its scale chunk's first 32 rows
// (see tile_geom: the B scale-factor TMEM column must be even).
int pick_bn(int64_t rows_b)
{
    if (rows_b <= 32) return 32;
    if (rows_b <= 64) return 64;
    if (rows_b <= 128) return 128;
    return 256;
}

}  // namespace

extern "C" {

int mxgemm_version(void) { return 100; }

const char *mxgemm_status_str(int status)
{
    switch (status) {
    case MXGEMM_OK: return "ok";
    case MXGEMM_ERR_ARG: return "invalid argument (NULL pointer or unknown enum/flag)";
    case MXGEMM_ERR_SHAPE: return "invalid shape (need M,N >= 1 and K a positive multiple of 128)";
    case MXGEMM_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case MXGEMM_ERR_WORKSPACE: return "workspace missing or too small";
    case MXGEMM_ERR_ARCH: return "current device is not an sm_103 GPU";
    case MXGEMM_ERR_CUDA: return "CUDA runtime or driver call failed";
    case MXGEMM_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting on a barrier (device timeout)";
    case MXGEMM_ERR_UNSUPPORTED: return "request not supported by this build";
    case MXGEMM_ERR_DEVICE_BOUNDS: return "a debug-build kernel skipped an out-of-range load or store";
    default: return "unknown status";
    }
}

size_t mxgemm_sf_bytes(int64_t rows, int64_t K)
{
    if (rows < 1 || K < 128 || K % 128 != 0)
        return 0;
    return static_cast<size_t>(ceil_div(rows, 128) * 128) * static_cast<size_t>(K / 32);
}

int mxgemm_plan_create(mxgemm_plan_t *plan, int64_t M, int64_t N, int64_t K, int fmt, int out, uint32_t flags)
{
    if (!plan)
        return MXGEMM_ERR_ARG;
    *plan = nullptr;
    if ((fmt != MXGEMM_FMT_MXFP8_E4M3 && fmt != MXGEMM_FMT_MXFP4_E2M1 && fmt != MXGEMM_FMT_BF16) ||
        (out != MXGEMM_OUT_F32 && out != MXGEMM_OUT_BF16))
        return MXGEMM_ERR_ARG;
    const bool bf16 = fmt == MXGEMM_FMT_BF16;
    const uint32_t known = MXGEMM_PLAN_FORCE_BN128 | MXGEMM_PLAN_FORCE_BN256 | MXGEMM_PLAN_FORCE_NOSWAP |
                           MXGEMM_PLAN_FORCE_SWAP | MXGEMM_PLAN_FORCE_PAIR | MXGEMM_PLAN_FORCE_SINGLE |
                           MXGEMM_PLAN_STREAMK | MXGEMM_PLAN_NO_STREAMK | MXGEMM_PLAN_FORCE_BN192 |
                           (0xFFu << MXGEMM_PLAN_SPLITK_SHIFT);
    if ((flags & ~known) != 0 || ((flags & MXGEMM_PLAN_FORCE_SWAP) && (flags & MXGEMM_PLAN_FORCE_NOSWAP)) ||
        ((flags & MXGEMM_PLAN_FORCE_BN192) &&
         (flags & (MXGEMM_PLAN_FORCE_BN128 | MXGEMM_PLAN_FORCE_BN256 | MXGEMM_PLAN_FORCE_SINGLE | MXGEMM_PLAN_STREAMK))) ||
        ((flags & MXGEMM_PLAN_STREAMK) && (flags & MXGEMM_PLAN_NO_STREAMK)) ||
        ((flags & MXGEMM_PLAN_FORCE_BN128) && (flags & MXGEMM_PLAN_FORCE_BN256)) ||
        ((flags & MXGEMM_PLAN_FORCE_PAIR) && (flags & MXGEMM_PLAN_FORCE_SINGLE)))
        return MXGEMM_ERR_ARG;
    // MX formats: K a multiple of 128 (the FlyDSL page's constraint); BF16: of 64
    // (one 128-byte k-stage row).
    if (M < 1 || N < 1 || K < (bf16 ? 64 : 128) || K % (bf16 ? 64 : 128) != 0)
        return MXGEMM_ERR_SHAPE;
    // 32-bit tile and row indices inside the kernels
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30))
        return MXGEMM_ERR_UNSUPPORTED;

    DeviceInfo *dev = nullptr;
    int st = device_info(&dev);
    if (st != MXGEMM_OK)
        return st;

    mxgemm_plan *p = new (std::nothrow) mxgemm_plan();
    if (!p)
        return MXGEMM_ERR_UNSUPPORTED;
    p->M = M;
    p->N = N;
    p->K = K;
    p->fmt = fmt;
    p->out = out;
    p->num_sms = dev->num_sms;
    cudaGetDevice(&p->device);

    // Operand roles: small token counts put the weight (B) in the 128-row MMA dimension.
    int swap = (M <= 64 && N >= 128) ? 1 : 0;
    // MXFP8 with 65..128 tokens and a long k-loop: the weight in the 256-row role
    // of CTA-pair tiles and the tokens as one 128-wide tile, which computes no
    // empty rows and fits an 8-stage ring (scales pre-laid-out: 128 x 5120 x
    // 8192 19.6 -> 16.5 us, 128 x 5120 x 25600 35.0 -> 29.3 us; no gain at K =
    // 5120).  Row-major activation scales then take a relayout launch (~2.4 us).
    const bool swap_pair =
        fmt == MXGEMM_FMT_MXFP8_E4M3 && M > 64 && M <= 128 && N >= 256 && K >= 8192 &&
        !(flags & (MXGEMM_PLAN_FORCE_SWAP | MXGEMM_PLAN_FORCE_NOSWAP | MXGEMM_PLAN_FORCE_SINGLE |
                   MXGEMM_PLAN_FORCE_PAIR | MXGEMM_PLAN_FORCE_BN128 | MXGEMM_PLAN_FORCE_BN256 |
                   MXGEMM_PLAN_FORCE_BN192 | MXGEMM_PLAN_STREAMK)) &&
        ((flags >> MXGEMM_PLAN_SPLITK_SHIFT) & 0xFFu) == 0;
    if (swap_pair) swap = 1;
    if (flags & MXGEMM_PLAN_FORCE_SWAP) swap = 1;
    if (flags & MXGEMM_PLAN_FORCE_NOSWAP) swap = 0;
    p->swap = swap;
    const int64_t rows_a = swap ? N : M;
    const int64_t rows_b = swap ? M : N;
    int bn = pick_bn(rows_b);
    if (flags & MXGEMM_PLAN_FORCE_BN128) bn = 128;
    if (flags & MXGEMM_PLAN_FORCE_BN256) bn = 256;
    // Pair tiles need 128- or 256-wide N tiles.  Default: every format with at
    // least 128 rows on each side runs 256 x 256 pair tiles (measured faster from
    // 128 tokens up): an MXFP4 k-stage moves the same operand bytes as an MXFP8
    // one in the same MMA time, so it gains the same from the pair tile's halved
    // B-operand loads (2048 x 4096 x 14336: 56.5 -> 43.8 us; 4096^3: 35.9 ->
    // 28.7 us; 256 x 28672 x 4096: 21.5 -> 19.7 us).  MXFP4 with fewer pair
    // tiles than half the pairs stays on single-CTA tiles, which need fewer
    // K-splits (128 x 5120 x 25600: pair 31.4 us, single 22.2 us); MXFP8 keeps
    // the pair tiles there, whose in-kernel activation-scale layout saves the
    // relayout launch.  Swapped decode shapes stay on single-CTA tiles.
    int mode = 0;
    const bool pair_ok = !swap && rows_a >= 128 && rows_b >= 256 && !(flags & MXGEMM_PLAN_FORCE_BN128) &&
                         ((flags >> MXGEMM_PLAN_SPLITK_SHIFT) & 0xFFu) == 0;
    const int64_t pair_tiles = ceil_div(rows_a, 256) * ceil_div(rows_b, 256);
    const int64_t pair_tiles192 = ceil_div(rows_a, 256) * ceil_div(rows_b, 192);
    // MXFP4 whose 256-wide pair tiles stay under half the pairs but whose
    // 192-wide ones reach half and fit in a wave, with k-loops of at most 32
    // stages: 192-wide pair tiles (256 x 8192 x 8192: single-CTA split-K 18.2
    // us, 256 x 192 pair tiles 16.2 us; with 112 k-stages, 256 x 8192 x 28672,
    // the single-CTA split-K plan stays faster: 37.0 against 41.5 us).
    bool fp4_192 = false;
    if (pair_ok && (fmt != MXGEMM_FMT_MXFP4_E2M1 || pair_tiles >= dev->num_sms / 4)) {
        mode = 1;
    } else if (pair_ok && fmt == MXGEMM_FMT_MXFP4_E2M1 && pair_tiles192 >= dev->num_sms / 4 &&
               pair_tiles192 <= dev->num_sms / 2 && ceil_div(K, 256) <= 32 &&
               !(flags & (MXGEMM_PLAN_FORCE_BN128 | MXGEMM_PLAN_FORCE_BN256 | MXGEMM_PLAN_STREAMK))) {
        mode = 1;
        fp4_192 = true;
    }
    // BF16 runs its MMAs at half the MX rate per operand byte, so it is bound by
    // the tensor pipe where MX formats wait on memory: with at most 128 tokens a
    // pair tile's M = 256 MMAs would compute half empty rows (128 x 10240 x 5120:
    // pair 30.5 us, 128 x 128 tiles 23.9 us) -- unless the narrower tiles need
    // more than one wave (128 x 51200 x 5120: pair 95.0 us, single 97.5 us).
    if (bf16 && rows_a <= 128 && ceil_div(rows_b, 128) <= dev->num_sms) mode = 0;
    if (swap_pair || (flags & (MXGEMM_PLAN_FORCE_PAIR | MXGEMM_PLAN_FORCE_BN192))) mode = 1;
    if (flags & MXGEMM_PLAN_FORCE_SINGLE) mode = 0;
    // pair tiles load two 128-byte K-slices per box: MXFP4 rows must be a whole
    // number of slices (K % 256 == 0), else single-CTA tiles
    if (fmt == MXGEMM_FMT_MXFP4_E2M1 && K % 256 != 0) mode = 0;
    if ((flags & MXGEMM_PLAN_FORCE_BN192) && mode != 1) {  // 192-wide tiles exist on CTA pairs only
        delete p;
        return MXGEMM_ERR_UNSUPPORTED;
    }
    // The activation scales' relayout (the FlyDSL page's extra layout copy) runs
    // inside the MXFP8 pair kernel when their row pitch K/32 allows 16-byte TMA
    // rows.
    p->sa_fuse = (mode == 1 && fmt == MXGEMM_FMT_MXFP8_E4M3 && !swap && K % 512 == 0) ? 1 : 0;
    if (mode != 0 && bn < 128) bn = 128;
    // BF16 with few tiles: 128-wide N tiles rather than a 256-wide tile count
    // below the work slots (which leaves SMs idle or needs split-K and its reduce
    // pass), as long as the narrower tiles still fit in one wave.  Measured
    // (256 tokens, K = 4096-8192): N = 6144 20.8 -> 17.4 us, N = 8192 35.7 ->
    // 31.8 us; 128 tokens: N = 5120 25.9 -> 20.5 us.
    if (bf16 && bn == 256 &&
        !(flags & (MXGEMM_PLAN_FORCE_BN128 | MXGEMM_PLAN_FORCE_BN256 | MXGEMM_PLAN_STREAMK))) {
        const int64_t units_m = mode == 0 ? ceil_div(rows_a, 128) : ceil_div(rows_a, 256);
        const int64_t slots_est = mode == 0 ? dev->num_sms : dev->num_sms / 2;
        if (units_m * ceil_div(rows_b, 256) < slots_est && units_m * ceil_div(rows_b, 128) <= slots_est)
            bn = 128;
    }
    // 192-wide pair tiles where the 256-wide ones fill less than a wave of pairs,
    // cannot be split two ways within one (the split-K rule below would then
    // split them), and the narrower ones still fit in one wave: more pairs at
    // work, each k-stage shorter.  Measured: 256 x 10240 x 8192 MXFP8 (40 -> 54
    // of 76 pairs) 27.8 -> 25.6 us, MXFP4 18.1 -> 16.7, BF16 45.9 -> 37.1;
    // where two-way split-K fits, 192-wide tiles without it lost (256 x 8192 x
    // 28672: 55.3 -> 72.0 us).
    if (mode == 1 && bn == 256 &&
        !(flags & (MXGEMM_PLAN_FORCE_BN128 | MXGEMM_PLAN_FORCE_BN256 | MXGEMM_PLAN_STREAMK))) {
        const int64_t units_m = ceil_div(rows_a, 256);
        const int64_t pairs_est = dev->num_sms / 2;
        const int64_t t256 = units_m * ceil_div(rows_b, 256), t192 = units_m * ceil_div(rows_b, 192);
        if (t256 < pairs_est && 2 * t256 > pairs_est && t192 <= pairs_est && t192 > t256)
            bn = 192;
    }
    if ((flags & MXGEMM_PLAN_FORCE_BN192) || (fp4_192 && mode == 1)) bn = 192;
    // Stream-K on CTA pairs runs on 256-wide tiles only (the pair kernel's
    // stream-K instantiation): a forced stream-K pair plan takes them.
    if ((flags & MXGEMM_PLAN_STREAMK) && mode == 1) bn = 256;
    p->mode = mode;
    p->bn = bn;
    // Weight-streaming decode with at most 32 tokens (swap-AB single-CTA MX
    // tiles of 32 columns) runs the lean form: two of its CTAs fit on an SM, so
    // the next GEMM's CTAs are resident (TMEM allocated, first ring warmed in
    // L2) while this one drains.  Measured: MXFP8 8 x 8192 x 8192 17.8 -> 16.9
    // us, 8 x 10240 x 8192 21.2 -> 20.1; MXFP4 8 x 8192 x 8192 13.7 -> 11.6.
    // Its ring is smaller (5 stages), which costs the 64-token tiles (4 stages:
    // 64 x 10240 x 8192 22.7 -> 26.3 us) and BF16 (8 x 8192 x 8192 26.2 ->
    // 27.2), so those keep the full form.
    p->lean = (swap && mode == 0 && bn == 32 && !bf16) ? 1 : 0;
    // tiles_m counts the work units along the A role: 128-row tiles (single),
    // 256-row tiles (pair).
    p->tiles_m = static_cast<int>(mode == 0 ? ceil_div(rows_a, 128) : ceil_div(rows_a, 256));
    p->tiles_n = static_cast<int>(ceil_div(rows_b, bn));
    // The MMA reads a B-role tile's scales from TMEM column (tn*BN % 128) / 32 of
    // its scale chunk, which must be even: a 32-wide tile other than the first
    // would start at an odd column (a misaligned-address fault).  BN = 32 is
    // picked only for at most 32 B-role rows; refuse anything else outright.
    if (bn == 32 && p->tiles_n > 1) {
        delete p;
        return MXGEMM_ERR_UNSUPPORTED;
    }
    p->kstages = static_cast<int>(fmt == MXGEMM_FMT_MXFP4_E2M1 ? ceil_div(K, 256) : bf16 ? K / 64 : K / 128);

    // Concurrent work units: SMs, or co-resident clusters of two.
    int64_t slots = p->num_sms;
    if (mode != 0) {
        const int max_clusters = fmt == MXGEMM_FMT_MXFP4_E2M1 ? mxg::gemm_pair_max_clusters_fp4(bn)
                                 : bf16                           ? mxg::gemm_pair_max_clusters_bf16(bn)
                                                                  : mxg::gemm_pair_max_clusters_fp8(bn);
        if (max_clusters < 1) {
            delete p;
            return MXGEMM_ERR_CUDA;
        }
        slots = max_clusters;
    }

    // Work decomposition.  Default: whole tiles, plus uniform split-K with a
    // separate reduce when the tiles alone cannot fill half the GPU.  Stream-K
    // (single-CTA or pair tiles): whole tiles in full waves over the work slots,
    // and the k-stages of the remaining tiles spread over the slots, fixed up in
    // the kernel -- by default for long k-loops with a poor last wave, always
    // (when the last wave is under 95% full) with MXGEMM_PLAN_STREAMK, never with
    // MXGEMM_PLAN_NO_STREAMK.
    const int64_t tiles = static_cast<int64_t>(p->tiles_m) * p->tiles_n;
    int splits = static_cast<int>((flags >> MXGEMM_PLAN_SPLITK_SHIFT) & 0xFFu);
    p->dp_tiles = static_cast<int>(tiles);
    p->sk_tiles = 0;
    p->sk_ctas = 0;
    p->sk_halves = mode == 1 ? 2 : 1;
    if (splits == 0) {
        const int64_t G = slots;
        const int64_t waves = ceil_div(tiles, G);
        const double dp_eff = static_cast<double>(tiles) / static_cast<double>(waves * G);
        // Default (256-wide tiles, last wave under 90% full): the fixup of a cut
        // tile (L2 round trips of the partial sums, several us with every SM
        // streaming operands into L2; longer for three or more partials) must
        // hide behind the whole tiles each slot computes after its segment, so
        //  - halves: each tile of the last wave cut into two segments (2 x its
        //    tiles <= slots), when the whole tiles give every slot >= 96
        //    k-stages (MXFP8 4096^3: +6.5%; MXFP4 4096^3 at 48: a loss);
        //  - spread: the last wave's k-stages over every slot (cuts of any
        //    length), for long k-loops (>= 96 k-stages a tile) with >= 3 waves
        //    of whole tiles (K = 25600: +10%).
        // With no full wave of whole tiles (every tile cut) the fixups run
        // back to back after the segments: measured 1.4x slower.
        const int64_t full_waves = tiles / G;
        const bool spread = p->kstages >= 96 && full_waves >= 3;
        const bool halves = full_waves * p->kstages >= 96 && 2 * (tiles % G) <= G;
        // Weight-streaming decode (swap-AB, single-CTA tiles of <= 64 tokens):
        // every SM should stream an equal share of the weight from the start,
        // so the k-stages of the tiles past the full waves are spread evenly
        // over all SMs; the cut tiles' partial sums are small (128 x BN FP32)
        // and are added by the epilogue warps of the last CTA to arrive, which
        // replaces the separate split-K reduce launch.
        const bool decode = swap && mode == 0 && p->bn <= 64;
        // By default decode takes stream-K where its fixed cost (the fixup of
        // the cut tiles after the last segment) is paid back: k-loops of at
        // least 64 stages, and either tiles that a uniform 2-way split-K would
        // spread over more than one wave, or long k-loops.  Otherwise split-K
        // with its reduce launch is faster (MXFP8 8 x 8192 x 8192: stream-K
        // 19.4 us, split 2 17.6; MXFP4 8 x 10240 x 8192: 18.1 vs split 5 15.7;
        // MXFP8 8 x 10240 x 8192: stream-K 22.0 vs split 8 24.4; 8 x 8192 x
        // 28672: 44.6 vs split 2 47.1).
        const bool decode_sk = decode && p->kstages >= 64 && (tiles * 2 > G || p->kstages >= 128);
        const bool want = (flags & MXGEMM_PLAN_STREAMK)
                              ? dp_eff < 0.95
                              : (!(flags & MXGEMM_PLAN_NO_STREAMK) && dp_eff < 0.90 &&
                                 ((p->bn == 256 && (spread || halves)) || decode_sk));
        if (want) {
            const int64_t dp = (tiles / G) * G;
            const int64_t sk_stages = (tiles - dp) * p->kstages;
            const int64_t min_seg = 4;  // k-stages per stream-K unit, at least
            // Long k-loops spread the cut tiles' stages over every slot.  Short
            // ones cut each tile in at most two segments, so that the fixup adds
            // two partial sums (one batch of loads) and stays short.
            const bool spread_units = (flags & MXGEMM_PLAN_STREAMK) ? (p->kstages >= 96 || decode) : (spread || decode);
            const int64_t units = spread_units ? std::min<int64_t>(G, sk_stages / min_seg)
                                               : std::min<int64_t>(G, 2 * (tiles - dp));
            p->dp_tiles = static_cast<int>(dp);
            p->sk_tiles = static_cast<int>(tiles - dp);
            p->sk_ctas = static_cast<int>(std::max<int64_t>(1, std::min(units, sk_stages / min_seg)));
        }
        if (flags & MXGEMM_PLAN_STREAMK)
            splits = 1;
    }
    if (splits == 0 && p->sk_ctas > 0)
        splits = 1;
    if (splits == 0) {
        splits = 1;
        const int64_t by_k = std::max<int64_t>(1, p->kstages / 4);
        if (tiles * 2 <= slots) {
            const int64_t by_sms = slots / tiles;
            splits = static_cast<int>(std::min<int64_t>(std::min(by_sms, by_k), 32));
        } else if (tiles < 2 * slots) {
            // Between half a wave and two waves of tiles: split K so that the
            // units fill the slots better (time ~ waves(s) / s), as long as the
            // FP32 partials stay within 10% of the operand bytes -- the
            // weight-streaming decode shapes (M <= 64), where a wave of 80
            // tiles on 152 SMs left half the SMs without a weight stream.
            const double e = fmt == MXGEMM_FMT_MXFP4_E2M1 ? 0.5 : bf16 ? 2.0 : 1.0;
            const double operand_bytes = static_cast<double>(M + N) * static_cast<double>(K) * e;
            const double split_bytes = 4.0 * static_cast<double>(M) * static_cast<double>(N);
            const int64_t by_traffic = static_cast<int64_t>(0.1 * operand_bytes / split_bytes);
            const int64_t max_s = std::min<int64_t>(std::min(by_k, by_traffic), 32);
            double best = static_cast<double>(ceil_div(tiles, slots));
            for (int64_t s2 = 2; s2 <= max_s; ++s2) {
                const double t = static_cast<double>(ceil_div(tiles * s2, slots)) / static_cast<double>(s2);
                if (t < 0.95 * best) {
                    best = t;
                    splits = static_cast<int>(s2);
                }
            }
        }
    }
    splits = std::max(1, std::min(splits, p->kstages));
    p->kstages_per_split = static_cast<int>(ceil_div(p->kstages, splits));
    p->splits = static_cast<int>(ceil_div(p->kstages, p->kstages_per_split));
    p->group_m = 8;
    const int64_t units = p->sk_ctas > 0 ? std::max<int64_t>(p->dp_tiles > 0 ? slots : 0, p->sk_ctas)
                                         : tiles * p->splits;
    p->grid = static_cast<int>(std::min<int64_t>(units, slots));  // CTAs, or clusters of 2 CTAs

    size_t off = 0;
    p->off_sfa = off;
    off = align256(off + (bf16 ? 0 : mxgemm_sf_bytes(M, K)));
    p->off_sfb = off;
    off = align256(off + (bf16 ? 0 : mxgemm_sf_bytes(N, K)));
    p->off_part = off;
    if (p->splits > 1)
        off = align256(off + static_cast<size_t>(p->splits) * ((M * N + 7) & ~7ll) * sizeof(float));
    p->off_cnt = off;
    p->off_skp = off;
    if (p->sk_ctas > 0) {
        p->cnt_n = p->sk_tiles * p->sk_halves;
        p->cnt_pool = counters_take(p->device, p->cnt_n);
        if (p->cnt_pool < 0)  // the library's counters are all taken: keep them in the workspace
            off = align256(off + static_cast<size_t>(p->cnt_n) * sizeof(int));
        p->off_skp = off;
        off = align256(off + static_cast<size_t>(2) * p->sk_ctas * p->sk_halves * 128 * bn * sizeof(float));
    }
    p->ws_bytes = off;
    *plan = p;
    return MXGEMM_OK;
}

int mxgemm_plan_destroy(mxgemm_plan_t plan)
{
    if (plan && plan->cnt_pool >= 0)
        counters_give_back(plan->device, plan->cnt_pool, plan->cnt_n);
    delete plan;
    return MXGEMM_OK;
}

size_t mxgemm_workspace_bytes(mxgemm_plan_t plan) { return plan ? plan->ws_bytes : 0; }

int mxgemm_plan_describe(mxgemm_plan_t plan, char *buf, size_t len)
{
    if (!plan || !buf || len == 0)
        return MXGEMM_ERR_ARG;
    const bool fp4 = plan->fmt == MXGEMM_FMT_MXFP4_E2M1;
    const bool bf16 = plan->fmt == MXGEMM_FMT_BF16;
    static const char *const kModes[2] = {"single", "pair"};
    const bool lean = plan->lean != 0;
    mxg::KernelInfo ki = plan->mode == 1 ? (fp4 ? mxg::gemm_pair_info_fp4(plan->bn)
                                                : bf16 ? mxg::gemm_pair_info_bf16(plan->bn)
                                                       : mxg::gemm_pair_info_fp8(plan->bn))
                                         : (fp4    ? mxg::gemm_info_fp4(plan->bn, lean)
                                            : bf16 ? mxg::gemm_info_bf16(plan->bn, lean)
                                                   : mxg::gemm_info_fp8(plan->bn, lean));
    snprintf(buf, len,
             "fmt=%s out=%s tile=%dx%d mode=%s swap_ab=%d split_k=%d streamk=%d+%d/%d units=%dx%d kstages=%d grid=%d%s "
             "stages=%d acc_stages=%d smem=%d sa=%s%s",
             fp4 ? "mxfp4" : bf16 ? "bf16" : "mxfp8", plan->out == MXGEMM_OUT_BF16 ? "bf16" : "f32",
             plan->mode == 1 ? 256 : 128,
             plan->bn, kModes[plan->mode], plan->swap, plan->splits, plan->dp_tiles, plan->sk_tiles, plan->sk_ctas,
             plan->tiles_m, plan->tiles_n, plan->kstages, plan->grid, plan->mode ? "x2" : "", ki.stages, ki.acc_stages,
             ki.smem_bytes, plan->sa_fuse ? "in-kernel" : "relayout", lean ? " lean" : "");
    return MXGEMM_OK;
}

int mxgemm_relayout_scales(const uint8_t *src, int64_t rows, int64_t K, uint8_t *dst, void *stream)
{
    if (!src || !dst)
        return MXGEMM_ERR_ARG;
    if (rows < 1 || K < 128 || K % 128 != 0 || rows > (1ll << 30))
        return MXGEMM_ERR_SHAPE;
    if (!aligned16(src) || !aligned16(dst))
        return MXGEMM_ERR_ALIGN;
    RelayoutJob j = make_job(src, rows, K, dst);
    return launch_relayout(j, nullptr, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MXGEMM_OK
                                                                                          : MXGEMM_ERR_CUDA;
}

int mxgemm_quantize(int fmt, int in_dtype, const void *x, int64_t rows, int64_t K, void *codes, uint8_t *scales,
                    uint32_t flags, void *stream)
{
    if (!x || !codes || !scales)
        return MXGEMM_ERR_ARG;
    if ((fmt != MXGEMM_FMT_MXFP8_E4M3 && fmt != MXGEMM_FMT_MXFP4_E2M1) ||
        (in_dtype != MXGEMM_IN_F32 && in_dtype != MXGEMM_IN_BF16) || (flags & ~MXGEMM_QUANT_SF_TILED) != 0)
        return MXGEMM_ERR_ARG;
    const bool tiled = (flags & MXGEMM_QUANT_SF_TILED) != 0;
    if (rows < 1 || rows > (1ll << 31) || K < 32 || K % 32 != 0 || K > (1ll << 31) || (tiled && K % 128 != 0))
        return MXGEMM_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(x) & 31u) != 0 || !aligned16(codes) || !aligned16(scales))
        return MXGEMM_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    const int st = device_info(&dev);
    if (st != MXGEMM_OK)
        return st;
    mxg::QuantParams p;
    p.x = x;
    p.codes = codes;
    p.scales = scales;
    p.rows = rows;
    p.K = K;
    p.fmt = fmt == MXGEMM_FMT_MXFP8_E4M3 ? mxg::kQuantFmtMxfp8 : mxg::kQuantFmtMxfp4;
    p.in_dtype = in_dtype == MXGEMM_IN_BF16 ? mxg::kQuantInBf16 : mxg::kQuantInF32;
    p.tiled = tiled ? 1 : 0;
    p.sf_words = K % 128 == 0 ? 1 : 0;
    return mxg::launch_quantize(p, dev->num_sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MXGEMM_OK
                                                                                                   : MXGEMM_ERR_CUDA;
}

// Phase 1 of a run: the relayout of whichever scales are not pre-laid-out into
// the workspace.  A plan whose stream-K counters had to go into the workspace
// (the library's array was full) also has them zeroed here, by the same launch
// (a memset when nothing is laid out): the kernel leaves them zero when it
// completes, but the workspace may be fresh or hold an aborted launch's.
// Arguments checked by the callers.
static int prepare_impl(mxgemm_plan_t plan, const uint8_t *SA, const uint8_t *SB, uint8_t *ws, uint32_t run_flags,
                        cudaStream_t s)
{
    RelayoutJob jobs[2];
    int njobs = 0;
    if (plan->fmt != MXGEMM_FMT_BF16) {
        if (!(run_flags & MXGEMM_RUN_SA_PRELAYOUT) && !plan->sa_fuse)
            jobs[njobs++] = make_job(SA, plan->M, plan->K, ws + plan->off_sfa);
        if (!(run_flags & MXGEMM_RUN_SB_PRELAYOUT))
            jobs[njobs++] = make_job(SB, plan->N, plan->K, ws + plan->off_sfb);
    }
    int *const sk_counters = reinterpret_cast<int *>(ws + plan->off_cnt);
    const int sk_ncnt = plan->cnt_pool < 0 ? plan->cnt_n : 0;
    if (njobs > 0) {
        if (launch_relayout(jobs[0], njobs > 1 ? &jobs[1] : nullptr, s, sk_counters, sk_ncnt) != cudaSuccess)
            return MXGEMM_ERR_CUDA;
    } else if (sk_ncnt > 0 &&
               cudaMemsetAsync(sk_counters, 0, static_cast<size_t>(sk_ncnt) * sizeof(int), s) != cudaSuccess) {
        return MXGEMM_ERR_CUDA;
    }
    return MXGEMM_OK;
}

// Debug build (MXGEMM_DEBUG): a run synchronises its stream and returns the
// device status word, so that a kernel's bounds check or timeout is reported
// by the call that caused it.  Release build: nothing (calls stay asynchronous).
static int debug_finish(cudaStream_t s)
{
#ifdef MXGEMM_DEBUG
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    return v;
#else
    (void)s;
    return MXGEMM_OK;
#endif
}

// dbg_short_rows: self-test of the debug build's bounds checks -- the GEMM
// kernel is told that C ends that many rows early.
static int run_impl(mxgemm_plan_t plan, const void *A, const uint8_t *SA, const void *B, const uint8_t *SB, void *C,
                    void *workspace, size_t ws_bytes, uint32_t run_flags, void *stream, int test_stall,
                    unsigned long long timeout_ns, int dbg_short_rows = 0)
{
    if (!plan || !A || !B || !C)
        return MXGEMM_ERR_ARG;
    const bool bf16 = plan->fmt == MXGEMM_FMT_BF16;  // no scales: SA and SB are not read
    if (run_flags & ~(MXGEMM_RUN_SA_PRELAYOUT | MXGEMM_RUN_SB_PRELAYOUT | MXGEMM_RUN_PREPARED | MXGEMM_RUN_B_STATIC))
        return MXGEMM_ERR_ARG;
    // after mxgemm_prepare, scales that were not pre-laid-out are in the workspace --
    // except row-major SA of a plan that lays it out inside the GEMM
    const bool prepared = (run_flags & MXGEMM_RUN_PREPARED) != 0;
    const bool fused = plan->sa_fuse && !(run_flags & MXGEMM_RUN_SA_PRELAYOUT);
    const bool read_sa = !bf16 && (!prepared || (run_flags & MXGEMM_RUN_SA_PRELAYOUT) || fused);
    const bool read_sb = !bf16 && (!prepared || (run_flags & MXGEMM_RUN_SB_PRELAYOUT));
    if ((read_sa && !SA) || (read_sb && !SB))
        return MXGEMM_ERR_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (read_sa && !aligned16(SA)) || (read_sb && !aligned16(SB)))
        return MXGEMM_ERR_ALIGN;
    if (plan->ws_bytes > 0 && (workspace == nullptr || ws_bytes < plan->ws_bytes))
        return MXGEMM_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace))
        return MXGEMM_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    int st = device_info(&dev);
    if (st != MXGEMM_OK)
        return st;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device)
        return MXGEMM_ERR_ARG;  // a plan runs on the device it was created on

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int64_t M = plan->M, N = plan->N, K = plan->K;
    const bool fp4 = plan->fmt == MXGEMM_FMT_MXFP4_E2M1;
    const int64_t row_bytes = fp4 ? K / 2 : bf16 ? 2 * K : K;

    // (1) scale relayout for whichever operand is not pre-laid-out, and the
    // stream-K counter reset -- unless mxgemm_prepare did both already
    if (bf16)
        run_flags = (run_flags & MXGEMM_RUN_PREPARED) | MXGEMM_RUN_SA_PRELAYOUT | MXGEMM_RUN_SB_PRELAYOUT;
    const uint8_t *sfa = (run_flags & MXGEMM_RUN_SA_PRELAYOUT) ? SA : ws + plan->off_sfa;
    const uint8_t *sfb = (run_flags & MXGEMM_RUN_SB_PRELAYOUT) ? SB : ws + plan->off_sfb;
    int *const sk_counters = reinterpret_cast<int *>(ws + plan->off_cnt);
    if (!(run_flags & MXGEMM_RUN_PREPARED)) {
        st = prepare_impl(plan, SA, SB, ws, run_flags, s);
        if (st != MXGEMM_OK)
            return st;
    }

    // (2) the GEMM, with operand roles per the plan
    const void *pa = plan->swap ? B : A;
    const void *pb = plan->swap ? A : B;
    const int64_t rows_a = plan->swap ? N : M;
    const int64_t rows_b = plan->swap ? M : N;
    // single-CTA tiles: 2-D maps, one k-stage per box; CTA pairs: 3-D maps, two per box
    if (plan->map_ptr_a != pa) {
        const int r = plan->mode ? encode_operand_map_2stage(&plan->map_a, pa, rows_a, row_bytes, 128)
                                 : encode_operand_map(&plan->map_a, pa, rows_a, row_bytes, 128);
        if (r != MXGEMM_OK)
            return MXGEMM_ERR_CUDA;
        plan->map_ptr_a = pa;
    }
    if (plan->map_ptr_b != pb) {
        const int r = plan->mode ? encode_operand_map_2stage(&plan->map_b, pb, rows_b, row_bytes, plan->bn / 2)
                                 : encode_operand_map(&plan->map_b, pb, rows_b, row_bytes, plan->bn);
        if (r != MXGEMM_OK)
            return MXGEMM_ERR_CUDA;
        plan->map_ptr_b = pb;
    }

    GemmParams p;
    memset(&p, 0, sizeof p);
    p.rows_a = static_cast<int>(rows_a);
    p.rows_b = static_cast<int>(rows_b);
    p.num_kt = static_cast<int>(bf16 ? K / 64 : K / 128);  // BF16: one "K-tile" per 64-value stage
    p.kstages = plan->kstages;
    p.kstages_per_split = plan->kstages_per_split;
    p.tiles_m = plan->tiles_m;
    p.tiles_n = plan->tiles_n;
    p.splits = plan->splits;
    p.group_m = plan->group_m;
    p.test_stall = test_stall;
    // An A-role tile is read once per B-role tile column and vice versa (in pair
    // mode one load of a B-role tile serves the pair).
    p.stream_a = plan->tiles_n <= 2 ? 1 : 0;
    p.stream_b = plan->tiles_m <= 2 ? 1 : 0;
    p.sfa = plan->swap ? sfb : sfa;
    p.sfb = plan->swap ? sfa : sfb;
    p.stride_i = plan->swap ? 1 : N;
    p.stride_j = plan->swap ? N : 1;
    p.timeout_ns = timeout_ns;
    p.status = dev->status_ptr;
    p.dp_tiles = plan->dp_tiles;
    p.sk_ctas = plan->sk_ctas;
    p.sk_stages = static_cast<long long>(plan->sk_tiles) * plan->kstages;
    p.sk_counters = plan->cnt_pool >= 0 ? dev->counters_ptr + plan->cnt_pool : sk_counters;
    p.sk_partials = reinterpret_cast<float *>(ws + plan->off_skp);
    const bool split = plan->splits > 1;
    const int osize = split ? 4 : (plan->out == MXGEMM_OUT_BF16 ? 2 : 4);
    if (split) {
        p.out = ws + plan->off_part;
        p.out_kind = mxg::OUT_F32;
        p.split_stride = (M * N + 7) & ~7ll;  // keeps every slab 32-byte aligned
    } else {
        p.out = C;
        p.out_kind = plan->out == MXGEMM_OUT_BF16 ? mxg::OUT_BF16 : mxg::OUT_F32;
        p.split_stride = 0;
    }
    p.vec_ok = vec_level(!plan->swap, N * osize, p.out);
    // the lean decode form may load the weight (B, its A role) before the grid wait
    p.early_a = (plan->lean && plan->swap && (run_flags & MXGEMM_RUN_B_STATIC)) ? 1 : 0;
    p.dbg_out_elems = split ? static_cast<long long>(plan->splits) * p.split_stride : M * N;
    p.dbg_out_elems -= static_cast<long long>(dbg_short_rows) * N;
    p.dbg_skp_elems = plan->sk_ctas > 0 ? 2ll * plan->sk_ctas * plan->sk_halves * 128 * plan->bn : 0;
    p.dbg_counters = plan->sk_ctas > 0 ? plan->cnt_n : 0;
#ifdef MXGEMM_DEBUG
    // C pre-filled with NaN (all-ones bytes in BF16 and FP32): an element that
    // no kernel writes reads back as NaN
    if (cudaMemsetAsync(C, 0xFF, static_cast<size_t>(M * N) * (plan->out == MXGEMM_OUT_BF16 ? 2 : 4), s) !=
        cudaSuccess)
        return MXGEMM_ERR_CUDA;
#endif

    cudaError_t e;
    if (plan->mode == 1 && bf16) {
        // the kernel reads no scale maps for BF16; pass valid descriptors anyway
        e = mxg::launch_gemm_pair_bf16(plan->bn, p, plan->map_a, plan->map_b, plan->map_a, plan->map_b, plan->map_a,
                                       plan->grid, s);
    } else if (plan->mode == 1) {
        const int ktps = fp4 ? 2 : 1;
        if (plan->map_ptr_sfa != p.sfa) {
            if (encode_sf_map(&plan->map_sfa, p.sfa, rows_a, K, ktps, 1) != MXGEMM_OK)
                return MXGEMM_ERR_CUDA;
            plan->map_ptr_sfa = p.sfa;
        }
        if (plan->map_ptr_sfb != p.sfb) {
            if (encode_sf_map(&plan->map_sfb, p.sfb, rows_b, K, ktps, static_cast<int>(ceil_div(plan->bn, 128))) !=
                MXGEMM_OK)
                return MXGEMM_ERR_CUDA;
            plan->map_ptr_sfb = p.sfb;
        }
        if (fused && plan->map_ptr_sarm != SA) {
            if (encode_rowmajor_sf_map(&plan->map_sarm, SA, M, K, ktps) != MXGEMM_OK)
                return MXGEMM_ERR_CUDA;
            plan->map_ptr_sarm = SA;
        }
        p.sa_fused = fused ? 1 : 0;
        const CUtensorMap &msarm = fused ? plan->map_sarm : plan->map_sfa;  // not read unless fused
        e = fp4 ? mxg::launch_gemm_pair_fp4(plan->bn, p, plan->map_a, plan->map_b, plan->map_sfa, plan->map_sfb,
                                            msarm, plan->grid, s)
                : mxg::launch_gemm_pair_fp8(plan->bn, p, plan->map_a, plan->map_b, plan->map_sfa, plan->map_sfb,
                                            msarm, plan->grid, s);
    } else if (bf16)
        e = mxg::launch_gemm_bf16(plan->bn, plan->lean != 0, p, plan->map_a, plan->map_b, plan->grid, s);
    else
        e = fp4 ? mxg::launch_gemm_fp4(plan->bn, plan->lean != 0, p, plan->map_a, plan->map_b, plan->grid, s)
                : mxg::launch_gemm_fp8(plan->bn, plan->lean != 0, p, plan->map_a, plan->map_b, plan->grid, s);
    if (e != cudaSuccess)
        return MXGEMM_ERR_CUDA;

    // (3) split-K reduce
    if (split) {
        const long long n = M * N;
        const long long n4 = n / 4;
        int blocks = static_cast<int>(std::min<long long>(std::max<long long>(1, (n4 + 255) / 256),
                                                          static_cast<long long>(plan->num_sms) * 8));
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = mxg::launch_config(blocks, 256, 0, s, attr, 1);
        if (cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, reinterpret_cast<const float *>(ws + plan->off_part),
                               plan->splits, n, (n + 7) & ~7ll, static_cast<void *>(C),
                               plan->out == MXGEMM_OUT_BF16 ? static_cast<int>(mxg::OUT_BF16)
                                                            : static_cast<int>(mxg::OUT_F32)) != cudaSuccess)
            return MXGEMM_ERR_CUDA;
    }
    return debug_finish(s);
}

int mxgemm_prepare(mxgemm_plan_t plan, const uint8_t *SA, const uint8_t *SB, void *workspace, size_t ws_bytes,
                   uint32_t run_flags, void *stream)
{
    if (!plan)
        return MXGEMM_ERR_ARG;
    if (run_flags & ~(MXGEMM_RUN_SA_PRELAYOUT | MXGEMM_RUN_SB_PRELAYOUT))
        return MXGEMM_ERR_ARG;
    const bool bf16 = plan->fmt == MXGEMM_FMT_BF16;
    const bool read_sa = !bf16 && !(run_flags & MXGEMM_RUN_SA_PRELAYOUT);
    const bool read_sb = !bf16 && !(run_flags & MXGEMM_RUN_SB_PRELAYOUT);
    if ((read_sa && !SA) || (read_sb && !SB))
        return MXGEMM_ERR_ARG;
    if ((read_sa && !aligned16(SA)) || (read_sb && !aligned16(SB)))
        return MXGEMM_ERR_ALIGN;
    if (plan->ws_bytes > 0 && (workspace == nullptr || ws_bytes < plan->ws_bytes))
        return MXGEMM_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace))
        return MXGEMM_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    int st = device_info(&dev);
    if (st != MXGEMM_OK)
        return st;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device)
        return MXGEMM_ERR_ARG;
    return prepare_impl(plan, SA, SB, static_cast<uint8_t *>(workspace), run_flags, static_cast<cudaStream_t>(stream));
}

int mxgemm_run(mxgemm_plan_t plan, const void *A, const uint8_t *SA, const void *B, const uint8_t *SB, void *C,
               void *workspace, size_t ws_bytes, uint32_t run_flags, void *stream)
{
    return run_impl(plan, A, SA, B, SB, C, workspace, ws_bytes, run_flags, stream, 0, MXGEMM_WAIT_LIMIT_NS);
}

int mxgemm_selftest_stall(mxgemm_plan_t plan, const void *A, const uint8_t *SA, const void *B, const uint8_t *SB,
                          void *C, void *workspace, size_t ws_bytes, void *stream)
{
    return run_impl(plan, A, SA, B, SB, C, workspace, ws_bytes, MXGEMM_RUN_SA_PRELAYOUT | MXGEMM_RUN_SB_PRELAYOUT,
                    stream, 1, 20000000ull);
}

int mxgemm_selftest_bounds(mxgemm_plan_t plan, const void *A, const uint8_t *SA, const void *B, const uint8_t *SB,
                           void *C, void *workspace, size_t ws_bytes, uint32_t run_flags, void *stream)
{
#ifdef MXGEMM_DEBUG
    if (!plan)
        return MXGEMM_ERR_ARG;
    if (plan->splits > 1)
        return MXGEMM_ERR_UNSUPPORTED;  // C is written by the reduce pass, not the GEMM kernel
    return run_impl(plan, A, SA, B, SB, C, workspace, ws_bytes, run_flags, stream, 0, MXGEMM_WAIT_LIMIT_NS, 1);
#else
    (void)plan, (void)A, (void)SA, (void)B, (void)SB, (void)C, (void)workspace, (void)ws_bytes, (void)run_flags,
        (void)stream;
    return MXGEMM_ERR_UNSUPPORTED;
#endif
}

int mxgemm_debug_build(void)
{
#ifdef MXGEMM_DEBUG
    return 1;
#else
    return 0;
#endif
}

// ------------------------------------------------------------- no-alloc --
// Scratch for mxgemm_run_noalloc: a fixed, file-scope device array, so callers
// that cannot allocate device memory still get the relayout and split-K space
// mxgemm_run takes from its workspace argument.  Host code never dereferences
// the symbol itself; it passes the device address found by
// cudaGetSymbolAddress (looked up once per device, with that device current).
static __device__ __align__(256) uint8_t g_noalloc_scratch[MXGEMM_NOALLOC_SCRATCH_BYTES];

namespace {
void *g_noalloc_addr[kMaxDevices];
std::mutex g_noalloc_mutex;
}  // namespace

int mxgemm_run_noalloc(mxgemm_plan_t plan, const void *A, const uint8_t *SA, const void *B, const uint8_t *SB,
                       void *C, uint32_t run_flags, void *stream)
{
    if (!plan || (run_flags & MXGEMM_RUN_PREPARED))  // the scratch is not the caller's to prepare
        return MXGEMM_ERR_ARG;
    if (plan->ws_bytes > MXGEMM_NOALLOC_SCRATCH_BYTES)
        return MXGEMM_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return MXGEMM_ERR_CUDA;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (g_noalloc_addr[dev] == nullptr) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
                return MXGEMM_ERR_CUDA;
            g_noalloc_addr[dev] = p;
        }
        scratch = g_noalloc_addr[dev];
    }
    return run_impl(plan, A, SA, B, SB, C, scratch, MXGEMM_NOALLOC_SCRATCH_BYTES, run_flags, stream, 0,
                    MXGEMM_WAIT_LIMIT_NS);
}

// ------------------------------------------------------------ grouped --
int mxgemm_grouped_plan_create(mxgemm_grouped_plan_t *plan, int64_t groups, int64_t rows, int64_t N, int64_t K,
                               int fmt, int out, uint32_t flags)
{
    if (!plan)
        return MXGEMM_ERR_ARG;
    *plan = nullptr;
    if ((fmt != MXGEMM_FMT_MXFP8_E4M3 && fmt != MXGEMM_FMT_MXFP4_E2M1) ||
        (out != MXGEMM_OUT_F32 && out != MXGEMM_OUT_BF16))
        return MXGEMM_ERR_ARG;
    const uint32_t known = MXGEMM_PLAN_FORCE_BN128 | MXGEMM_PLAN_FORCE_BN256 | MXGEMM_PLAN_FORCE_NOSWAP |
                           MXGEMM_PLAN_FORCE_SWAP | MXGEMM_PLAN_FORCE_PAIR | MXGEMM_PLAN_FORCE_SINGLE;
    if ((flags & ~known) != 0 || ((flags & MXGEMM_PLAN_FORCE_SWAP) && (flags & MXGEMM_PLAN_FORCE_NOSWAP)) ||
        ((flags & MXGEMM_PLAN_FORCE_BN128) && (flags & MXGEMM_PLAN_FORCE_BN256)) ||
        ((flags & MXGEMM_PLAN_FORCE_PAIR) && (flags & MXGEMM_PLAN_FORCE_SINGLE)))
        return MXGEMM_ERR_ARG;
    if (groups < 1 || groups > mxg::kMaxGroups || rows < 1 || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0)
        return MXGEMM_ERR_SHAPE;
    if (rows > (1ll << 30) || groups * N > (1ll << 30) || K > (1ll << 30) ||
        (ceil_div(rows, 32) + groups) * ceil_div(N, 32) >= (1ll << 31))
        return MXGEMM_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    const int st = device_info(&dev);
    if (st != MXGEMM_OK)
        return st;
    mxgemm_grouped_plan *p = new (std::nothrow) mxgemm_grouped_plan();
    if (!p)
        return MXGEMM_ERR_UNSUPPORTED;
    p->G = groups;
    p->T = rows;
    p->N = N;
    p->K = K;
    p->fmt = fmt;
    p->out = out;
    p->num_sms = dev->num_sms;
    cudaGetDevice(&p->device);
    // Expected tokens per group: few -> the weights fill the 128-row MMA dimension.
    const int64_t avg = std::max<int64_t>(1, rows / groups);
    int swap = avg <= 64 ? 1 : 0;
    if (flags & MXGEMM_PLAN_FORCE_SWAP) swap = 1;
    if (flags & MXGEMM_PLAN_FORCE_NOSWAP) swap = 0;
    p->swap = swap;
    // Token tiles in the B role are at least 64 rows: a B-role tile that starts
    // 32 rows into its 128-row scale chunk would put the MMA's B scale factors at
    // an odd TMEM column, which the hardware rejects (misaligned address).
    int bn = swap ? std::min(std::max(pick_bn(avg), 64), 128) : (N >= 256 ? 256 : 128);
    if (flags & MXGEMM_PLAN_FORCE_BN128) bn = 128;
    if (flags & MXGEMM_PLAN_FORCE_BN256) bn = 256;
    // Prefill-sized groups (>= 512 tokens on average) run 256 x 256 CTA-pair
    // tiles: half the B-role operand bytes per FLOP of a 128 x 256 tile.
    int mode = (!swap && avg >= 512) ? 1 : 0;
    if (flags & MXGEMM_PLAN_FORCE_PAIR) mode = 1;
    if (flags & (MXGEMM_PLAN_FORCE_SINGLE | MXGEMM_PLAN_FORCE_BN128)) mode = 0;
    if (swap || N < 256 || (fmt == MXGEMM_FMT_MXFP4_E2M1 && K % 256 != 0)) mode = 0;
    if (mode == 1) {
        bn = 256;
        p->clusters = fmt == MXGEMM_FMT_MXFP4_E2M1 ? mxg::gemm_grouped_pair_max_clusters_fp4()
                                                   : mxg::gemm_grouped_pair_max_clusters_fp8();
        if (p->clusters < 1)
            mode = 0;
    }
    p->mode = mode;
    p->bn = bn;
    p->kstages = static_cast<int>(fmt == MXGEMM_FMT_MXFP4_E2M1 ? ceil_div(K, 256) : K / 128);
    p->tok_sf_cap = static_cast<int>(ceil_div(rows, 128) + groups);
    p->off_tok_sf = 0;
    p->off_w_sf = align256(static_cast<size_t>(p->tok_sf_cap) * 128 * static_cast<size_t>(K / 32));
    p->ws_bytes = align256(p->off_w_sf + static_cast<size_t>(groups * N) * static_cast<size_t>(K / 32));
    *plan = p;
    return MXGEMM_OK;
}

int mxgemm_grouped_plan_destroy(mxgemm_grouped_plan_t plan)
{
    delete plan;
    return MXGEMM_OK;
}

size_t mxgemm_grouped_workspace_bytes(mxgemm_grouped_plan_t plan) { return plan ? plan->ws_bytes : 0; }

int mxgemm_grouped_plan_describe(mxgemm_grouped_plan_t plan, char *buf, size_t len)
{
    if (!plan || !buf || len == 0)
        return MXGEMM_ERR_ARG;
    const bool fp4 = plan->fmt == MXGEMM_FMT_MXFP4_E2M1;
    const bool pair = plan->mode == 1;
    mxg::KernelInfo ki = pair ? (fp4 ? mxg::gemm_grouped_pair_info_fp4() : mxg::gemm_grouped_pair_info_fp8())
                              : (fp4 ? mxg::gemm_info_fp4(plan->bn) : mxg::gemm_info_fp8(plan->bn));
    snprintf(buf, len,
             "grouped fmt=%s out=%s groups=%lld rows=%lld N=%lld K=%lld tile=%dx%d mode=%s swap_ab=%d kstages=%d "
             "grid=%d%s stages=%d acc_stages=%d smem=%d",
             fp4 ? "mxfp4" : "mxfp8", plan->out == MXGEMM_OUT_BF16 ? "bf16" : "f32", static_cast<long long>(plan->G),
             static_cast<long long>(plan->T), static_cast<long long>(plan->N), static_cast<long long>(plan->K),
             pair ? 256 : 128, plan->bn, pair ? "pair" : "single", plan->swap, plan->kstages,
             pair ? plan->clusters : plan->num_sms, pair ? "x2" : "", ki.stages, ki.acc_stages, ki.smem_bytes);
    return MXGEMM_OK;
}

int mxgemm_grouped_run(mxgemm_grouped_plan_t plan, const int64_t *group_offsets, const void *A, const uint8_t *SA,
                       const void *B, const uint8_t *SB, void *C, void *workspace, size_t ws_bytes, uint32_t run_flags,
                       void *stream)
{
    if (!plan || !group_offsets || !A || !SA || !B || !SB || !C)
        return MXGEMM_ERR_ARG;
    if (run_flags & ~MXGEMM_RUN_SB_PRELAYOUT)
        return MXGEMM_ERR_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(SA) || !aligned16(SB) ||
        (reinterpret_cast<uintptr_t>(group_offsets) & 7u) != 0)
        return MXGEMM_ERR_ALIGN;
    if (workspace == nullptr || ws_bytes < plan->ws_bytes)
        return MXGEMM_ERR_WORKSPACE;
    if (!aligned16(workspace))
        return MXGEMM_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    int st = device_info(&dev);
    if (st != MXGEMM_OK)
        return st;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device)
        return MXGEMM_ERR_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const bool fp4 = plan->fmt == MXGEMM_FMT_MXFP4_E2M1;
    const int64_t G = plan->G, T = plan->T, N = plan->N, K = plan->K;
    const int64_t row_bytes = fp4 ? K / 2 : K;
    const int num_kt = static_cast<int>(K / 128);
    const long long *offs = reinterpret_cast<const long long *>(group_offsets);

    // (1) token scales -> per-group tile blocks; (2) weight scales -> tile layout
    uint8_t *tok_sf = ws + plan->off_tok_sf;
    {
        const int blocks_x = static_cast<int>(ceil_div(num_kt, kRelayoutKt));
        grouped_relayout_kernel<<<static_cast<unsigned>(plan->tok_sf_cap) * blocks_x, 256, 0, s>>>(
            SA, offs, static_cast<int>(G), static_cast<int>(T), num_kt, blocks_x, plan->tok_sf_cap, tok_sf);
        if (cudaGetLastError() != cudaSuccess)
            return MXGEMM_ERR_CUDA;
    }
    const uint8_t *w_sf = SB;
    if (!(run_flags & MXGEMM_RUN_SB_PRELAYOUT)) {
        RelayoutJob j = make_job(SB, G * N, K, ws + plan->off_w_sf);
        if (launch_relayout(j, nullptr, s) != cudaSuccess)
            return MXGEMM_ERR_CUDA;
        w_sf = ws + plan->off_w_sf;
    }

    // (3) the GEMM: tokens in the A role (128-row tiles) or, swapped, the B role
    if (plan->map_ptr_tok != A) {
        if (encode_operand_map(&plan->map_tok, A, T, row_bytes, plan->swap ? plan->bn : 128) != MXGEMM_OK)
            return MXGEMM_ERR_CUDA;
        plan->map_ptr_tok = A;
    }
    if (plan->map_ptr_w != B) {
        if (encode_operand_map(&plan->map_w, B, G * N, row_bytes, plan->swap ? 128 : plan->bn) != MXGEMM_OK)
            return MXGEMM_ERR_CUDA;
        plan->map_ptr_w = B;
    }
    GemmParams p;
    memset(&p, 0, sizeof p);
    p.rows_a = static_cast<int>(plan->swap ? G * N : T);
    p.rows_b = static_cast<int>(plan->swap ? T : G * N);
    p.num_kt = num_kt;
    p.kstages = plan->kstages;
    p.kstages_per_split = plan->kstages;
    p.tiles_m = 1;
    p.tiles_n = 1;
    p.splits = 1;
    p.group_m = 8;
    p.out = C;
    p.out_kind = plan->out == MXGEMM_OUT_BF16 ? mxg::OUT_BF16 : mxg::OUT_F32;
    const int osize = plan->out == MXGEMM_OUT_BF16 ? 2 : 4;
    p.stride_i = plan->swap ? 1 : N;
    p.stride_j = plan->swap ? N : 1;
    p.vec_ok = vec_level(!plan->swap, N * osize, C);
    // the weights are streamed when each group has at most two token tiles
    const int64_t avg = std::max<int64_t>(1, T / G);
    const bool stream_w = ceil_div(avg, plan->swap ? plan->bn : 128) <= 2;
    p.stream_a = (plan->swap && stream_w) ? 1 : 0;
    p.stream_b = (!plan->swap && stream_w) ? 1 : 0;
    p.sfa = plan->swap ? w_sf : tok_sf;
    p.sfb = plan->swap ? tok_sf : w_sf;
    p.timeout_ns = MXGEMM_WAIT_LIMIT_NS;
    p.status = dev->status_ptr;
    p.grouped = 1;
    p.groups = static_cast<int>(G);
    p.tok_b = plan->swap;
    p.group_n = static_cast<int>(N);
    p.rows_total = static_cast<int>(T);
    p.tok_sf_cap = plan->tok_sf_cap;
    p.group_offsets = offs;
    p.dbg_out_elems = static_cast<long long>(T) * N;
    if (plan->mode == 1) {
        // CTA-pair tiles: 3-D operand maps (two 128-byte K-slices a box; 128
        // token rows, 128 weight rows a box) and 3-D maps of both scale regions
        const int ktps = fp4 ? 2 : 1;
        if (plan->map_ptr_tok3 != A) {
            if (encode_operand_map_2stage(&plan->map_tok3, A, T, row_bytes, 128) != MXGEMM_OK)
                return MXGEMM_ERR_CUDA;
            plan->map_ptr_tok3 = A;
        }
        if (plan->map_ptr_w3 != B) {
            if (encode_operand_map_2stage(&plan->map_w3, B, G * N, row_bytes, 128) != MXGEMM_OK)
                return MXGEMM_ERR_CUDA;
            plan->map_ptr_w3 = B;
        }
        if (plan->map_ptr_sftok != tok_sf) {
            if (encode_sf_map(&plan->map_sftok, tok_sf, static_cast<int64_t>(plan->tok_sf_cap) * 128, K, ktps, 1) !=
                MXGEMM_OK)
                return MXGEMM_ERR_CUDA;
            plan->map_ptr_sftok = tok_sf;
        }
        if (plan->map_ptr_sfw != w_sf) {
            if (encode_sf_map(&plan->map_sfw, w_sf, G * N, K, ktps, 2) != MXGEMM_OK)
                return MXGEMM_ERR_CUDA;
            plan->map_ptr_sfw = w_sf;
        }
        p.stream_a = 0;
        p.stream_b = stream_w ? 1 : 0;
        const cudaError_t e =
            fp4 ? mxg::launch_gemm_grouped_pair_fp4(p, plan->map_tok3, plan->map_w3, plan->map_sftok, plan->map_sfw,
                                                    plan->clusters, s)
                : mxg::launch_gemm_grouped_pair_fp8(p, plan->map_tok3, plan->map_w3, plan->map_sftok, plan->map_sfw,
                                                    plan->clusters, s);
        return e == cudaSuccess ? debug_finish(s) : MXGEMM_ERR_CUDA;
    }
    const CUtensorMap &ma = plan->swap ? plan->map_w : plan->map_tok;
    const CUtensorMap &mb = plan->swap ? plan->map_tok : plan->map_w;
    const cudaError_t e = fp4 ? mxg::launch_gemm_grouped_fp4(plan->bn, p, ma, mb, plan->num_sms, s)
                              : mxg::launch_gemm_grouped_fp8(plan->bn, p, ma, mb, plan->num_sms, s);
    return e == cudaSuccess ? debug_finish(s) : MXGEMM_ERR_CUDA;
}

int mxgemm_placement_scan(int k, const int *sa, const int *sb, int npairs, long long *counts, long long *first_diff,
                          void *stream)
{
    if (!sa || !sb || !counts || !first_diff)
        return MXGEMM_ERR_ARG;
    if (k < 1 || k > 4 || npairs < 1 || npairs > (1 << 24))
        return MXGEMM_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(sa) & 3u) || (reinterpret_cast<uintptr_t>(sb) & 3u) ||
        (reinterpret_cast<uintptr_t>(counts) & 7u) || (reinterpret_cast<uintptr_t>(first_diff) & 7u))
        return MXGEMM_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    const int st = device_info(&dev);
    if (st != MXGEMM_OK)
        return st;
    return mxg::launch_placement_scan(k, sa, sb, npairs, counts, first_diff, dev->num_sms,
                                      static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MXGEMM_OK
               : MXGEMM_ERR_CUDA;
}

int mxgemm_device_status(void *stream, int reset)
{
    DeviceInfo *dev = nullptr;
    int st = device_info(&dev);
    if (st != MXGEMM_OK)
        return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess)
        return MXGEMM_ERR_CUDA;
    if (reset) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess)
            return MXGEMM_ERR_CUDA;
        // a launch that gave up may have left stream-K arrival counters nonzero
        if (v == MXGEMM_ERR_DEVICE_TIMEOUT &&
            (cudaMemset(dev->counters_ptr, 0, sizeof(int) * kCounterPool) != cudaSuccess ||
             cudaDeviceSynchronize() != cudaSuccess))
            return MXGEMM_ERR_CUDA;
    }
    return v;
}

}  // extern "C"
