// gemm_kernel.cuh -- the persistent, warp-specialised MX block-scaled GEMM for
// sm_103a (tcgen05 tensor cores, TMA, TMEM accumulators).
//
// Computes D[i, j] = sum_k a_i[k] * b_j[k] with a per-32 E8M0 scale on each
// operand, i over the rows of the "A role" operand (the MMA M dimension, 128
// per tile) and j over the rows of the "B role" operand (the MMA N dimension,
// BN per tile).  Normally the A role is the GEMM's A and the B role its B; for
// small token counts the host swaps them (C^T = B * A^T) so that the weight
// fills the 128-row MMA dimension.
//
// Operation: the MXFP8 / MXFP4 scaled GEMM of "Accelerating PyTorch on AMD
// GPUs with FlyDSL" (English digest, section "API compatibility is not
// universal input coverage": E8M0 scale per 32 values along K, K % 128 == 0),
// FP32 accumulation (AI-compiler daily 2026-10-22, item 1).  The page's own
// kernel (half-tile-interleaved LDS pipeline on MI355X, section "Explicit
// layouts bring optimization close to hardware") is replaced here by a TMA ->
// shared-memory ring -> tcgen05.mma pipeline with mbarrier hand-off.
//
// Warp roles (320 threads; 384 with the stream-K fixup warps):
//   warp 0      TMA producer: per k-stage, A and B tiles (128-byte swizzle) and
//               the tile-layout scale chunks (bulk copies) into ring slot s.
//   warp 1      TMEM owner and MMA issuer: per k-stage, tcgen05.cp of the scale
//               chunks into TMEM, then BK/32 (MXFP8) or BK/64 (MXFP4)
//               block-scaled MMAs accumulating in TMEM; commits free the slot.
//   warps 2..9  epilogue: warp w owns TMEM lane quarter w%4 and one half of the
//               tile's columns; it loads its whole share of the accumulator into
//               registers, releases the TMEM stage to the MMA warp at once, and
//               only then converts (BF16) and stores to global (masked edges), so
//               the stores overlap the next tile's MMAs.
//   warps 10,11 stream-K fixup: add the partial sums of a tile cut between CTAs
//               (posted by the epilogue when this CTA's segment arrived last)
//               and store it, concurrently with everything else.  Tiles of at
//               most 64 columns have the epilogue warps add them instead.
// The lean form (weight-streaming decode, 192 threads) keeps warps 0 and 1 and
// four epilogue warps that own all the tile's columns and add cut tiles
// themselves; its ring fits two CTAs on an SM.
// Every mbarrier wait is bounded in time; on expiry the CTA records
// MXGEMM_ERR_DEVICE_TIMEOUT in *status, drains its in-flight copies and MMAs,
// frees its TMEM and exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace mxg {

constexpr int kEpiWarps = 8;  // epilogue warps (two per TMEM lane quarter)
constexpr int kFixWarps = 2;  // stream-K fixup warps (one per column half)
constexpr int kFixWarp0 = 2 + kEpiWarps;
constexpr int kThreads = 64 + 32 * kEpiWarps;         // producer + MMA + epilogue
constexpr int kThreadsSk = kThreads + 32 * kFixWarps;  // ... + stream-K fixup warps
// Both allow 168 registers a thread (10 or 12 warps over the four SM
// sub-partitions), but the 128 x 256 single-CTA tile only fits without spills in
// the 10-warp form, so it has a separate stream-K instantiation.
constexpr int kBM = 128;            // MMA M (rows of the A role per tile)
constexpr int kRowBytes = 128;      // bytes of one operand row per k-stage
constexpr int kSfChunk = 512;       // bytes of one scale chunk (128 rows x 4 K-blocks)
constexpr int kSmemBudget = 232448; // 227 KiB opt-in shared memory per block
// The lean form of the single-CTA kernel (weight-streaming decode tiles of 32
// or 64 columns; the planner uses it for 32): four epilogue warps, no fixup
// warps, a ring that leaves room for a second CTA on the SM and at most 256
// TMEM columns, so that the next GEMM's CTAs can be resident (allocated, L2
// warmed, waiting on the grid dependency) while this one drains.
constexpr int kLeanEpiWarps = 4;
constexpr int kLeanThreads = 64 + 32 * kLeanEpiWarps;
constexpr int kLeanSmemBudget = 112 * 1024;
// Scale factors travel in groups of kSfGroup k-stages: one copy per operand
// brings a group's chunks into one of two shared-memory group slots, and the
// MMA warp moves the whole group into TMEM at the group's first stage.  A TMA
// or bulk copy has a fixed cost of its own, and per-stage scale copies (three
// small ones per k-stage beside two operand tiles) cost more main-loop time
// than the operand tiles themselves (measured: skipping them took a long-K
// CTA-pair GEMM from 0.359 to 0.320 us per k-stage).
constexpr int kSfGroup = 4;

enum OutKind : int { OUT_F32 = 0, OUT_BF16 = 1 };

struct GemmParams {
    int rows_a;               // extent of the A role (MMA M)
    int rows_b;               // extent of the B role (MMA N)
    int num_kt;               // K / 128: scale K-tiles
    int kstages;              // k-stages over the whole K (FP8: K/128, FP4: ceil(K/256))
    int kstages_per_split;    // k-stages per split (the last split may get fewer)
    int tiles_m, tiles_n, splits;
    int group_m;              // raster: tiles of the A role walked together
    int out_kind;             // OutKind
    int vec_ok;               // stride_j == 1 and rows 16-byte (1) or 32-byte (2) aligned; else 0
    int test_stall;           // self-test: the producer issues nothing (waits expire)
    int stream_a, stream_b;   // 1: that operand is read by at most two tiles (load it evict-first)
    int sa_fused;             // CTA-pair kernel: 1 = A-role scales are row-major (laid out in the kernel)
    int early_a;              // lean form: 1 = no preceding kernel writes the A-role operand, so the
                              // first ring of its tiles is loaded before the grid dependency wait
    const uint8_t *sfa;       // tile-layout scales of the A role
    const uint8_t *sfb;       // tile-layout scales of the B role
    void *out;                // output base (C, or split-K partial slabs)
    long long stride_i;       // elements between consecutive A-role rows in out
    long long stride_j;       // elements between consecutive B-role rows in out
    long long split_stride;   // elements between split partial slabs (0: no split)
    unsigned long long timeout_ns;
    int *status;              // sticky device status word
    // Stream-K: the first dp_tiles tiles in raster order are computed whole,
    // round-robin over the grid; the k-stages of the remaining tiles are divided
    // evenly over CTAs (CTA pairs, in the pair kernel) 0..sk_ctas-1.  A tile cut between CTAs is
    // finished by the last of them to arrive, which adds the others' FP32 partial
    // sums in k order (deterministic).  sk_ctas == 0: no stream-K phase.
    int dp_tiles;
    int sk_ctas;
    long long sk_stages;      // (tiles - dp_tiles) * kstages
    int *sk_counters;         // one arrival counter per stream-K tile and 128-row share, zero at launch
    float *sk_partials;       // two 128 x BN FP32 slots per stream-K CTA (per CTA of a pair)
    // Grouped (mixture-of-experts) GEMM (single-CTA kernel, or the pair kernel
    // with the tokens in the A role): group e owns the token rows
    // [off[e], off[e+1]) of A and C and the weight rows [e*group_n,
    // (e+1)*group_n) of B.  Offsets are read on the device and sanitised
    // (clamped to [0, rows_total], end >= start) before use.
    int grouped;              // 0: plain GEMM
    int groups;               // G <= kMaxGroups
    int tok_b;                // 1: the tokens are the B role (swap-AB), 0: the A role
    int group_n;              // weight rows per group, a multiple of 128
    int rows_total;           // T: rows of A and C
    int tok_sf_cap;           // 128-row blocks in the tokens' tile-layout scale region
    const long long *group_offsets;  // G + 1 row offsets (device)
    // Extents of the buffers the kernels reach with plain loads and stores,
    // set for every launch; a debug build (MXGEMM_DEBUG) checks each such
    // access against them (dbg_ok below).
    long long dbg_out_elems;  // elements addressable from out
    long long dbg_skp_elems;  // floats in sk_partials
    long long dbg_counters;   // ints in sk_counters
};

constexpr int kMaxGroups = 512;

// Per-CTA table of the groups, built once at kernel start from the offsets.
struct GroupTable {
    int tile_start[kMaxGroups + 1];  // first global tile of each group (prefix sum)
    int tok_rb[kMaxGroups + 1];      // first 128-row block of each group's token scales
    int row0[kMaxGroups];            // sanitised first token row
    int rows[kMaxGroups];            // sanitised token row count
};

// One warp scans the groups: sanitise each group's rows from the offsets, count
// its tiles (token tiles of tok_tile rows x w_tiles weight tiles) and its
// 128-row scale blocks, and write the exclusive prefix sums; entry G of
// tile_start / tok_rb holds the totals.  Sanitising: a group starts at its
// offset clamped to [0, T] but not before the end of any earlier group, and
// ends at the next offset clamped to [start, T].  For valid (non-decreasing,
// in-range) offsets this is the identity; for any others the groups stay
// disjoint inside [0, T], so the totals stay within what the plan validated.
// The GEMM and the grouped scale relayout both use it, so they agree on where
// each group's scales live whatever the offsets hold.
static __device__ __noinline__ void group_scan(const long long *offsets, int G, long long T, int tok_tile,
                                               int w_tiles, int lane, int *tile_start, int *tok_rb, int *row0,
                                               int *rows)
{
    int carry_t = 0, carry_b = 0;
    long long carry_end = 0;  // largest end of the groups already scanned
    for (int base = 0; base < G; base += 32) {
        const int e = base + lane;
        long long s = 0, end = 0;
        if (e < G) {
            s = min(max(offsets[e], 0ll), T);
            end = min(max(offsets[e + 1], s), T);
        }
        // exclusive prefix max of the ends (within the warp, then the carry)
        long long prev = end;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long x = __shfl_up_sync(0xFFFFFFFFu, prev, o);
            if (lane >= o) prev = max(prev, x);
        }
        long long before = __shfl_up_sync(0xFFFFFFFFu, prev, 1);
        if (lane == 0) before = 0;
        before = max(before, carry_end);
        carry_end = max(carry_end, __shfl_sync(0xFFFFFFFFu, prev, 31));
        int tiles = 0, blocks = 0, s0 = 0, m = 0;
        if (e < G) {
            const long long s2 = max(s, before);
            const long long end2 = max(end, s2);
            s0 = static_cast<int>(s2);
            m = static_cast<int>(end2 - s2);
            tiles = ((m + tok_tile - 1) / tok_tile) * w_tiles;
            blocks = (m + 127) / 128;
        }
        int ti = tiles, bi = blocks;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xFFFFFFFFu, ti, o);
            const int y = __shfl_up_sync(0xFFFFFFFFu, bi, o);
            if (lane >= o) {
                ti += x;
                bi += y;
            }
        }
        if (e < G) {
            if (tile_start) tile_start[e] = carry_t + ti - tiles;
            tok_rb[e] = carry_b + bi - blocks;
            row0[e] = s0;
            rows[e] = m;
        }
        carry_t += __shfl_sync(0xFFFFFFFFu, ti, 31);
        carry_b += __shfl_sync(0xFFFFFFFFu, bi, 31);
    }
    if (lane == 0) {
        if (tile_start) tile_start[G] = carry_t;
        tok_rb[G] = carry_b;
    }
}

template <int BN>
__device__ __forceinline__ void build_group_table(const GemmParams &p, GroupTable &g, int lane)
{
    const int tok_tile = p.tok_b ? BN : kBM;
    const int w_tiles = p.tok_b ? p.group_n / kBM : (p.group_n + BN - 1) / BN;
    group_scan(p.group_offsets, p.groups, p.rows_total, tok_tile, w_tiles, lane, g.tile_start, g.tok_rb, g.row0,
               g.rows);
}

// Element kind of the operands: MX block-scaled E4M3 or E2M1, or plain BF16.
enum ElemKind : int { K_MXFP8 = 0, K_MXFP4 = 1, K_BF16 = 2 };

template <int KIND, int BN, bool LEAN = false>
struct Cfg {
    static constexpr bool kFp4 = KIND == K_MXFP4;
    static constexpr bool kScaled = KIND != K_BF16;           // MX kinds carry E8M0 scales
    // A k-stage is 128 bytes of K per row: 128 E4M3, 256 E2M1 or 64 BF16 values.
    static constexpr int kKtPerStage = kFp4 ? 2 : 1;          // scale K-tiles per k-stage
    static constexpr int kSubPerKt = kFp4 ? 2 : 4;            // MMAs per K-tile (K = 32 B each)
    static constexpr int kChunksB = BN >= 128 ? BN / 128 : 1; // 128-row scale chunks of B per K-tile
    static constexpr int kABytes = kBM * kRowBytes;
    static constexpr int kBBytes = BN * kRowBytes;
    static constexpr int kStageBytes = kABytes + kBBytes;     // operand ring slot
    // scale group slot: SFA chunks [stage][K-tile], then SFB chunks [128-row block][stage][K-tile]
    static constexpr int kSfaGrpBytes = kScaled ? kSfGroup * kKtPerStage * kSfChunk : 0;
    static constexpr int kSfbGrpBytes = kScaled ? kChunksB * kSfGroup * kKtPerStage * kSfChunk : 0;
    static constexpr int kSfGrpBytes = kSfaGrpBytes + kSfbGrpBytes;
    static constexpr int kStagesRaw = ((LEAN ? kLeanSmemBudget : kSmemBudget) - 1024 - 256 - 2 * kSfGrpBytes) / kStageBytes;
    static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
    static constexpr int kSfaCols = kScaled ? 4 * kKtPerStage : 0;
    static constexpr int kSfbCols = kScaled ? 4 * kKtPerStage * kChunksB : 0;
    // Scale columns: one (SFA, SFB) region per stage of two scale groups, so the
    // copies of a group never overwrite scales that MMAs of the group before
    // still read (a group's regions are reused two groups later, after the MMAs
    // that read them have completed).
    static constexpr int kSfSlotCols = kSfaCols + kSfbCols;
    static constexpr int kSfRegions = kScaled ? 2 * kSfGroup : 0;
    static constexpr int kAccStages = (2 * BN + kSfRegions * kSfSlotCols <= 512) ? 2 : 1;
    static constexpr int kSfCol0 = kAccStages * BN;
    static constexpr int kColsUsed = kSfCol0 + kSfRegions * kSfSlotCols;
    static constexpr int kTmemCols = LEAN ? (kColsUsed <= 128 ? 128 : 256) : 512;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 2 * kSfGrpBytes + 256;
    static constexpr uint32_t kIdesc = kScaled ? idesc_block_scaled(kFp4 ? 1u : 0u, kBM, BN) : idesc_bf16(kBM, BN);
    static_assert(kStages >= 2, "shared memory too small for two stages");
    static_assert(kSfCol0 + kSfRegions * kSfSlotCols <= kTmemCols, "TMEM overflow");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN must be 32..256, multiple of 32");
    static_assert(!LEAN || (BN <= 64 && kColsUsed <= 256), "the lean form is for tiles of at most 64 columns");
};

__device__ __forceinline__ void tile_coords(const GemmParams &p, int unit, int &tm, int &tn, int &split)
{
    split = unit % p.splits;
    const int t = unit / p.splits;
    const int per_group = p.group_m * p.tiles_n;
    const int group = t / per_group;
    const int first_m = group * p.group_m;
    const int gsz = min(p.tiles_m - first_m, p.group_m);
    const int local = t - group * per_group;
    tm = first_m + local % gsz;
    tn = local / gsz;
}

// Raster position of tile t (grouped along the A role for L2 reuse).
__device__ __forceinline__ void tile_xy(const GemmParams &p, int t, int &tm, int &tn)
{
    const int per_group = p.group_m * p.tiles_n;
    const int group = t / per_group;
    const int first_m = group * p.group_m;
    const int gsz = min(p.tiles_m - first_m, p.group_m);
    const int local = t - group * per_group;
    tm = first_m + local % gsz;
    tn = local / gsz;
}

// One piece of work: k-stages [ks0, ks1) of tile (tm, tn).
struct Work {
    int tile, tm, tn, ks0, ks1;
    int grp;    // grouped GEMM: the group of the tile (tm, tn are group-local)
    int kind;   // 0: the whole K of the tile; 1: stream-K segment; 2: split-K slab
    int slot;   // kind 1: partial-sum slot (0: first segment of this CTA, 1: last)
                // kind 2: split index
};

// The sequence of Work of one CTA; producer, MMA and epilogue warps each walk
// an identical copy.
struct WorkIter {
    int u, step, units, spl, tok_tile;
    long long pos, end, begin;
    const GroupTable *gt;

    // gt: the group table (grouped GEMM only); tok_tile: token rows per tile.
    __device__ void init(const GemmParams &p, int cta, int ctas, const GroupTable *g = nullptr, int tok_tile_ = 0)
    {
        u = cta;
        step = ctas;
        gt = g;
        tok_tile = tok_tile_;
        spl = p.sk_ctas > 0 ? 1 : p.splits;
        units = p.sk_ctas > 0 ? p.dp_tiles : p.tiles_m * p.tiles_n * p.splits;
        if (g)
            units = g->tile_start[p.groups];
        pos = end = 0;
        if (p.sk_ctas > 0 && cta < p.sk_ctas) {
            pos = p.sk_stages * cta / p.sk_ctas;
            end = p.sk_stages * (cta + 1) / p.sk_ctas;
        }
        begin = pos;
    }

    // Grouped: the group holding global tile t (the last group whose first tile
    // is <= t, so empty groups are skipped), then the tile inside the group --
    // token tiles fastest, so neighbouring CTAs share a weight tile in L2.
    __device__ void group_xy(const GemmParams &p, int t, Work &w) const
    {
        int lo = 0, hi = p.groups - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (gt->tile_start[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int local = t - gt->tile_start[lo];
        const int ntok = max(1, (gt->rows[lo] + tok_tile - 1) / tok_tile);
        const int tok_i = local % ntok, w_i = local / ntok;
        w.grp = lo;
        w.tm = p.tok_b ? w_i : tok_i;
        w.tn = p.tok_b ? tok_i : w_i;
    }

    // Stream-K segments come first, so that the fixup of a cut tile (run by its
    // last CTA's epilogue or fixup warps) overlaps the whole tiles computed after it.
    __device__ bool next(const GemmParams &p, Work &w)
    {
        if (pos < end) {
            w.tile = p.dp_tiles + static_cast<int>(pos / p.kstages);
            w.ks0 = static_cast<int>(pos % p.kstages);
            w.ks1 = static_cast<int>(min(static_cast<long long>(p.kstages), w.ks0 + (end - pos)));
            w.kind = (w.ks0 == 0 && w.ks1 == p.kstages) ? 0 : 1;
            w.slot = pos == begin ? 0 : 1;
            w.grp = 0;
            tile_xy(p, w.tile, w.tm, w.tn);
            pos += w.ks1 - w.ks0;
            return true;
        }
        if (u < units) {
            w.tile = u / spl;
            w.slot = u % spl;
            w.ks0 = w.slot * p.kstages_per_split;
            w.ks1 = min(p.kstages, w.ks0 + p.kstages_per_split);
            w.kind = spl > 1 ? 2 : 0;
            w.grp = 0;
            if (gt)
                group_xy(p, w.tile, w);
            else
                tile_xy(p, w.tile, w.tm, w.tn);
            u += step;
            return true;
        }
        return false;
    }
};

// Where one tile's operands, scales and outputs live.  Epilogue indices: A-role
// row i = tm*128 + r and B-role row j = tn*BN + c are stored at
// out_base + i*stride_i + j*stride_j when i < lim_i and j < lim_j.
struct TileGeom {
    int a_row, b_row;      // TMA row coordinates of the A- and B-role tiles
    int sfa_rb, sfb_rb0;   // 128-row block of the A-role scales / first of the B role
    bool has_sfa;
    int nchunk_b;          // B-role scale chunks to load
    int sub_off;           // B-role 32-row group inside its scale chunk (BN < 128)
    int lim_i, lim_j;
    long long out_base;
};

template <int BN, int kChunksB>
__device__ __forceinline__ void tile_geom(const GemmParams &p, const GroupTable *g, const Work &w, TileGeom &t)
{
    // The MMA reads the B-role scales of this tile from TMEM column sub_off of
    // the chunk (32-row group).  It must be even: an odd column (a BN = 32 tile
    // starting 32 or 96 rows into its chunk) faulted with a misaligned address,
    // so plans use BN = 32 only when the whole B role is one tile (sub_off = 0).
    t.sub_off = ((w.tn * BN) % 128) / 32;
    if (g == nullptr) {
        const int nrb_b = (p.rows_b + 127) / 128;
        t.a_row = w.tm * kBM;
        t.b_row = w.tn * BN;
        t.sfa_rb = w.tm;
        t.has_sfa = w.tm < (p.rows_a + 127) / 128;
        t.sfb_rb0 = (w.tn * BN) / 128;
        t.nchunk_b = min(kChunksB, nrb_b - t.sfb_rb0);
        t.lim_i = p.rows_a;
        t.lim_j = p.rows_b;
        t.out_base = 0;
        return;
    }
    const int e = w.grp;
    const int s0 = g->row0[e], m = g->rows[e];
    const int wrow = e * p.group_n;             // first weight row of the group
    const int wblocks = (p.groups * p.group_n) / 128;
    t.out_base = static_cast<long long>(s0) * p.group_n;
    if (!p.tok_b) {                              // tokens: A role, 128-row tiles
        t.a_row = s0 + w.tm * kBM;
        t.sfa_rb = g->tok_rb[e] + w.tm;
        t.has_sfa = t.sfa_rb >= 0 && t.sfa_rb < p.tok_sf_cap;
        t.b_row = wrow + w.tn * BN;
        t.sfb_rb0 = (wrow + w.tn * BN) / 128;
        t.nchunk_b = max(0, min(kChunksB, wblocks - t.sfb_rb0));
        t.lim_i = m;
        t.lim_j = p.group_n;
    } else {                                     // tokens: B role, BN-row tiles
        t.a_row = wrow + w.tm * kBM;
        t.sfa_rb = wrow / 128 + w.tm;
        t.has_sfa = t.sfa_rb < wblocks;
        t.b_row = s0 + w.tn * BN;
        t.sfb_rb0 = g->tok_rb[e] + (w.tn * BN) / 128;
        t.nchunk_b = t.sfb_rb0 < 0 ? 0 : max(0, min(kChunksB, p.tok_sf_cap - t.sfb_rb0));
        t.lim_i = p.group_n;
        t.lim_j = m;
    }
}

// The stream-K CTA whose stage range contains stream-K stage x.
__device__ __forceinline__ int sk_cta_of(const GemmParams &p, long long x)
{
    return static_cast<int>(((x + 1) * p.sk_ctas + p.sk_stages - 1) / p.sk_stages - 1);
}

template <int kEpi = kEpiWarps>
__device__ __forceinline__ void epi_bar_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpi) : "memory");
}

__device__ __forceinline__ void record_timeout(const GemmParams &p, volatile int *abort)
{
    *abort = 1;
    atomicExch(p.status, -7 /* MXGEMM_ERR_DEVICE_TIMEOUT */);
}

// Debug build (compiled with MXGEMM_DEBUG): every plain global store and load
// of the GEMM kernels -- C or the split-K slabs, the stream-K partial slots
// and arrival counters -- is checked against its buffer's extent (and the
// vector stores against their alignment) before it is made.  An access that
// fails is skipped (a load then reads nothing, a fixup gives up) and
// MXGEMM_ERR_DEVICE_BOUNDS is recorded in the status word; nothing traps.
// Tensor-map (TMA) loads are bounded by their maps and need no check.  In the
// release build the checks compile to nothing.
#ifdef MXGEMM_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

__device__ __forceinline__ bool dbg_fail(const GemmParams &p)
{
    atomicCAS(p.status, 0, -9 /* MXGEMM_ERR_DEVICE_BOUNDS */);
    return false;
}

// [lo, hi) inside [0, cap)
__device__ __forceinline__ bool dbg_ok(const GemmParams &p, long long lo, long long hi, long long cap)
{
    if constexpr (!kDebugChecks)
        return true;
    if (lo >= 0 && lo <= hi && hi <= cap)
        return true;
    return dbg_fail(p);
}

// Store 32 consecutive B-role values of one A-role row: out[off .. off+32).
__device__ __forceinline__ void st_global_v8(void *dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t e,
                                             uint32_t f, uint32_t g, uint32_t h)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a), "r"(b), "r"(c), "r"(d),
                 "r"(e), "r"(f), "r"(g), "r"(h)
                 : "memory");
}

// kWide: 32-byte stores where rows are 32-byte aligned.  The epilogue's stores
// are one row per thread, so each store instruction touches 32 rows; 32-byte
// stores fill whole sectors with half the instructions.  The stream-K fixup
// paths (out-of-line functions) keep 16-byte stores: there the 32-byte form
// stored only its first word in a GPU test.
template <bool kWide = false>
__device__ __forceinline__ void store_row32_vec(const GemmParams &p, long long off, const uint32_t (&r)[32])
{
    if constexpr (kDebugChecks) {
        const unsigned long long esz = p.out_kind == OUT_BF16 ? 2u : 4u;
        const unsigned long long a = reinterpret_cast<unsigned long long>(p.out) + static_cast<unsigned long long>(off) * esz;
        const unsigned long long need = (kWide && p.vec_ok == 2) ? 32u : 16u;
        if (!dbg_ok(p, off, off + 32, p.dbg_out_elems))
            return;
        if (a % need != 0) {
            dbg_fail(p);
            return;
        }
    }
    if (kWide && p.vec_ok == 2) {
        if (p.out_kind == OUT_BF16) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                w[e] = *reinterpret_cast<uint32_t *>(&h);
            }
            uint32_t *dst = reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(p.out) + off);
            st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            st_global_v8(dst + 8, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
        } else {
            uint32_t *dst = reinterpret_cast<uint32_t *>(static_cast<float *>(p.out) + off);
#pragma unroll
            for (int v = 0; v < 4; ++v)
                st_global_v8(dst + 8 * v, r[8 * v], r[8 * v + 1], r[8 * v + 2], r[8 * v + 3], r[8 * v + 4],
                             r[8 * v + 5], r[8 * v + 6], r[8 * v + 7]);
        }
        return;
    }
    if (p.out_kind == OUT_BF16) {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + off);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[v * 8 + 2 * e]),
                                                         __uint_as_float(r[v * 8 + 2 * e + 1]));
                w[e] = *reinterpret_cast<uint32_t *>(&h);
            }
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<float *>(p.out) + off);
#pragma unroll
        for (int v = 0; v < 8; ++v)
            dst[v] = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
    }
}

// Element-wise store of n (<= 32) values at out[base + (j0+e)*stride_j].
__device__ __forceinline__ void store_row32_masked(const GemmParams &p, long long base, int j0, int n,
                                                   const uint32_t (&r)[32])
{
    if constexpr (kDebugChecks) {  // stride_j >= 1: the first and last element bound the run
        if (n > 0 && !dbg_ok(p, base + static_cast<long long>(j0) * p.stride_j,
                             base + static_cast<long long>(j0 + n - 1) * p.stride_j + 1, p.dbg_out_elems))
            return;
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        if (e < n) {
            const long long off = base + static_cast<long long>(j0 + e) * p.stride_j;
            if (p.out_kind == OUT_BF16)
                static_cast<__nv_bfloat16 *>(p.out)[off] = __float2bfloat16_rn(__uint_as_float(r[e]));
            else
                static_cast<float *>(p.out)[off] = __uint_as_float(r[e]);
        }
    }
}

// The fixup of a tile cut between CTAs that this CTA finishes (its segment
// arrived last), handed from the epilogue to the fixup warps through one
// shared-memory slot guarded by a full / empty mbarrier pair (the empty one
// counts one arrival per fixup warp).  tile < 0: stop.
struct SkFix {
    int tile, tn, c_first, c_last, row0;
};

// Post a job (one thread).  Bounded: false if the slot did not free in time.
__device__ __forceinline__ bool sk_post(SkFix &slot, const SkFix &job, uint32_t bar_full, uint32_t bar_empty,
                                        uint32_t &posted, const volatile int *abort, uint64_t lim)
{
    if (!mbar_wait(bar_empty, (posted & 1u) ^ 1u, abort, lim))
        return false;
    slot = job;
    mbar_arrive(bar_full);  // release: the job's fields are visible to the waiting warps
    ++posted;
    return true;
}

// Chunks c0 and c0 + 1 of a tile cut in exactly two segments, for this
// thread's row: all 32 loads issued before any add (the fixup warps hold no
// accumulator, so the registers go to loads in flight).  Same sums as
// sk_fixup_chunk: (0 + first) + second.
template <int BN, int kCols, int kChunks>
__device__ __noinline__ void sk_fixup_two(const GemmParams &p, int tile, int tn, int c_first, int halves, int half,
                                          int row0, int h, int row_local, int c0)
{
    constexpr size_t kSlot = static_cast<size_t>(kBM) * BN;
    const int i = row0 + row_local;
    if (i >= p.rows_a)
        return;
    const float4 *src[2];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const int cc = c_first + g;
        const long long beg = p.sk_stages * cc / p.sk_ctas;
        const int slot = (beg / p.kstages == tile - p.dp_tiles) ? 0 : 1;
        const long long so = static_cast<long long>((2 * cc + slot) * halves + half) * kSlot;
        if (!dbg_ok(p, so, so + static_cast<long long>(kSlot), p.dbg_skp_elems))
            return;
        src[g] = reinterpret_cast<const float4 *>(p.sk_partials + so) + row_local;
    }
    float4 x[2][2][8];  // [segment][chunk][4-column group]
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int v = 0; v < 8; ++v)
                x[g][k][v] = __ldcg(src[g] + ((h * kChunks + c0 + k) * 8 + v) * kBM);
    const long long base_off = static_cast<long long>(i) * p.stride_i;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int j0 = tn * BN + h * kCols + (c0 + k) * 32;
        if (j0 >= p.rows_b)
            break;
        uint32_t bits[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            bits[4 * v] = __float_as_uint((0.0f + x[0][k][v].x) + x[1][k][v].x);
            bits[4 * v + 1] = __float_as_uint((0.0f + x[0][k][v].y) + x[1][k][v].y);
            bits[4 * v + 2] = __float_as_uint((0.0f + x[0][k][v].z) + x[1][k][v].z);
            bits[4 * v + 3] = __float_as_uint((0.0f + x[0][k][v].w) + x[1][k][v].w);
        }
        if (p.vec_ok && j0 + 32 <= p.rows_b)
            store_row32_vec(p, base_off + j0, bits);
        else
            store_row32_masked(p, base_off, j0, min(32, p.rows_b - j0), bits);
    }
}

// One 32-column chunk of a cut tile, for this thread's row: the segments'
// partials added in k order (deterministic), then stored to C.  Cold code,
// kept out of line so that its registers do not count against the hot loops.
template <int BN, int kCols, int kChunks>
__device__ __noinline__ void sk_fixup_chunk(const GemmParams &p, int tile, int tn, int c_first, int c_last,
                                            int halves, int half, int row0, int h, int row_local, int c)
{
    constexpr size_t kSlot = static_cast<size_t>(kBM) * BN;
    const int i = row0 + row_local;
    const int j0 = tn * BN + h * kCols + c * 32;
    if (i >= p.rows_a || j0 >= p.rows_b)
        return;
    const long long base_off = static_cast<long long>(i) * p.stride_i;
    float sum[32];
#pragma unroll
    for (int e = 0; e < 32; ++e)
        sum[e] = 0.0f;
    // three segments' 32 columns are loaded at once (many loads in flight)
#pragma unroll 1
    for (int cc0 = c_first; cc0 <= c_last; cc0 += 3) {
        float4 x[3][8];
#pragma unroll
        for (int g = 0; g < 3; ++g) {
            const int cc = min(cc0 + g, c_last);
            const long long beg = p.sk_stages * cc / p.sk_ctas;
            const int slot = (beg / p.kstages == tile - p.dp_tiles) ? 0 : 1;
            const long long so = static_cast<long long>((2 * cc + slot) * halves + half) * kSlot;
            if (!dbg_ok(p, so, so + static_cast<long long>(kSlot), p.dbg_skp_elems))
                return;
            const float4 *src = reinterpret_cast<const float4 *>(p.sk_partials + so) +
                                (h * kChunks + c) * 8 * kBM + row_local;
            if (cc0 + g <= c_last) {  // uniform over the CTA: no load past the last segment
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    x[g][v] = __ldcg(src + v * kBM);
            } else {
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    x[g][v] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
#pragma unroll
        for (int g = 0; g < 3; ++g) {
            const bool keep = cc0 + g <= c_last;  // a select, not a product: partials may hold NaN
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                sum[4 * v] += keep ? x[g][v].x : 0.0f;
                sum[4 * v + 1] += keep ? x[g][v].y : 0.0f;
                sum[4 * v + 2] += keep ? x[g][v].z : 0.0f;
                sum[4 * v + 3] += keep ? x[g][v].w : 0.0f;
            }
        }
    }
    uint32_t bits[32];
#pragma unroll
    for (int e = 0; e < 32; ++e)
        bits[e] = __float_as_uint(sum[e]);
    if (p.vec_ok && j0 + 32 <= p.rows_b)
        store_row32_vec(p, base_off + j0, bits);
    else
        store_row32_masked(p, base_off, j0, min(32, p.rows_b - j0), bits);
}

// The fixup warps: take jobs until the stop job (or an abort / time-out).
// Warp fw adds column half fw of the CTA's 128 rows, four lane quarters (a
// tile of 32 columns has one half: warp 1 then only takes part in the hand-off).
template <int BN, int kCols, int kChunks>
__device__ __noinline__ void sk_fixup_warps(const GemmParams &p, const SkFix &slot, uint32_t bar_full,
                                               uint32_t bar_empty, int halves, int half, volatile int *abort,
                                               uint64_t lim)
{
    const int fw = static_cast<int>(threadIdx.x >> 5) - kFixWarp0;
    const bool has_cols = fw * kCols < BN;
    const int lane = static_cast<int>(threadIdx.x & 31);
    for (uint32_t j = 0;; ++j) {
        if (!warp_wait(bar_full, j & 1u, abort, lim)) {
            if (lane == 0) record_timeout(p, abort);
            return;
        }
        const SkFix job = slot;
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar_empty);  // this warp holds the job: the slot may be reused
        if (job.tile < 0)
            return;
        if (!has_cols)
            continue;
        __threadfence();  // the other segments' partials, published before their arrivals
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
            const int row_local = q * 32 + lane;
            if (job.c_last == job.c_first + 1 && kChunks % 2 == 0) {
#pragma unroll 1
                for (int c = 0; c < kChunks; c += 2)
                    sk_fixup_two<BN, kCols, kChunks>(p, job.tile, job.tn, job.c_first, halves, half, job.row0, fw,
                                                     row_local, c);
            } else {
#pragma unroll 1
                for (int c = 0; c < kChunks; ++c)
                    sk_fixup_chunk<BN, kCols, kChunks>(p, job.tile, job.tn, job.c_first, job.c_last, halves, half,
                                                       job.row0, fw, row_local, c);
            }
        }
    }
}

// Stream-K epilogue of one CTA's 128-row share of a tile cut between CTAs (or
// CTA pairs): publish this segment's FP32 partial sum; if it is the last
// segment of the tile to arrive, the tile's segments are added in k order --
// by the fixup warps (the job is posted through `fx`; this CTA's own partial is
// re-read from its slot), or, with kEpiFix, by these epilogue warps themselves:
// 256 threads with two segments' loads in flight at a time take a quarter of
// the L2 round trips of the two fixup warps.  kEpiFix serves the single-CTA
// weight-streaming decode tiles (at most 64 columns, partials of 16-32 KB) and
// every CTA-pair tile (the pair kernel has no fixup warps; the epilogue has
// handed its accumulator back before the fixup, so the next tile's MMAs go on
// meanwhile).  The own segment comes from registers for tiles of at most 64
// columns per column half, else from its slot (fewer live registers).  Either
// way each element is ((0 + s_first) + ...) + s_last.
//   unit:   the CTA's (or pair's) stream-K index; slots are numbered
//           ((2 * unit + w.slot) * halves + half) -- `halves` 128-row shares
//           per tile (1: single CTA, 2: CTA pair), `half` this CTA's share;
//   row0:   first A-role row of this CTA's share.
// Slot layout [h][chunk][4-column group][row]: each warp access is 32
// consecutive 16-byte vectors (the rows of one TMEM lane quarter).
template <int BN, int kCols, int kChunks, bool kEpiFix = false, int kEpi = kEpiWarps>
__device__ __forceinline__ void sk_epilogue(const GemmParams &p, const Work &w, const uint32_t (&r)[kChunks][32],
                                            int unit, int halves, int half, int row0, int h, int row_local,
                                            bool has_cols, int *sk_last, SkFix *fx, uint32_t fix_full,
                                            uint32_t fix_empty, uint32_t *posted, volatile int *abort, uint64_t lim)
{
    constexpr size_t kSlot = static_cast<size_t>(kBM) * BN;
    const long long mine_off = static_cast<long long>((2 * unit + w.slot) * halves + half) * kSlot;
    uint4 *const mine = reinterpret_cast<uint4 *>(p.sk_partials + mine_off);
    if (has_cols && dbg_ok(p, mine_off, mine_off + static_cast<long long>(kSlot), p.dbg_skp_elems)) {
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
                mine[((h * kChunks + c) * 8 + v) * kBM + row_local] =
                    make_uint4(r[c][4 * v], r[c][4 * v + 1], r[c][4 * v + 2], r[c][4 * v + 3]);
        }
    }
    // Arrival: the epilogue barrier orders every thread's partial before thread
    // 64's acquire-release add on the tile's counter, which publishes them at
    // GPU scope and, for the last arrival, makes the other segments' partials
    // (published the same way) visible to the loads after the next barrier.
    // One atomic round trip instead of a fence on each side of a relaxed add.
    epi_bar_sync<kEpi>();
    const long long t0 = static_cast<long long>(w.tile - p.dp_tiles) * p.kstages;
    const int c_first = sk_cta_of(p, t0);
    const int c_last = sk_cta_of(p, t0 + p.kstages - 1);
    const int cidx = (w.tile - p.dp_tiles) * halves + half;
    int *const counter = p.sk_counters + cidx;
    if (threadIdx.x == 64) {
        if (!dbg_ok(p, cidx, cidx + 1, p.dbg_counters)) {
            *sk_last = 0;
        } else {
            const int old = atom_add_acq_rel_gpu(counter, 1);
            const int last = old == c_last - c_first;
            if (last)
                *counter = 0;  // ready for the next launch
            *sk_last = last;
        }
    }
    epi_bar_sync<kEpi>();
    const bool last = *sk_last != 0;
    epi_bar_sync<kEpi>();  // sk_last is read before the next segment may rewrite it
    if (!last)
        return;
    if constexpr (kEpiFix) {
        // The own segment's values stay in registers for tiles of at most 64
        // columns per column half; wider ones re-read it from its slot (fewer
        // live registers), which makes it one more load of a batch.
        constexpr bool kOwnRegs = kChunks <= 2;
        constexpr int kBatch = kOwnRegs ? 2 : 3;
        auto own = [&](int c, float4 (&x)[8]) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
                x[v] = make_float4(__uint_as_float(r[c][4 * v]), __uint_as_float(r[c][4 * v + 1]),
                                   __uint_as_float(r[c][4 * v + 2]), __uint_as_float(r[c][4 * v + 3]));
        };
        const int i = row0 + row_local;
        if (!has_cols || i >= p.rows_a)
            return;
        const long long base_off = static_cast<long long>(i) * p.stride_i;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            const int j0 = w.tn * BN + h * kCols + c * 32;
            if (j0 >= p.rows_b)
                break;
            float sum[32];
#pragma unroll
            for (int e = 0; e < 32; ++e)
                sum[e] = 0.0f;
            auto add = [&](const float4 (&x)[8], bool keep) {  // a select, not a product: partials may hold NaN
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    sum[4 * v] += keep ? x[v].x : 0.0f;
                    sum[4 * v + 1] += keep ? x[v].y : 0.0f;
                    sum[4 * v + 2] += keep ? x[v].z : 0.0f;
                    sum[4 * v + 3] += keep ? x[v].w : 0.0f;
                }
            };
            // Batches of kBatch loaded segments (uniform over the CTA): all of a
            // batch's loads are issued before its adds, so a tile of up to
            // kBatch other segments costs one L2 round trip per chunk; the adds
            // then follow k order, the own segment (from registers) in its place.
            int cc = c_first;
            bool own_added = !kOwnRegs;
#pragma unroll 1
            while (cc <= c_last) {
                float4 x[kBatch][8];
                int seg[kBatch];
                int nxt = cc;
#pragma unroll
                for (int g = 0; g < kBatch; ++g) {
                    if (kOwnRegs && nxt == unit)
                        ++nxt;
                    seg[g] = nxt <= c_last ? nxt : -1;
                    const int sg = seg[g] < 0 ? c_first : seg[g];
                    const long long beg = p.sk_stages * sg / p.sk_ctas;
                    const int slot = (beg / p.kstages == w.tile - p.dp_tiles) ? 0 : 1;
                    const long long so = static_cast<long long>((2 * sg + slot) * halves + half) * kSlot;
                    const float4 *src = reinterpret_cast<const float4 *>(p.sk_partials + so) +
                                        (h * kChunks + c) * 8 * kBM + row_local;
                    if (seg[g] >= 0 && dbg_ok(p, so, so + static_cast<long long>(kSlot), p.dbg_skp_elems)) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            x[g][v] = __ldcg(src + v * kBM);
                    } else {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            x[g][v] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    }
                    ++nxt;
                }
                // segments [cc, stop) are added now
                int stop = seg[kBatch - 1] >= 0 ? seg[kBatch - 1] + 1 : c_last + 1;
                if (kOwnRegs && stop == unit)
                    ++stop;
#pragma unroll
                for (int g = 0; g < kBatch; ++g) {
                    if (kOwnRegs && !own_added && seg[g] >= 0 && unit < seg[g]) {
                        float4 y[8];
                        own(c, y);
                        add(y, true);
                        own_added = true;
                    }
                    add(x[g], seg[g] >= 0);
                }
                if (kOwnRegs && !own_added && unit < stop) {
                    float4 y[8];
                    own(c, y);
                    add(y, true);
                    own_added = true;
                }
                cc = stop;
            }
            uint32_t bits[32];
#pragma unroll
            for (int e = 0; e < 32; ++e)
                bits[e] = __float_as_uint(sum[e]);
            if (p.vec_ok && j0 + 32 <= p.rows_b)
                store_row32_vec(p, base_off + j0, bits);
            else
                store_row32_masked(p, base_off, j0, min(32, p.rows_b - j0), bits);
        }
    } else {
        if (threadIdx.x == 64) {
            __threadfence();
            const SkFix job{w.tile, w.tn, c_first, c_last, row0};
            if (!sk_post(*fx, job, fix_full, fix_empty, *posted, abort, lim))
                record_timeout(p, abort);
        }
    }
}

// GROUPED = true: the grouped (mixture-of-experts) form, tiles of all groups
// walked through the per-CTA group table (p.grouped must be 1); plain GEMMs
// use GROUPED = false, so none of its code or shared memory is in them.
// LEAN = true: the lean decode form (kLeanEpiWarps epilogue warps, which also
// add stream-K segments; two CTAs fit on an SM).
template <int KIND, int BN, bool GROUPED = false, bool SK = false, bool LEAN = false>
__global__ void __launch_bounds__(LEAN ? kLeanThreads : (SK ? kThreadsSk : kThreads), LEAN ? 2 : 1)
    mx_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b)
{
    using C = Cfg<KIND, BN, LEAN>;
    constexpr int S = C::kStages;
    constexpr int kEpi = LEAN ? kLeanEpiWarps : kEpiWarps;  // epilogue warps 2 .. 2 + kEpi - 1

    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base_holder;
    __shared__ int abort_flag;
    __shared__ GroupTable gtab;  // grouped GEMM only
    __shared__ uint64_t fix_bars[2];  // stream-K fixup hand-off: full, empty
    __shared__ SkFix sk_fix;
    constexpr bool kSk = SK;  // this instantiation runs stream-K plans (fixup warps 10, 11 unless lean)
    constexpr bool kFixW = SK && !LEAN;
    static_assert(!SK || !GROUPED, "stream-K: plain (not grouped) tiles only");
    static_assert(!LEAN || !GROUPED, "the lean form is for plain tiles");

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    // Layout: [A x S][B x S][scale group x 2][barriers]
    const uint32_t sA = base;
    const uint32_t sB = sA + S * C::kABytes;
    const uint32_t sSF = sB + S * C::kBBytes;
    const uint32_t sBar = sSF + 2 * C::kSfGrpBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(gbase + (sBar - base));
    (void)bars;
    (void)gbase;
    auto full_bar = [&](int s) { return sBar + 8u * s; };
    auto empty_bar = [&](int s) { return sBar + 8u * (S + s); };
    auto accf_bar = [&](int a) { return sBar + 8u * (2 * S + a); };
    auto acce_bar = [&](int a) { return sBar + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = sBar + 8u * (2 * S + 4);
    // scale groups: slot landed (sfull), slot copied to TMEM (sempty), the
    // group's TMEM regions read by all its MMAs (tfree)
    auto sfull_bar = [&](int g) { return sBar + 8u * (2 * S + 5 + g); };
    auto sempty_bar = [&](int g) { return sBar + 8u * (2 * S + 7 + g); };
    auto tfree_bar = [&](int g) { return sBar + 8u * (2 * S + 9 + g); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int *abort = &abort_flag;
    int never_abort = 0;  // drain waits ignore the abort flag (still time-bounded)
    const volatile int *no_abort = &never_abort;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), kEpi);
            mbar_init(sfull_bar(a), 1);
            mbar_init(sempty_bar(a), 1);
            mbar_init(tfree_bar(a), 1);
        }
        mbar_init(drain_bar, 1);
        mbar_init(smem_addr(&fix_bars[0]), 1);
        mbar_init(smem_addr(&fix_bars[1]), kFixWarps);
        fence_mbar_init();
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&tmem_base_holder), C::kTmemCols);
        tmem_relinquish();
    }
    // The kernel that follows in the stream may be scheduled as SMs free up
    // (it waits for this grid before it touches memory).
    griddep_launch_dependents();
    int npre = 0;         // k-stages of the first unit whose A-role tile was loaded before the grid wait
    bool sfa_pre = false;  // and its first scale group's A-role chunks
    if constexpr (!GROUPED) {
        if (warp == 0 && !p.test_stall) {
            WorkIter wi0;
            wi0.init(p, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x));
            Work w0;
            if (wi0.next(p, w0)) {
                TileGeom g0;
                tile_geom<BN, C::kChunksB>(p, nullptr, w0, g0);
                const int n0 = min(S, w0.ks1 - w0.ks0);
                if (LEAN && p.early_a) {
                    // The A-role operand is static (the caller's promise): arm the
                    // first ring slots for both tiles and load the A-role tiles now,
                    // while the preceding kernel drains; the B-role tiles follow the
                    // grid wait.  (The barriers were initialised by thread 0 of this warp.)
                    __syncwarp();
                    const uint64_t pol_a0 = p.stream_a ? l2_policy_evict_first() : l2_policy_evict_last();
                    if (elect_one()) {
                        if (C::kScaled && g0.has_sfa) {
                            // the first scale group: arm for both operands, copy the A-role chunks
                            const int kt0 = w0.ks0 * C::kKtPerStage;
                            const int nkt_g = min(kSfGroup * C::kKtPerStage, p.num_kt - kt0);
                            mbar_arrive_expect_tx(sfull_bar(0), nkt_g * kSfChunk * (1 + g0.nchunk_b));
                            bulk_load(sSF, p.sfa + (static_cast<size_t>(g0.sfa_rb) * p.num_kt + kt0) * kSfChunk,
                                      nkt_g * kSfChunk, sfull_bar(0));
                        }
                        for (int j = 0; j < n0; ++j) {
                            mbar_arrive_expect_tx(full_bar(j), C::kABytes + C::kBBytes);
                            tma_load_2d(sA + j * C::kABytes, &map_a, full_bar(j), (w0.ks0 + j) * kRowBytes, g0.a_row,
                                        pol_a0);
                        }
                    }
                    npre = n0;
                    sfa_pre = C::kScaled && g0.has_sfa;
                } else if (elect_one()) {
                    // Warm L2 with the first ring's worth of this CTA's operand boxes
                    // while the preceding kernel drains: a prefetch is only a hint and
                    // L2 is where that kernel's writes land, so no stale data can be
                    // read by it.
                    for (int j = 0; j < n0; ++j) {
                        tma_prefetch_2d(&map_a, (w0.ks0 + j) * kRowBytes, g0.a_row);
                        tma_prefetch_2d(&map_b, (w0.ks0 + j) * kRowBytes, g0.b_row);
                    }
                }
            }
            __syncwarp();
        }
    }
    // Everything above overlaps the end of the preceding kernel (programmatic
    // dependent launch); from here on global memory it wrote may be read.
    griddep_wait();
    if constexpr (GROUPED) {
        if (warp == 2)
            build_group_table<BN>(p, gtab, lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_holder;

    // Work: output tiles (x splits, or stream-K segments).
    const GroupTable *gt = nullptr;  // grouped kernels only (a constant null pointer otherwise)
    if constexpr (GROUPED)
        gt = &gtab;
    const int tok_tile = p.tok_b ? BN : kBM;
    const int first_unit = static_cast<int>(blockIdx.x);
    const int unit_step = static_cast<int>(gridDim.x);
    const uint64_t lim = p.timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // The whole warp runs the loop (so loop state stays warp-uniform); one
        // elected lane issues the barrier arm and the copies.
        if (!p.test_stall) {
            // Operands re-read by many tiles stay in L2 (evict-last); a streamed operand
            // (the weight of a decode GEMM) is loaded evict-first so it does not push
            // the re-used one out.
            const uint64_t pol_a = p.stream_a ? l2_policy_evict_first() : l2_policy_evict_last();
            const uint64_t pol_b = p.stream_b ? l2_policy_evict_first() : l2_policy_evict_last();
            int st = 0;
            uint32_t ph = 0;
            uint32_t armed = 0;      // bit s: slot s armed at least once
            uint32_t armed_ph = 0;   // bit s: parity of slot s's last arm
            int gi = 0;              // scale groups issued
            uint32_t sarmed = 0, sarmed_ph = 0;  // the same for the two scale group slots
            bool ok = true;
            int pre_left = npre;     // first-unit stages whose slot is armed and A-role tile loading
            armed = npre > 0 ? (1u << npre) - 1u : 0u;  // (phase 0)
            WorkIter wi;
            wi.init(p, first_unit, unit_step, gt, tok_tile);
            Work w;
            while (ok && wi.next(p, w)) {
                TileGeom g;
                tile_geom<BN, C::kChunksB>(p, gt, w, g);
                const bool has_sfa = g.has_sfa;
                const int ks0 = w.ks0;
                const int ks1 = w.ks1;
                // B-role scale chunks present for this tile (row blocks past the end are skipped)
                const int rb_b0 = g.sfb_rb0;
                const int nchunk_b = g.nchunk_b;
                for (int ks = ks0; ks < ks1; ++ks) {
                    const int kt0 = ks * C::kKtPerStage;
                    if (C::kScaled && (ks - ks0) % kSfGroup == 0) {
                        // the scales of k-stages [ks, ks + kSfGroup) into group slot gs:
                        // one bulk copy per operand (per 128-row block of the B role)
                        const int gs = gi & 1;
                        const uint32_t use = static_cast<uint32_t>(gi >> 1);
                        if (gi >= 2 && !warp_wait(sempty_bar(gs), (use & 1u) ^ 1u, abort, lim)) {
                            if (lane == 0) record_timeout(p, abort);
                            ok = false;
                            break;
                        }
                        const int nkt_g = min(kSfGroup * C::kKtPerStage, p.num_kt - kt0);
                        const uint32_t gbytes = nkt_g * kSfChunk * ((has_sfa ? 1 : 0) + nchunk_b);
                        const uint32_t dst = sSF + gs * C::kSfGrpBytes;
                        // the first group's A-role chunks may have gone out before the grid wait
                        const bool pre = gi == 0 && sfa_pre;
                        if (elect_one()) {
                            if (!pre)
                                mbar_arrive_expect_tx(sfull_bar(gs), gbytes);
                            if (has_sfa && !pre)
                                bulk_load(dst, p.sfa + (static_cast<size_t>(g.sfa_rb) * p.num_kt + kt0) * kSfChunk,
                                          nkt_g * kSfChunk, sfull_bar(gs));
                            for (int c = 0; c < nchunk_b; ++c)
                                bulk_load(dst + C::kSfaGrpBytes + c * kSfGroup * C::kKtPerStage * kSfChunk,
                                          p.sfb + (static_cast<size_t>(rb_b0 + c) * p.num_kt + kt0) * kSfChunk,
                                          nkt_g * kSfChunk, sfull_bar(gs));
                        }
                        __syncwarp();
                        sarmed |= 1u << gs;
                        sarmed_ph = (sarmed_ph & ~(1u << gs)) | ((use & 1u) << gs);
                        ++gi;
                    }
                    if (pre_left > 0) {
                        // slot st was armed and its A-role tile loaded before the grid wait
                        if (elect_one())
                            tma_load_2d(sB + st * C::kBBytes, &map_b, full_bar(st), ks * kRowBytes, g.b_row, pol_b);
                        --pre_left;
                    } else {
                        if (!warp_wait(empty_bar(st), ph ^ 1u, abort, lim)) {
                            if (lane == 0) record_timeout(p, abort);
                            ok = false;
                            break;
                        }
                        if (elect_one()) {
                            mbar_arrive_expect_tx(full_bar(st), C::kABytes + C::kBBytes);
                            tma_load_2d(sA + st * C::kABytes, &map_a, full_bar(st), ks * kRowBytes, g.a_row, pol_a);
                            tma_load_2d(sB + st * C::kBBytes, &map_b, full_bar(st), ks * kRowBytes, g.b_row, pol_b);
                        }
                    }
                    __syncwarp();
                    armed |= 1u << st;
                    armed_ph = (armed_ph & ~(1u << st)) | (ph << st);
                    if (++st == S) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Drain: let every armed stage and scale group finish landing before the CTA exits.
                for (int s2 = 0; s2 < S; ++s2)
                    if (armed & (1u << s2))
                        warp_wait(full_bar(s2), (armed_ph >> s2) & 1u, no_abort, lim);
                for (int g2 = 0; g2 < 2; ++g2)
                    if (sarmed & (1u << g2))
                        warp_wait(sfull_bar(g2), (sarmed_ph >> g2) & 1u, no_abort, lim);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        // Warp-uniform loop; every tcgen05 instruction is issued by the same
        // elected lane (tcgen05.commit tracks that lane's earlier operations).
        int st = 0;
        uint32_t ph = 0;
        int it = 0;
        int gi = 0;  // scale groups started
        bool ok = true;
        bool issued = false;
        // Scale group in, at the group's first k-stage k_ (n_ stages of this work
        // unit in the group): wait until the group slot has landed and the TMEM
        // regions it goes to are no longer read (the MMAs of the group two
        // before have completed), tcgen05.cp every stage's chunks into its own
        // TMEM region, and commit so the producer may refill the slot.
        auto group_in = [&](int k_, int n_) -> bool {
            const int gs = gi & 1;
            const uint32_t use = static_cast<uint32_t>(gi >> 1);
            if (!warp_wait(sfull_bar(gs), use & 1u, abort, lim))
                return false;
            if (gi >= 2 && !warp_wait(tfree_bar(gs), (use & 1u) ^ 1u, abort, lim))
                return false;
            tc_fence_after();
            const uint32_t src = sSF + gs * C::kSfGrpBytes;
            // one elected lane issues the group's copies (and, below, the MMAs
            // and commits) in one block: separate elect blocks per instruction
            // measured up to 10% slower on long k-loops
            if (elect_one()) {
#pragma unroll 1
                for (int j = 0; j < n_; ++j) {
                    const int nkt_ = min(C::kKtPerStage, p.num_kt - (k_ + j) * C::kKtPerStage);
                    const uint32_t sfa_col_ = tmem + C::kSfCol0 + (gs * kSfGroup + j) * C::kSfSlotCols;
                    const uint32_t sfb_col_ = sfa_col_ + C::kSfaCols;
#pragma unroll
                    for (int t = 0; t < C::kKtPerStage; ++t) {
                        if (t < nkt_) {
                            tc_cp_32x128b_warpx4(sfa_col_ + 4 * t,
                                                 sdesc_sf_chunk(src + (j * C::kKtPerStage + t) * kSfChunk));
#pragma unroll
                            for (int c = 0; c < C::kChunksB; ++c)
                                tc_cp_32x128b_warpx4(
                                    sfb_col_ + 4 * (t * C::kChunksB + c),
                                    sdesc_sf_chunk(src + C::kSfaGrpBytes +
                                                   ((c * kSfGroup + j) * C::kKtPerStage + t) * kSfChunk));
                        }
                    }
                }
                tc_commit(sempty_bar(gs));
            }
            __syncwarp();
            issued = true;
            ++gi;
            return true;
        };
        WorkIter wi;
        wi.init(p, first_unit, unit_step, gt, tok_tile);
        Work w;
        for (; ok && wi.next(p, w); ++it) {
            const int tn = w.tn;
            const int acc = it % C::kAccStages;
            const uint32_t acc_par = static_cast<uint32_t>((it / C::kAccStages) & 1);
            if (!warp_wait(acce_bar(acc), acc_par ^ 1u, abort, lim)) {
                if (lane == 0) record_timeout(p, abort);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + acc * BN;
            const uint32_t sub_off = static_cast<uint32_t>(((tn * BN) % 128) / 32);  // BN < 128 only
            const int ks0 = w.ks0;
            const int ks1 = w.ks1;
            for (int ks = ks0; ks < ks1; ++ks) {
                const int rel = ks - ks0;
                if (C::kScaled && rel % kSfGroup == 0 && !group_in(ks, min(kSfGroup, ks1 - ks))) {
                    if (lane == 0) record_timeout(p, abort);
                    ok = false;
                    break;
                }
                if (!warp_wait(full_bar(st), ph, abort, lim)) {
                    if (lane == 0) record_timeout(p, abort);
                    ok = false;
                    break;
                }
                tc_fence_after();
                issued = true;
                const int nkt = min(C::kKtPerStage, p.num_kt - ks * C::kKtPerStage);
                const int gcur = gi - 1;  // the group this stage belongs to
                const uint32_t sfa_col =
                    tmem + C::kSfCol0 + ((gcur & 1) * kSfGroup + rel % kSfGroup) * C::kSfSlotCols;
                const uint32_t sfb_col = sfa_col + C::kSfaCols;
                const bool group_end = C::kScaled && (rel % kSfGroup == kSfGroup - 1 || ks == ks1 - 1);
                const uint64_t adesc = sdesc_kmajor_sw128(sA + st * C::kABytes);
                const uint64_t bdesc = sdesc_kmajor_sw128(sB + st * C::kBBytes);
                const uint32_t acc0 = (ks > ks0) ? 1u : 0u;
                if (elect_one()) {
#pragma unroll
                    for (int s = 0; s < C::kKtPerStage * C::kSubPerKt; ++s) {
                        constexpr int kSub = C::kSubPerKt;
                        const int t = s / kSub;
                        if (t < nkt) {
                            const uint32_t sf_id =
                                C::kFp4 ? static_cast<uint32_t>((s % 2) * 2) : static_cast<uint32_t>(s % 4);
                            const uint32_t idesc = idesc_with_sf_ids(C::kIdesc, sf_id, sf_id);
                            const uint32_t sfa_t = sfa_col + 4 * t;
                            const uint32_t sfb_t = sfb_col + 4 * t * C::kChunksB + sub_off;
                            // advance 32 bytes along K per MMA (32 FP8 or 64 FP4 elements)
                            const uint64_t koff = static_cast<uint64_t>((s * 32) >> 4);
                            const uint32_t accum = (s > 0) ? 1u : acc0;
                            if constexpr (KIND == K_BF16)
                                mma_bf16(d_tmem, adesc + koff, bdesc + koff, C::kIdesc, accum);
                            else if constexpr (C::kFp4)
                                mma_mxf4(d_tmem, adesc + koff, bdesc + koff, idesc, sfa_t, sfb_t, accum);
                            else
                                mma_mxf8f6f4(d_tmem, adesc + koff, bdesc + koff, idesc, sfa_t, sfb_t, accum);
                        }
                    }
                    tc_commit(empty_bar(st));
                    if (group_end)
                        tc_commit(tfree_bar(gcur & 1));  // this group's TMEM scale regions are free again
                }
                __syncwarp();
                if (++st == S) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            if (elect_one())
                tc_commit(accf_bar(acc));
            __syncwarp();
        }
        if (!ok && issued) {
            // Drain the tensor pipe before TMEM is released.
            if (elect_one())
                tc_commit(drain_bar);
            __syncwarp();
            warp_wait(drain_bar, 0, no_abort, lim);
        }
    } else if (warp >= 2 && warp < 2 + kEpi) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                     // TMEM lane quarter this warp may access
        const int h = LEAN ? 0 : (warp - 2) >> 2;   // column half (the lean form: all columns)
        constexpr int kCols = LEAN ? BN : (BN / 2 >= 32 ? BN / 2 : 32);
        constexpr int kChunks = kCols / 32;
        const bool has_cols = h * kCols < BN;
        __shared__ int sk_last;
        const int row_local = q * 32 + lane;
        uint32_t sk_posted = 0;  // jobs posted to the fixup warps (thread 64)
        int it = 0;
        WorkIter wi;
        wi.init(p, first_unit, unit_step, gt, tok_tile);
        Work w;
        for (; wi.next(p, w); ++it) {
            const int tm = w.tm;
            const int tn = w.tn;
            const int acc = it % C::kAccStages;
            const uint32_t acc_par = static_cast<uint32_t>((it / C::kAccStages) & 1);
            bool ok = true;
            if (lane == 0) ok = mbar_wait(accf_bar(acc), acc_par, abort, lim);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) record_timeout(p, abort);
                break;
            }
            tc_fence_after();
            uint32_t r[kChunks][32];
            if (has_cols) {
                const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + h * kCols;
                if constexpr (kChunks % 2 == 0) {
#pragma unroll
                    for (int c = 0; c < kChunks; c += 2)
                        tmem_ld_32x32b_x64(tbase + c * 32, r[c], r[c + 1]);
                } else {
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        tmem_ld_32x32b_x32(tbase + c * 32, r[c]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
                    reg_fence(r[c]);
            }
            // The accumulator stage is in registers now: hand it back to the MMA warp.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(acc));

            if constexpr (kSk) {
                if (w.kind == 1) {
                    // stream-K segment: publish, and queue the tile's fixup if this CTA is last
                    sk_epilogue<BN, kCols, kChunks, (LEAN || BN <= 64), kEpi>(
                        p, w, r, first_unit, 1, 0, tm * kBM, h, row_local, has_cols, &sk_last, &sk_fix,
                        smem_addr(&fix_bars[0]), smem_addr(&fix_bars[1]), &sk_posted, abort, lim);
                    continue;
                }
            }

            // Output limits and origin (computed after the release: fewer live registers)
            TileGeom g;
            tile_geom<BN, C::kChunksB>(p, gt, w, g);
            const int i = tm * kBM + row_local;  // A-role row owned by this thread
            if (has_cols && i < g.lim_i) {
                const long long base_off = g.out_base +
                                           (w.kind == 2 ? static_cast<long long>(w.slot) * p.split_stride : 0ll) +
                                           static_cast<long long>(i) * p.stride_i;
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    const int j0 = tn * BN + h * kCols + c * 32;
                    if (j0 >= g.lim_j) break;
                    if (p.vec_ok && j0 + 32 <= g.lim_j)
                        store_row32_vec<true>(p, base_off + j0, r[c]);
                    else
                        store_row32_masked(p, base_off, j0, min(32, g.lim_j - j0), r[c]);
                }
            }
        }
        if constexpr (kFixW) {
            if (p.sk_ctas > 0 && threadIdx.x == 64) {
                const SkFix stop{-1, 0, 0, 0, 0};
                if (!sk_post(sk_fix, stop, smem_addr(&fix_bars[0]), smem_addr(&fix_bars[1]), sk_posted, abort, lim))
                    record_timeout(p, abort);
            }
        }
    } else if (warp >= kFixWarp0) {
        // ------------------------------------------------- stream-K fixup
        if constexpr (kFixW) {
            if (p.sk_ctas > 0) {
                constexpr int kCols = BN / 2 >= 32 ? BN / 2 : 32;  // as in the epilogue
                sk_fixup_warps<BN, kCols, kCols / 32>(p, sk_fix, smem_addr(&fix_bars[0]), smem_addr(&fix_bars[1]),
                                                      1, 0, abort, lim);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace mxg
