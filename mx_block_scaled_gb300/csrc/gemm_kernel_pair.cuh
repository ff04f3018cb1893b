// gemm_kernel_pair.cuh -- the MX block-scaled GEMM on CTA pairs (tcgen05
// cta_group::2): a cluster of two CTAs on two SMs computes one 256 x BN output
// tile with M = 256 MMAs issued by the even CTA.
//
// Same operation and pipeline as mx_gemm_kernel (gemm_kernel.cuh); what changes:
//   * CTA r of the pair loads A-role rows [256*tm + 128*r, +128) and the r-th
//     half of the B-role tile (BN/2 rows) into its own shared memory; an MMA of
//     the pair reads A from each CTA's own half and B from both halves, so each
//     SM fetches 1/3 fewer operand bytes per FLOP than a 128 x BN tile, and one
//     MMA instruction covers twice the work.
//   * both CTAs hold the full B-role scales (they are needed for every output
//     column) and the scales of their own 128 A-role rows; the even CTA's
//     tcgen05.cp (cta_group::2) moves each CTA's scale chunks into its own TMEM.
//   * the loads of both CTAs (operand tiles and scale chunks, all TMA tensor
//     copies) complete on the even CTA's `full` barrier, which the even CTA arms
//     with the pair's total bytes; so a stage's MMAs are issued as soon as both
//     halves are resident.  The even CTA's commits arrive on `empty` / `acc_full`
//     in both CTAs (multicast); both CTAs' epilogue warps arrive on the even
//     CTA's `acc_empty`.
//   * every CTA holds its 128 rows x BN FP32 accumulator in its own TMEM, and its
//     epilogue stores those rows.
//   * with stream-K, a pair's segment of a cut tile is published per CTA (each
//     its 128 rows, its own arrival counter), and the last pair to arrive adds
//     the segments in k order, each CTA for its own rows, in its epilogue warps
//     (there are no fixup warps: 4096^3 MXFP8 49.2 -> 48.2 us per call).
// All waits are bounded as in the single-CTA kernel; the CTAs meet at a cluster
// barrier before TMEM is released.
#pragma once

#include "gemm_kernel.cuh"

namespace mxg {

// GROUPED = true: the grouped (mixture-of-experts) form: token tiles of 256 rows
// inside each group, the group table in static shared memory, no in-kernel
// scale layout (the tokens' scales are laid out per group before the GEMM).
template <int KIND, int BN, bool GROUPED = false>
struct CfgPair {
    static constexpr bool kFp4 = KIND == K_MXFP4;
    static constexpr bool kScaled = KIND != K_BF16;
    static constexpr int kKtPerStage = kFp4 ? 2 : 1;
    static constexpr int kSubPerKt = kFp4 ? 2 : 4;
    // B-role scale chunks per K-tile: all BN rows.  A 192-wide tile starts 0 or 64
    // rows into a 128-row chunk, so it spans two chunks and its MMAs read the B
    // scales from TMEM column 0 or 2 of them (an even column, as required).
    static constexpr int kChunksB = (BN + 127) / 128;
    static constexpr int kABytes = kBM * kRowBytes;           // own 128 A-role rows
    static constexpr int kBBytes = (BN / 2) * kRowBytes;      // own half of the B-role tile
    static constexpr int kStageBytes = kABytes + kBBytes;     // operands of one k-stage
    // Operand ring slots hold two k-stages each, loaded by one 3-D box per
    // operand: a CTA's TMA engine streams 32 KB boxes of two 128-byte K-slices
    // at ~150 GB/s, one-slice 16 KB boxes at ~100 GB/s (measured, all SMs), and
    // the MMAs of a 256 x 256 pair tile need ~125 GB/s per SM.
    static constexpr int kSlotBytes = 2 * kStageBytes;
    // scale group slot (see kSfGroup): SFA chunks of this CTA's 128 rows
    // [stage][K-tile], then the SFB chunks of all BN rows [128-row block][stage][K-tile]
    static constexpr int kSfaGrpBytes = kScaled ? kSfGroup * kKtPerStage * kSfChunk : 0;
    static constexpr int kSfbGrpBytes = kScaled ? kChunksB * kSfGroup * kKtPerStage * kSfChunk : 0;
    static constexpr int kSfGrpBytes = kSfaGrpBytes + kSfbGrpBytes;
    // Scale group slots (shared memory and TMEM regions): MXFP8 keeps three, so
    // a group's copies and layout may start two groups ahead of its MMAs; MXFP4's
    // scale columns leave TMEM room for two.
    static constexpr int kGrp = (kScaled && !kFp4) ? 3 : 2;
    // Row-major A-role scales laid out in the kernel (MXFP8): per group, a
    // staging buffer for both CTAs' 256 rows x 4 bytes per K-tile, and the even
    // CTA's chunks as built by the odd CTA.  (MXFP4 plans take pre-laid scales:
    // their ring leaves no room for the buffers.)
    static constexpr bool kFuseSa = kScaled && !kFp4 && !GROUPED;
    static constexpr int kSaRawBytes = kFuseSa ? 2 * kBM * 4 * kSfGroup * kKtPerStage : 0;
    static constexpr int kSaLeadBytes = kFuseSa ? kSfaGrpBytes : 0;
    static constexpr int kSaBytes = 2 * kSaRawBytes + kGrp * kSaLeadBytes;
    static constexpr int kStaticBytes = GROUPED ? static_cast<int>(sizeof(GroupTable)) : 0;
    static constexpr int kSlotsRaw =
        (kSmemBudget - kStaticBytes - 1024 - 512 - kGrp * kSfGrpBytes - kSaBytes) / kSlotBytes;
    static constexpr int kSlots = kSlotsRaw > 4 ? 4 : kSlotsRaw;
    static constexpr int kStages = 2 * kSlots;                // k-stages resident in the ring
    static constexpr int kSfaCols = kScaled ? 4 * kKtPerStage : 0;
    static constexpr int kSfbCols = kScaled ? 4 * kKtPerStage * kChunksB : 0;
    static constexpr int kSfSlotCols = kSfaCols + kSfbCols;
    static constexpr int kSfRegions = kScaled ? kGrp * kSfGroup : 0;
    static constexpr int kAccStages = (2 * BN + kSfRegions * kSfSlotCols <= 512) ? 2 : 1;
    static constexpr int kSfCol0 = kAccStages * BN;
    static constexpr int kColsUsed = kSfCol0 + kSfRegions * kSfSlotCols;
    static constexpr int kTmemCols = kColsUsed <= 32 ? 32 : kColsUsed <= 64 ? 64 : kColsUsed <= 128 ? 128
                                   : kColsUsed <= 256 ? 256 : 512;
    static constexpr int kSmemBytes = 1024 + kSlots * kSlotBytes + kGrp * kSfGrpBytes + kSaBytes + 512;
    static constexpr uint32_t kIdesc =
        kScaled ? idesc_block_scaled(kFp4 ? 1u : 0u, 2 * kBM, BN) : idesc_bf16(2 * kBM, BN);
    static_assert(BN == 128 || BN == 192 || BN == 256, "pair tiles are 256 x 128, 256 x 192 or 256 x 256");
    static_assert(kSlots >= 2, "shared memory too small for two slots");
    static_assert(kSfGroup % 2 == 0, "scale groups start on a slot boundary");
    static_assert(kColsUsed <= 512, "TMEM overflow");
    static_assert(!kFuseSa || kSfGroup * kKtPerStage == 4, "the fused layout moves one 16-byte row word per chunk");
};

// Where one CTA of a pair works on tile w: the TMA rows of its A-role rows and
// of its half of the B-role tile, its A-role scale block (and the odd CTA's, for
// the even CTA's byte count), the tile's first B-role scale block, and the
// output rows and limits of its 128 rows.  Grouped tiles are group-local: the
// tokens' rows and scale blocks start at the group's, the weights' at e * N.
struct PairGeom {
    int a_row, b_row;
    int sfa_rb;
    bool has_sfa, peer_has_sfa;
    int rb_b0;
    int row0;              // first output row (within the group) of this CTA's 128 rows
    int lim_i, lim_j;
    long long out_base;
};

template <int BN>
__device__ __forceinline__ void pair_geom(const GemmParams &p, const GroupTable *g, const Work &w, int rank,
                                          PairGeom &t)
{
    int base_rb = 0, a0 = 0, b0 = 0, nrb = (p.rows_a + 127) / 128;
    t.lim_i = p.rows_a;
    t.lim_j = p.rows_b;
    t.out_base = 0;
    if (g != nullptr) {
        const int e = w.grp;
        base_rb = g->tok_rb[e];
        a0 = g->row0[e];
        b0 = e * p.group_n;
        nrb = p.tok_sf_cap;
        t.lim_i = g->rows[e];
        t.lim_j = p.group_n;
        t.out_base = static_cast<long long>(a0) * p.group_n;
    }
    t.row0 = (2 * w.tm + rank) * kBM;
    t.a_row = a0 + t.row0;
    t.sfa_rb = base_rb + 2 * w.tm + rank;
    t.has_sfa = t.sfa_rb >= 0 && t.sfa_rb < nrb;
    const int peer_rb = base_rb + 2 * w.tm + 1;
    t.peer_has_sfa = peer_rb >= 0 && peer_rb < nrb;
    t.b_row = b0 + w.tn * BN + rank * (BN / 2);
    t.rb_b0 = (b0 + w.tn * BN) / 128;
}

// SK = true: the instantiation for stream-K plans (the epilogue publishes and
// adds the cut tiles' segments); plans without cut tiles run the other form.
// GROUPED = true: the grouped form (p.grouped = 1, non-swapped, BN = 256).
template <int KIND, int BN, bool SK = false, bool GROUPED = false>
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_pair_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_sfa,
                        const __grid_constant__ CUtensorMap map_sfb, const __grid_constant__ CUtensorMap map_sarm)
{
    using C = CfgPair<KIND, BN, GROUPED>;
    constexpr int S = C::kSlots;  // ring slots, two k-stages each
    static_assert(!(SK && GROUPED), "the grouped form has no stream-K");

    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base_holder;
    __shared__ int abort_flag;
    __shared__ GroupTable gtab;  // grouped form only

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    // Layout: [A: slot x 2 stages][B: slot x 2 stages][scale group x kGrp]
    //         [row-major A-role scale staging x 2][even CTA's A-role chunks x kGrp][barriers]
    const uint32_t sA = base;
    const uint32_t sB = sA + S * 2 * C::kABytes;
    const uint32_t sSF = sB + S * 2 * C::kBBytes;
    const uint32_t sRaw = sSF + C::kGrp * C::kSfGrpBytes;
    const uint32_t sLead = sRaw + 2 * C::kSaRawBytes;
    const uint32_t sBar = sLead + C::kGrp * C::kSaLeadBytes;
    auto full_bar = [&](int s) { return sBar + 8u * s; };
    auto empty_bar = [&](int s) { return sBar + 8u * (S + s); };
    auto accf_bar = [&](int a) { return sBar + 8u * (3 * S + a); };
    auto acce_bar = [&](int a) { return sBar + 8u * (3 * S + 2 + a); };  // used in the even CTA
    const uint32_t drain_bar = sBar + 8u * (3 * S + 4);
    // scale groups (sfull and tfree used in the even CTA, sempty in both)
    constexpr int G = C::kGrp;
    auto sfull_bar = [&](int g) { return sBar + 8u * (3 * S + 5 + g); };
    auto sempty_bar = [&](int g) { return sBar + 8u * (3 * S + 5 + G + g); };
    auto tfree_bar = [&](int g) { return sBar + 8u * (3 * S + 5 + 2 * G + g); };
    auto araw_bar = [&](int b) { return sBar + 8u * (3 * S + 5 + 3 * G + b); };  // staging landed (odd CTA)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    volatile int *abort = &abort_flag;
    int never_abort = 0;
    const volatile int *no_abort = &never_abort;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), 2 * kEpiWarps);
            mbar_init(araw_bar(a), 1);
        }
        for (int g = 0; g < G; ++g) {
            mbar_init(sfull_bar(g), 1);
            mbar_init(sempty_bar(g), 1);
            mbar_init(tfree_bar(g), 1);
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
        tma_prefetch_map(&map_sfa);
        tma_prefetch_map(&map_sfb);
        if (p.sa_fused)
            tma_prefetch_map(&map_sarm);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&tmem_base_holder), C::kTmemCols);
        tmem_relinquish_pair();
    }
    // The kernel that follows in the stream may be scheduled as SMs free up
    // (it waits for this grid before it touches memory).
    griddep_launch_dependents();
    if (!GROUPED && warp == 0 && !p.test_stall) {
        // Warm L2 with the first ring's worth of this CTA's operand boxes while
        // the preceding kernel drains: a prefetch is only a hint and L2 is where
        // that kernel's writes land, so no stale data can be read by it.
        WorkIter wi0;
        wi0.init(p, static_cast<int>(cluster_id_x()), static_cast<int>(cluster_count_x()));
        Work w0;
        if (wi0.next(p, w0) && elect_one()) {
            const int kb0 = w0.ks0 & ~1;
            for (int kb = kb0; kb < w0.ks1 && kb < kb0 + 2 * S; kb += 2) {
                tma_prefetch_3d(&map_a, 0, (2 * w0.tm + static_cast<int>(rank)) * kBM, kb);
                tma_prefetch_3d(&map_b, 0, w0.tn * BN + static_cast<int>(rank) * (BN / 2), kb);
            }
            if constexpr (C::kScaled) {
                // and the first scale group (the first MMAs wait for it)
                const int gkt0 = (kb0 - kb0 % kSfGroup) * C::kKtPerStage;
                const int rb_a0 = 2 * w0.tm + static_cast<int>(rank);
                if (rank == 0)
                    tma_prefetch_3d(&map_sfb, 0, 2 * gkt0, (w0.tn * BN) / 128);
                if (p.sa_fused) {
                    if (rank == 1)
                        tma_prefetch_2d(&map_sarm, 4 * gkt0, 2 * w0.tm * kBM);
                } else if (rb_a0 < (p.rows_a + 127) / 128) {
                    tma_prefetch_3d(&map_sfa, 0, 2 * gkt0, rb_a0);
                }
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // barriers of both CTAs initialised before any cross-CTA arrive
    tc_fence_after();
    // Everything above (the cluster barrier included) overlaps the end of the
    // preceding kernel (programmatic dependent launch); from here on global
    // memory it wrote may be read.
    griddep_wait();
    // Grouped: one warp reads the offsets (written by the preceding kernel) into
    // this CTA's group table; both CTAs of a pair build the same table.
    if constexpr (GROUPED) {
        if (warp == 2)
            group_scan(p.group_offsets, p.groups, p.rows_total, 2 * kBM, (p.group_n + BN - 1) / BN, lane,
                       gtab.tile_start, gtab.tok_rb, gtab.row0, gtab.rows);
        __syncthreads();
    }
    const uint32_t tmem = tmem_base_holder;
    const GroupTable *gt = nullptr;  // grouped form only (a constant null pointer otherwise)
    if constexpr (GROUPED)
        gt = &gtab;

    // Work of this pair (tiles_m counts 256-row pair tiles): stream-K segments,
    // then whole tiles (or split-K slabs) round-robin over the clusters.
    const int first_unit = static_cast<int>(cluster_id_x());
    const int unit_step = static_cast<int>(cluster_count_x());
    const uint64_t lim = p.timeout_ns;

    // Slots and scale groups are aligned to absolute k-stage indices: slot =
    // k-stages (2j, 2j+1), scale group = k-stages [4g, 4g+4).  A work unit that
    // starts or ends inside one (stream-K segments, split-K slabs) loads the
    // whole of it and uses its own stages only.  The alignment keeps the
    // row-major scale box of a group on a 16-byte boundary.
    auto group_start = [&](int kb, int kb0) { return C::kScaled && (kb % kSfGroup == 0 || kb == kb0); };
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // Both CTAs load their own halves; every copy completes on the even CTA's
        // `full` barrier, which only the even CTA arms (with both CTAs' bytes).
        if (!p.test_stall) {
            // Operands re-read by many tiles stay in L2 (evict-last); a streamed
            // one (read by at most two tiles) is loaded evict-first.
            const uint64_t pol_a = p.stream_a ? l2_policy_evict_first() : l2_policy_evict_last();
            const uint64_t pol_b = p.stream_b ? l2_policy_evict_first() : l2_policy_evict_last();
            int st = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_ph = 0;
            int gi = 0;  // scale groups issued
            uint32_t sarmed = 0, sarmed_ph = 0;
            bool ok = true;
            WorkIter wi;
            wi.init(p, first_unit, unit_step, gt, 2 * kBM);
            Work w;
            while (ok && wi.next(p, w)) {
                const int ks0 = w.ks0, ks1 = w.ks1;
                PairGeom pg;
                pair_geom<BN>(p, gt, w, static_cast<int>(rank), pg);
                const int rb_a = pg.sfa_rb;  // own 128-row block of the A-role scales
                const bool has_sfa = pg.has_sfa;
                const bool peer_has_sfa = pg.peer_has_sfa;
                const int rb_b0 = pg.rb_b0;
                // bytes of both CTAs' copies, as counted by TMA (whole boxes; a box
                // partly or wholly past the tensor is zero-filled and counted in full)
                const uint32_t slot_bytes = 2 * C::kSlotBytes;
                // (fused: the even CTA's A-role chunks, sent by the odd CTA)
                const uint32_t group_bytes =
                    2 * C::kSfbGrpBytes +
                    (p.sa_fused ? 1u : ((has_sfa ? 1u : 0u) + (peer_has_sfa ? 1u : 0u))) * C::kSfaGrpBytes;
                const int kb0 = ks0 & ~1;
                for (int kb = kb0; kb < ks1; kb += 2) {
                    if (group_start(kb, kb0)) {
                        // the scales of the group holding k-stage kb: every B-role row, one
                        // 3-D box (chunks of 2 rows x 256 B), and this CTA's A-role rows, a
                        // 3-D box of tile-layout chunks (unless the odd CTA lays them out)
                        const int gkt0 = (kb - kb % kSfGroup) * C::kKtPerStage;
                        const int gs = gi % G;
                        const uint32_t use = static_cast<uint32_t>(gi / G);
                        if (gi >= G && !warp_wait_cluster(sempty_bar(gs), (use & 1u) ^ 1u, abort, lim)) {
                            if (lane == 0) record_timeout(p, abort);
                            ok = false;
                            break;
                        }
                        const uint32_t dst = sSF + gs * C::kSfGrpBytes;
                        if (elect_one()) {
                            const uint32_t bar = map_to_cta(sfull_bar(gs), 0);
                            if (leader)
                                mbar_arrive_expect_tx(sfull_bar(gs), group_bytes);
                            if (!p.sa_fused && has_sfa)
                                tma_load_3d_pair(dst, &map_sfa, bar, 0, 2 * gkt0, rb_a);
                            tma_load_3d_pair(dst + C::kSfaGrpBytes, &map_sfb, bar, 0, 2 * gkt0, rb_b0);
                        }
                        __syncwarp();
                        sarmed |= 1u << gs;
                        sarmed_ph = (sarmed_ph & ~(1u << gs)) | ((use & 1u) << gs);
                        ++gi;
                    }
                    if (!warp_wait_cluster(empty_bar(st), ph ^ 1u, abort, lim)) {
                        if (lane == 0) record_timeout(p, abort);
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        // A: this CTA's 128 rows, B: its BN/2 rows, k-stages kb and kb + 1
                        // (3-D maps: 128-byte K-slice x rows x slice index)
                        const uint32_t bar = map_to_cta(full_bar(st), 0);
                        if (leader)
                            mbar_arrive_expect_tx(full_bar(st), slot_bytes);
                        tma_load_3d_pair_hint(sA + st * 2 * C::kABytes, &map_a, bar, 0, pg.a_row, kb, pol_a);
                        tma_load_3d_pair_hint(sB + st * 2 * C::kBBytes, &map_b, bar, 0, pg.b_row, kb, pol_b);
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
                // let every armed copy finish landing before the CTA exits
                for (int s2 = 0; s2 < S; ++s2)
                    if (leader && (armed & (1u << s2)))
                        warp_wait(full_bar(s2), (armed_ph >> s2) & 1u, no_abort, lim);
                for (int g2 = 0; g2 < G; ++g2)
                    if (leader && (sarmed & (1u << g2)))
                        warp_wait(sfull_bar(g2), (sarmed_ph >> g2) & 1u, no_abort, lim);
            }
        }
    } else if (warp == 1 && !leader) {
        // ------------ odd CTA: lays out the pair's row-major A-role scales
        // Per scale group one 2-D box brings both CTAs' 256 rows x 16 bytes into
        // a staging buffer (loaded one group ahead).  The warp writes this CTA's
        // rows as tensor-core chunks into its group slot and the even CTA's rows
        // into a side buffer, orders those writes before its async-proxy
        // operations, and sends the side buffer to the even CTA's group slot by
        // a bulk copy that completes on the even CTA's sfull barrier, so the
        // barrier also covers this CTA's own chunks.  (A thread's arrive on the
        // other CTA's barrier measured ~0.9 us per group here; the copy is
        // asynchronous, and the even CTA's MMA warp does no layout work.)
        if constexpr (C::kFuseSa) {
            if (p.sa_fused && !p.test_stall) {
                const uint64_t pol_a = p.stream_a ? l2_policy_evict_first() : l2_policy_evict_last();
                WorkIter wi;
                wi.init(p, first_unit, unit_step, gt, 2 * kBM);
                Work w;
                bool in_unit = false;
                int kb = 0, kb0 = 0;
                // the next scale group in the order the producer and MMA warps meet them
                auto next_group = [&](int &kt0, int &row0) -> bool {
                    for (;;) {
                        if (!in_unit) {
                            if (!wi.next(p, w))
                                return false;
                            in_unit = true;
                            kb0 = w.ks0 & ~1;
                            kb = kb0;
                        }
                        while (kb < w.ks1) {
                            const int k = kb;
                            kb += 2;
                            if (group_start(k, kb0)) {
                                kt0 = (k - k % kSfGroup) * C::kKtPerStage;
                                row0 = 2 * w.tm * kBM;
                                return true;
                            }
                        }
                        in_unit = false;
                    }
                };
                uint32_t armed = 0, armed_ph = 0;  // staging loads in flight
                auto load_raw = [&](int b, uint32_t use, int kt0, int row0) {
                    if (elect_one()) {
                        mbar_arrive_expect_tx(araw_bar(b), C::kSaRawBytes);
                        tma_load_2d(sRaw + b * C::kSaRawBytes, &map_sarm, araw_bar(b), 4 * kt0, row0, pol_a);
                    }
                    __syncwarp();
                    armed |= 1u << b;
                    armed_ph = (armed_ph & ~(1u << b)) | ((use & 1u) << b);
                };
                int kt_cur = 0, row_cur = 0, kt_nxt = 0, row_nxt = 0;
                bool has_cur = next_group(kt_cur, row_cur);
                if (has_cur)
                    load_raw(0, 0u, kt_cur, row_cur);
                bool ok = true;
                for (int gi = 0; has_cur; ++gi) {
                    const int rb = gi & 1;  // staging buffer
                    const int gs = gi % G;  // group slot and side buffer
                    const uint32_t use = static_cast<uint32_t>(gi / G);
                    // prefetch the next group (its staging buffer was last read by the
                    // layout of group gi - 1, already done)
                    const bool has_nxt = next_group(kt_nxt, row_nxt);
                    if (has_nxt)
                        load_raw(rb ^ 1, static_cast<uint32_t>((gi + 1) >> 1), kt_nxt, row_nxt);
                    // staging landed; group slot gs (and side buffer gs) no longer read:
                    // the MMA warp's copies of group gi - G have completed
                    if (!warp_wait(araw_bar(rb), static_cast<uint32_t>(gi >> 1) & 1u, abort, lim) ||
                        (gi >= G && !warp_wait_cluster(sempty_bar(gs), (use & 1u) ^ 1u, abort, lim))) {
                        if (lane == 0) record_timeout(p, abort);
                        ok = false;
                        break;
                    }
                    armed &= ~(1u << rb);
                    // chunk u (K-tile u of the group), byte 16p + 4q + c = row 32q + p,
                    // K-block c; staging row r = the pair's row r (even CTA: 0..127)
                    const uint8_t *src = smem_raw + (sRaw - raw) + rb * C::kSaRawBytes;
                    uint8_t *own = smem_raw + (sSF - raw) + gs * C::kSfGrpBytes;
                    uint8_t *lead = smem_raw + (sLead - raw) + gs * C::kSaLeadBytes;
                    uint4 rowv[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        rowv[q] = reinterpret_cast<const uint4 *>(src)[32 * q + lane];
#pragma unroll
                    for (int u = 0; u < kSfGroup; ++u) {
                        auto word = [&](const uint4 &x) { return u == 0 ? x.x : u == 1 ? x.y : u == 2 ? x.z : x.w; };
                        reinterpret_cast<uint4 *>(lead + u * kSfChunk)[lane] =
                            make_uint4(word(rowv[0]), word(rowv[1]), word(rowv[2]), word(rowv[3]));
                        reinterpret_cast<uint4 *>(own + u * kSfChunk)[lane] =
                            make_uint4(word(rowv[4]), word(rowv[5]), word(rowv[6]), word(rowv[7]));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (elect_one())
                        bulk_copy_s2s_cluster(map_to_cta(sSF + gs * C::kSfGrpBytes, 0), sLead + gs * C::kSaLeadBytes,
                                              C::kSaLeadBytes, map_to_cta(sfull_bar(gs), 0));
                    __syncwarp();
                    kt_cur = kt_nxt;
                    row_cur = row_nxt;
                    has_cur = has_nxt;
                }
                if (!ok)
                    for (int b2 = 0; b2 < 2; ++b2)
                        if (armed & (1u << b2))
                            warp_wait(araw_bar(b2), (armed_ph >> b2) & 1u, no_abort, lim);
            }
        }
    } else if (warp == 1 && leader) {
        // -------------------------------------- even CTA: MMA issuer for the pair
        int st = 0;
        uint32_t ph = 0;
        int it = 0;
        int gi = 0;  // scale groups started
        bool ok = true;
        bool issued = false;
        // Scale group in, for the group holding k-stage kb, whose stages
        // [lo, hi) belong to the work unit: wait until both CTAs' group slots
        // are complete (copies landed, fused layouts done) and the TMEM
        // regions the group goes to are no longer read (the MMAs of the group
        // kGrp before have completed); copy each CTA's chunks of the unit's stages
        // into its own TMEM (one region per stage); commit so both producers may
        // refill their slot.
        auto group_in = [&](int kb, int lo, int hi) -> bool {
            const int gs = gi % G;
            const uint32_t use = static_cast<uint32_t>(gi / G);
            if (!warp_wait_cluster(sfull_bar(gs), use & 1u, abort, lim))
                return false;
            if (gi >= G && !warp_wait(tfree_bar(gs), (use & 1u) ^ 1u, abort, lim))
                return false;
            tc_fence_after();
            const uint32_t src = sSF + gs * C::kSfGrpBytes;
            const int g0 = kb - kb % kSfGroup;
            // one elected lane issues the group's copies (and, below, the MMAs
            // and commits) in one block: separate elect blocks per instruction
            // measured up to 10% slower on long k-loops
            if (elect_one()) {
#pragma unroll 1
                for (int k = lo; k < hi; ++k) {
                    const int j = k - g0;
                    const int nkt_ = min(C::kKtPerStage, p.num_kt - k * C::kKtPerStage);
                    const uint32_t sfa_col_ = tmem + C::kSfCol0 + (gs * kSfGroup + j) * C::kSfSlotCols;
                    const uint32_t sfb_col_ = sfa_col_ + C::kSfaCols;
#pragma unroll
                    for (int t = 0; t < C::kKtPerStage; ++t) {
                        if (t < nkt_) {
                            tc_cp_pair_32x128b_warpx4(sfa_col_ + 4 * t,
                                                      sdesc_sf_chunk(src + (j * C::kKtPerStage + t) * kSfChunk));
#pragma unroll
                            for (int c = 0; c < C::kChunksB; ++c)
                                tc_cp_pair_32x128b_warpx4(
                                    sfb_col_ + 4 * (t * C::kChunksB + c),
                                    sdesc_sf_chunk(src + C::kSfaGrpBytes +
                                                   ((c * kSfGroup + j) * C::kKtPerStage + t) * kSfChunk));
                        }
                    }
                }
                tc_commit_pair(sempty_bar(gs), 0x3);
            }
            __syncwarp();
            issued = true;
            ++gi;
            return true;
        };
        // A unit's first scale group is copied in before the accumulator wait:
        // its TMEM regions are not the accumulator's, so the copies overlap the
        // previous tile's drain and epilogue instead of delaying the first MMAs
        // (at a tile start the group's waits and copies took ~1.5 us).
        auto first_group_in = [&](const Work &u) -> bool {
            if constexpr (!C::kScaled) {
                return true;
            } else {
                const int kb0 = u.ks0 & ~1;
                const int g0 = kb0 - kb0 % kSfGroup;
                return group_in(kb0, max(u.ks0, g0), min(u.ks1, g0 + kSfGroup));
            }
        };
        WorkIter wi;
        wi.init(p, first_unit, unit_step, gt, 2 * kBM);
        Work w;
        bool have = wi.next(p, w);
        if (have && !first_group_in(w)) {
            if (lane == 0) record_timeout(p, abort);
            ok = false;
        }
        for (; ok && have; ++it) {
            const int acc = it % C::kAccStages;
            const uint32_t acc_par = static_cast<uint32_t>((it / C::kAccStages) & 1);
            if (!warp_wait_cluster(acce_bar(acc), acc_par ^ 1u, abort, lim)) {
                if (lane == 0) record_timeout(p, abort);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + acc * BN;
            const int ks0 = w.ks0, ks1 = w.ks1;
            const int kb0 = ks0 & ~1;
            // 32-row group of the tile's first B-role row in its scale chunk (0 unless BN = 192)
            const uint32_t sub_b = static_cast<uint32_t>(((w.tn * BN) & 127) >> 5);
            for (int kb = kb0; kb < ks1; kb += 2) {
                if (kb != kb0 && group_start(kb, kb0)) {
                    const int g0 = kb - kb % kSfGroup;
                    if (!group_in(kb, max(ks0, g0), min(ks1, g0 + kSfGroup))) {
                        if (lane == 0) record_timeout(p, abort);
                        ok = false;
                        break;
                    }
                }
                if (!warp_wait_cluster(full_bar(st), ph, abort, lim)) {
                    if (lane == 0) record_timeout(p, abort);
                    ok = false;
                    break;
                }
                tc_fence_after();
                issued = true;
                const int gcur = gi - 1;  // the scale group of the slot's stages
                // the group's TMEM regions are free again after the MMAs of its last slot
                const bool group_end = C::kScaled && ((kb + 2) % kSfGroup == 0 || kb + 2 >= ks1);
                if (elect_one()) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int kk = kb + h;
                        if (kk >= ks0 && kk < ks1) {
                            const int nkt = min(C::kKtPerStage, p.num_kt - kk * C::kKtPerStage);
                            const uint32_t sfa_col =
                                tmem + C::kSfCol0 + ((gcur % G) * kSfGroup + kk % kSfGroup) * C::kSfSlotCols;
                            const uint32_t sfb_col = sfa_col + C::kSfaCols;
                            const uint64_t adesc = sdesc_kmajor_sw128(sA + (st * 2 + h) * C::kABytes);
                            const uint64_t bdesc = sdesc_kmajor_sw128(sB + (st * 2 + h) * C::kBBytes);
                            const uint32_t acc0 = (kk > ks0) ? 1u : 0u;
#pragma unroll
                            for (int s = 0; s < C::kKtPerStage * C::kSubPerKt; ++s) {
                                const int t = s / C::kSubPerKt;
                                if (t < nkt) {
                                    const uint32_t sf_id = C::kFp4 ? static_cast<uint32_t>((s % 2) * 2)
                                                                   : static_cast<uint32_t>(s % 4);
                                    const uint32_t idesc = idesc_with_sf_ids(C::kIdesc, sf_id, sf_id);
                                    const uint32_t sfa_t = sfa_col + 4 * t;
                                    const uint32_t sfb_t = sfb_col + 4 * t * C::kChunksB + sub_b;
                                    const uint64_t koff = static_cast<uint64_t>((s * 32) >> 4);
                                    const uint32_t accum = (s > 0) ? 1u : acc0;
                                    if constexpr (KIND == K_BF16)
                                        mma_pair_bf16(d_tmem, adesc + koff, bdesc + koff, C::kIdesc, accum);
                                    else if constexpr (C::kFp4)
                                        mma_pair_mxf4(d_tmem, adesc + koff, bdesc + koff, idesc, sfa_t, sfb_t, accum);
                                    else
                                        mma_pair_mxf8f6f4(d_tmem, adesc + koff, bdesc + koff, idesc, sfa_t, sfb_t,
                                                          accum);
                                }
                            }
                        }
                    }
                    tc_commit_pair(empty_bar(st), 0x3);
                    if (group_end)
                        tc_commit_pair(tfree_bar(gcur % G), 0x1);
                }
                __syncwarp();
                if (++st == S) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            if (elect_one())
                tc_commit_pair(accf_bar(acc), 0x3);
            __syncwarp();
            have = wi.next(p, w);
            if (have && !first_group_in(w)) {
                if (lane == 0) record_timeout(p, abort);
                ok = false;
            }
        }
        if (!ok && issued) {
            if (elect_one())
                tc_commit_pair(drain_bar, 0x1);
            __syncwarp();
            warp_wait(drain_bar, 0, no_abort, lim);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        constexpr int kCols = BN / 2;
        constexpr int kChunks = kCols / 32;
        __shared__ int sk_last;
        int it = 0;
        WorkIter wi;
        wi.init(p, first_unit, unit_step, gt, 2 * kBM);
        Work w;
        for (; wi.next(p, w); ++it) {
            const int tm = w.tm, tn = w.tn;
            const int acc = it % C::kAccStages;
            const uint32_t acc_par = static_cast<uint32_t>((it / C::kAccStages) & 1);
            if (!warp_wait_cluster(accf_bar(acc), acc_par, abort, lim)) {
                if (lane == 0) record_timeout(p, abort);
                break;
            }
            tc_fence_after();
            uint32_t r[kChunks][32];
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
            // Hand the accumulator stage back to the even CTA's MMA warp.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_cta(acce_bar(acc), 0));

            const int row0 = (2 * tm + static_cast<int>(rank)) * kBM;  // this CTA's 128 rows
            if constexpr (SK) {
                if (w.kind == 1) {
                    // stream-K segment: publish, and add the tile's segments if this pair is last
                    sk_epilogue<BN, kCols, kChunks, true>(p, w, r, first_unit, 2, static_cast<int>(rank), row0, h,
                                                          q * 32 + lane, true, &sk_last, nullptr, 0u, 0u, nullptr,
                                                          abort, lim);
                    continue;
                }
            }
            // Output limits and origin (plain: the whole C; grouped: the group's rows)
            int lim_i = p.rows_a, lim_j = p.rows_b;
            long long out0 = 0;
            if constexpr (GROUPED) {
                PairGeom pg;
                pair_geom<BN>(p, gt, w, static_cast<int>(rank), pg);
                lim_i = pg.lim_i;
                lim_j = pg.lim_j;
                out0 = pg.out_base;
            }
            const int i = row0 + q * 32 + lane;
            if (i < lim_i) {
                const long long base_off = out0 +
                                           (w.kind == 2 ? static_cast<long long>(w.slot) * p.split_stride : 0ll) +
                                           static_cast<long long>(i) * p.stride_i;
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    const int j0 = tn * BN + h * kCols + c * 32;
                    if (j0 >= lim_j) break;
                    if (p.vec_ok && j0 + 32 <= lim_j)
                        store_row32_vec<true>(p, base_off + j0, r[c]);
                    else
                        store_row32_masked(p, base_off, j0, min(32, lim_j - j0), r[c]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still touch its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::kTmemCols);
    }
}

}  // namespace mxg
