// The two GEMMs of the tensor-parallel MLP block on CTA pairs (tcgen05 cta_group::2).
//
// Same computation and epilogues as tpmlp_gemm.cuh (Y_i = GeLU(X W1_i + b1_i) for every shard;
// Z = b2 + sum_i Y_i W2_i with the sum over shards taken in one fp32 accumulator), but each
// output tile is 256 x 256 and is computed by a cluster of two CTAs on two SMs:
//
//   CTA rank r (r = 0, 1) of the pair loads rows [m0 + 128 r, +128) of A and rows
//   [n0 + 128 r, +128) of B into its own shared memory. One thread of rank 0 issues
//   tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): the tensor cores read A and B from
//   both CTAs and write rows [128 r, +128) of the 256 x 256 fp32 accumulator into CTA r's
//   tensor memory.
//
// Per CTA a pipeline stage is 32 KB (instead of 48 KB for a 128 x 256 tile on one SM), so the
// same shared memory holds more stages in flight, and every operand byte fetched from L2
// feeds twice as many multiply-adds.
//
// Synchronisation:
//   full[s]   (rank 0)  rank 0 arms it with both CTAs' bytes; both CTAs' TMA loads complete on it
//   empty[s]  (both)    the MMA thread's multicast commit frees stage s in both CTAs
//   tfull[a]  (both)    multicast commit: accumulator a is complete in both CTAs
//   tempty[a] (rank 0)  one arrival per epilogue warp of both CTAs: accumulator a has been read
// All waits are bounded (ptx::mbar_wait); see tpmlp_gemm.cuh for the abort protocol.
#pragma once

#include "tpmlp_gemm.cuh"

namespace tpmlp {

// How long the first pair of a split tile waits for the others' partial sums before it hands
// the tile over (see the epilogue).
#ifndef TPMLP_SPLIT_WAIT_NS
#define TPMLP_SPLIT_WAIT_NS 50000
#endif
constexpr uint64_t kSplitWaitNs = TPMLP_SPLIT_WAIT_NS;

constexpr int kPairBM = 256;  // output rows per pair tile (128 per CTA)
constexpr int kPairBN = 256;  // output columns per pair tile (B: 128 rows per CTA)

// TALL: a stage also holds the CTA's 128 rows of A of a tall unit's second half (after the
// first half's), so that one B tile feeds both halves' MMAs (see GemmArgs::tall_units).
template <int STAGES, int NUM_ACC, bool TALL = false>
struct PairSmem {
    static constexpr uint32_t kABytes = (TALL ? 2 : 1) * 128 * kBK * 2;  // this CTA's A rows
    static constexpr uint32_t kBBytes = 128 * kBK * 2;  // this CTA's 128 rows of B
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kCtrlBytes = 8 * (2 * STAGES + 2 * NUM_ACC + 1) + 8;
    static constexpr uint32_t kEpiOffset = STAGES * kStageBytes + (kCtrlBytes + 127) / 128 * 128;
    static constexpr uint32_t kTotal = 1024 + kEpiOffset + kEpiWarps * kStageSliceBytes;
    static_assert(kTotal <= 232448, "dynamic shared memory per CTA");
    static constexpr uint32_t kTmemCols = NUM_ACC * kPairBN;  // 256 or 512
};

// MN: both operands M-/N-contiguous (the weight-gradient GEMMs): each CTA loads its 128 rows
// of A and of B as two 64 (MN) x 64 (K) boxes each (see tpmlp_gemm_kernel).
// TALL (second-GEMM modes, two accumulators): each pair first computes tall units of
// 512 x 256 outputs (whole 512-row blocks), args.tall_units of them round robin, with both
// accumulators: per
// reduction block one B tile and the A tiles of both 256-row halves, two MMAs per 16-deep
// step. Against two 256 x 256 tiles that is a quarter less operand traffic per multiply-add;
// the accumulators are not double-buffered then, so a unit's epilogue does not overlap the
// next unit's MMAs. The launch's tiles follow as usual (see decode_tile).
template <int STAGES, int NUM_ACC, Mode MODE, bool OUT_F32, bool MN = false, bool TALL = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kNumThreads, 1)
    tpmlp_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmB2, const GemmArgs args) {
    static_assert(!TALL || ((MODE == Mode::kGemm2 || MODE == Mode::kGemm2Residual) && !MN &&
                            NUM_ACC == 2),
                  "tall units: second GEMM, two accumulators");
    using L = PairSmem<STAGES, NUM_ACC, TALL>;
    constexpr uint32_t kIdesc = idesc_bf16_f32(kPairBM, kPairBN, MN);
    constexpr int kCode = (static_cast<int>(MODE) << 8) | 0x80;  // 0x80: pair kernel

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    const uint32_t ctrl = base + STAGES * L::kStageBytes;
    auto full_bar = [&](int s) { return ctrl + 8u * s; };
    auto empty_bar = [&](int s) { return ctrl + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return ctrl + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return ctrl + 8u * (2 * STAGES + NUM_ACC + b); };
    const uint32_t drain_bar = ctrl + 8u * (2 * STAGES + 2 * NUM_ACC);
    uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(
        base_ptr + STAGES * L::kStageBytes + 8 * (2 * STAGES + 2 * NUM_ACC + 1));
    volatile uint32_t* const abort_flag = tmem_holder + 1;

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 5, 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < NUM_ACC; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), 2 * kEpiWarps);
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        if (!is_gemm1(MODE) && !MN && args.k2 < args.k) ptx::prefetch_tensormap(&tmB2);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_addr(tmem_holder), L::kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();  // barriers of both CTAs initialised, tensor memory allocated
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // The set-up above overlaps the previous kernel's tail; global memory only from here on.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------- TMA producer (both CTAs)
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            // the B rows and the A rows of reduction block kb of the second GEMM (shard-major)
            auto load_b = [&](uint32_t sb, uint32_t fb, int kb, int nb) {
                const int i = kb / args.kb_shard;
                const int kk = (kb - i * args.kb_shard) * kBK;
                const bool second = i >= args.k2;
                if (args.b_blocked)  // block (shard i, rows nb / 128, columns kk / 64)
                    ptx::tma_load_2d_pair(
                        sb, &tmB, fb, 0,
                        ((i * (args.ldo / 128) + nb / 128) * (args.f / kBK) + kk / kBK) * 128);
                else
                    ptx::tma_load_3d_pair(sb, second ? &tmB2 : &tmB, fb, kk, nb,
                                          second ? i - args.k2 : i);
            };
            auto load_a = [&](uint32_t sa, uint32_t fb, int kb, int m0) {
                const int i = kb / args.kb_shard;
                ptx::tma_load_2d_pair(sa, &tmA, fb, i * args.f + (kb - i * args.kb_shard) * kBK, m0);
            };
            if constexpr (TALL) {
                for (int u = pair; ok && u < args.tall_units; u += num_pairs) {
                    int tm, n_blk;
                    decode_tile_mn(args.group_m, args.tall_m_blocks, args.n_blocks, u, tm, n_blk);
                    const int m0 = tm * 2 * kPairBM + static_cast<int>(rank) * 128;
                    const int nb = n_blk * kPairBN + static_cast<int>(rank) * 128;
                    constexpr uint32_t bytes = 2 * L::kStageBytes;  // both CTAs: two A boxes, B
                    const bool backwards = args.tall_serpentine && ((u / num_pairs) & 1);
                    for (int i = 0; i < args.kb_tile; ++i) {
                        const int kb = backwards ? args.kb_tile - 1 - i : i;
                        if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.status,
                                            kCode | kSiteProducer)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sa = base + stage * L::kStageBytes;
                        const uint32_t fb = ptx::mapa_shared(full_bar(stage), 0);
                        if (leader) ptx::mbar_arrive_expect_tx(full_bar(stage), bytes);
                        load_a(sa, fb, kb, m0);
                        load_a(sa + 128 * kBK * 2, fb, kb, m0 + kPairBM);
                        load_b(sa + L::kABytes, fb, kb, nb);
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            WorkCursor cur = work_begin(args.sk_iters, pair, num_pairs);
            int t, kb0, kb1;
            while (ok && work_next(args.sk_first, args.kb_tile, num_pairs, cur, t, kb0, kb1)) {
                int m_blk, n_blk;
                decode_tile(args, t, m_blk, n_blk);
                const int m0 = m_blk * kPairBM + static_cast<int>(rank) * 128;  // this CTA's A rows
                const int n0 = n_blk * kPairBN;
                const int nb = n0 + static_cast<int>(rank) * 128;  // this CTA's B rows
                const int shard1 = is_gemm1(MODE) ? n0 / args.f : 0;
                const int nb_in_shard1 = nb - shard1 * args.f;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.status,
                                        kCode | kSiteProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + stage * L::kStageBytes;
                    const uint32_t sb = sa + L::kABytes;
#ifdef TPMLP_TEST_SKIP_STAGE
                    // test builds only: rank 0 never arms this stage, so the MMA's wait runs out
                    if (leader && issued == TPMLP_TEST_SKIP_STAGE) {
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
#endif
                    const uint32_t fb = ptx::mapa_shared(full_bar(stage), 0);  // rank 0's barrier
                    if (leader)  // both CTAs' A (one 128-row box each) and B tiles
                        ptx::mbar_arrive_expect_tx(full_bar(stage), 2 * (128 * kBK * 2 + L::kBBytes));
                    if constexpr (MN) {
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            ptx::tma_load_2d_pair(sa + b * 8192, &tmA, fb, m0 + 64 * b, kb * kBK);
                            ptx::tma_load_2d_pair(sb + b * 8192, &tmB, fb, nb + 64 * b, kb * kBK);
                        }
                    } else if constexpr (is_gemm1(MODE)) {
                        ptx::tma_load_2d_pair(sa, &tmA, fb, kb * kBK, m0);
                        ptx::tma_load_3d_pair(sb, &tmB, fb, kb * kBK, nb_in_shard1, shard1);
                    } else {
                        load_a(sa, fb, kb, m0);
                        load_b(sb, fb, kb, nb);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (leader) {
                    for (uint32_t s = 0; s < STAGES && s < issued; ++s) {
                        const uint32_t last = s + ((issued - 1 - s) / STAGES) * STAGES;
                        ptx::mbar_wait_drain(full_bar(s), (last / STAGES) & 1u);
                    }
                } else {
                    // this CTA's copies complete on rank 0's barriers: give them time to land
                    const uint64_t t0 = ptx::globaltimer_ns();
                    while (ptx::globaltimer_ns() - t0 < 2000000ull) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer (rank 0)
        if (leader && lane == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            if constexpr (TALL) {
                // a tall unit takes both accumulators (acc is 0 at the start of each: units
                // come first and take two each)
                for (int u = pair; ok && u < args.tall_units; u += num_pairs) {
                    if (!ptx::mbar_wait(tempty_bar(0), acc_phase ^ 1u, abort_flag, args.status,
                                        kCode | kSiteMmaAccum) ||
                        !ptx::mbar_wait(tempty_bar(1), acc_phase ^ 1u, abort_flag, args.status,
                                        kCode | kSiteMmaAccum)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    for (int kb = 0; kb < args.kb_tile; ++kb) {
                        if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag, args.status,
                                            kCode | kSiteMmaFull)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t sa = base + stage * L::kStageBytes;
                        const uint64_t da0 = sdesc_k128(sa);
                        const uint64_t da1 = sdesc_k128(sa + 128 * kBK * 2);
                        const uint64_t db = sdesc_k128(sa + L::kABytes);
#pragma unroll
                        for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                            const uint32_t accumulate = (kb != 0 || kk != 0) ? 1u : 0u;
                            ptx::mma_bf16_ss_pair(tmem_base, da0 + 2u * kk, db + 2u * kk, kIdesc,
                                                  accumulate);
                            ptx::mma_bf16_ss_pair(tmem_base + kPairBN, da1 + 2u * kk,
                                                  db + 2u * kk, kIdesc, accumulate);
                        }
                        ptx::mma_commit_pair(empty_bar(stage), 0x3);  // stage s free in both CTAs
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit_pair(tfull_bar(0), 0x3);  // both accumulators ready
                    ptx::mma_commit_pair(tfull_bar(1), 0x3);
                    acc_phase ^= 1u;
                }
            }
            WorkCursor cur = work_begin(args.sk_iters, pair, num_pairs);
            int t, kb0, kb1;
            while (ok && work_next(args.sk_first, args.kb_tile, num_pairs, cur, t, kb0, kb1)) {
                if (!ptx::mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.status,
                                    kCode | kSiteMmaAccum)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kPairBN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag, args.status,
                                        kCode | kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = base + stage * L::kStageBytes;
                    const uint64_t da = MN ? sdesc_mn128(sa) : sdesc_k128(sa);
                    const uint64_t db = MN ? sdesc_mn128(sa + L::kABytes) : sdesc_k128(sa + L::kABytes);
                    constexpr uint32_t kStep = MN ? 128u : 2u;  // 16 K: 32 B (K-major), 2 KB (MN)
#pragma unroll
                    for (int kk = 0; kk < kBK / kUmmaK; ++kk)
                        ptx::mma_bf16_ss_pair(d_tmem, da + kStep * kk, db + kStep * kk, kIdesc,
                                              (kb != kb0 || kk != 0) ? 1u : 0u);
                    ptx::mma_commit_pair(empty_bar(stage), 0x3);  // stage s free in both CTAs
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit_pair(tfull_bar(acc), 0x3);  // accumulator ready in both CTAs
                if (++acc == NUM_ACC) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            ptx::mma_commit_pair(drain_bar, 0x1);
            ptx::mbar_wait_drain(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- epilogue (both CTAs)
        const int q = warp & 3;
        const int part = (warp - 2) >> 2;
        uint32_t acc = 0, acc_phase = 0;
        const int ew = warp - 2;  // epilogue warp index: its arrival counter in a split tile
        bool ok_tall = true;
        if constexpr (TALL) {
            const uint32_t stage_buf = base + L::kEpiOffset + (warp - 2) * kStageSliceBytes;
            for (int u = pair; u < args.tall_units; u += num_pairs) {
                int tm, n_blk;
                decode_tile_mn(args.group_m, args.tall_m_blocks, args.n_blocks, u, tm, n_blk);
                const bool ok = ptx::mbar_wait(tfull_bar(0), acc_phase, abort_flag, args.status,
                                               kCode | kSiteEpilogue) &&
                                ptx::mbar_wait(tfull_bar(1), acc_phase, abort_flag, args.status,
                                               kCode | kSiteEpilogue);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok_tall = false;
                    break;
                }
                ptx::tc_fence_after();
                const int row0 = tm * 2 * kPairBM + static_cast<int>(rank) * 128 + q * 32 + lane;
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
                auto release = [&] {  // both accumulators' columns are in registers
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::mbar_arrive_cluster_relaxed(ptx::mapa_shared(tempty_bar(0), 0));
                        ptx::mbar_arrive_cluster_relaxed(ptx::mapa_shared(tempty_bar(1), 0));
                    }
                };
                drain_tall<MODE, OUT_F32, kPairBN>(taddr, taddr + kPairBN, args, row0,
                                                   row0 + kPairBM, n_blk * kPairBN, part,
                                                   stage_buf, release);
                acc_phase ^= 1u;
            }
        }
        WorkCursor cur = work_begin(args.sk_iters, pair, num_pairs);
        int t, kb0, kb1;
        if (!TALL) {
            WorkCursor first = cur;
            if (work_next(args.sk_first, args.kb_tile, num_pairs, first, t, kb0, kb1))
                prefetch_tile_bias<MODE, kPairBN>(args, t, part);
        }
        while (ok_tall && work_next(args.sk_first, args.kb_tile, num_pairs, cur, t, kb0, kb1)) {
            int m_blk, n_blk;
            decode_tile(args, t, m_blk, n_blk);
            const int m0 = m_blk * kPairBM + static_cast<int>(rank) * 128;
            const int n0 = n_blk * kPairBN;
            bool ok = ptx::mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.status,
                                     kCode | kSiteEpilogue);
            if (!__all_sync(0xffffffffu, ok)) break;
            ptx::tc_fence_after();
            const int row = m0 + q * 32 + lane;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kPairBN;
            const uint32_t empty = ptx::mapa_shared(tempty_bar(acc), 0);  // rank 0's barrier
            auto release = [&] {  // the accumulator's columns are in registers: hand it back
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster_relaxed(empty);
            };
            const uint32_t stage_buf = base + L::kEpiOffset + (warp - 2) * kStageSliceBytes;
            bool epilogue = true;
            if (kb0 != 0 || kb1 != args.kb_tile) {
                // Part of a split tile, held by pairs p_first .. p_last. The other pairs publish
                // their partial sums and count in. The pair holding the tile's first blocks
                // works on them last in its share, so the others are normally in by then: it
                // waits for them (kSplitWaitNs at most), then sums all parts in pair order from
                // its accumulator and the published partials and runs the epilogue. If they are
                // not all in by then (a pair not yet resident while other work holds SMs), it
                // publishes its own part and counts in too, and whichever pair counts in last
                // finishes the tile. The count reaches its total only through the first pair,
                // so exactly one warp finishes each tile, and no wait outlives kSplitWaitNs.
                const int lrow = q * 32 + lane;
                const long long i0 = static_cast<long long>(t - args.sk_first) * args.kb_tile;
                const int p_first = work_pair_of(args.sk_iters, num_pairs, i0);
                const int p_last = work_pair_of(args.sk_iters, num_pairs, i0 + args.kb_tile - 1);
                const uint32_t n_parts = static_cast<uint32_t>(p_last - p_first + 1);
                uint32_t* const counter =
                    args.sk_count + (static_cast<size_t>(t - args.sk_first) * 2 + rank) * kEpiWarps + ew;
                bool finish = false;
                if (kb0 == 0) {
                    uint32_t in = 0;
                    if (lane == 0)
                        in = ptx::epoch_count_wait(counter, args.sk_epoch, n_parts - 1, kSplitWaitNs,
                                                   abort_flag);
                    finish = __shfl_sync(0xffffffffu, in, 0) == n_parts - 1;
                }
                if (!finish) {
                    save_partial<MODE, kPairBN>(
                        taddr, part, split_slot(args.sk_partial, pair, kb0 > 0 ? 0 : 1, rank), lrow);
                    __threadfence();  // the partial is visible before the arrival is
                    __syncwarp();
#ifdef TPMLP_TEST_LATE_PARTIALS
                    // test builds only: the other pairs count in late, so that the first pair
                    // hands its tiles over and they finish them
                    if (kb0 > 0) {
                        const uint64_t t_late = ptx::globaltimer_ns();
                        while (ptx::globaltimer_ns() - t_late < 200000ull) {
                        }
                    }
#endif
                    uint32_t arrivals = 0;
                    bool counted = true;
                    if (lane == 0)
                        counted = ptx::epoch_arrive(counter, args.sk_epoch, &arrivals, abort_flag,
                                                    args.status, kCode | kSiteSplitCount);
                    arrivals = __shfl_sync(0xffffffffu, arrivals, 0);
                    counted = __shfl_sync(0xffffffffu, counted, 0);
                    finish = counted && arrivals == n_parts;
                }
                if (finish) {
                    __threadfence();  // every other partial of the tile is visible
                    if (pair == p_first)
                        fold_partials<MODE, kPairBN>(taddr, part, args.sk_partial, rank, p_first,
                                                     p_last, lrow);
                    else
                        reduce_partials<MODE, kPairBN>(taddr, part, args.sk_partial, rank,
                                                       p_first, p_last, pair, lrow);
                } else {
                    release();
                }
                epilogue = finish;
            }
            if (epilogue)
                drain_accumulator<MODE, OUT_F32, kPairBN>(taddr, args, row, n0, part, stage_buf,
                                                          release);
            if (++acc == NUM_ACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_sync();  // no CTA leaves while its peer may still signal it
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, L::kTmemCols);
    }
}

}  // namespace tpmlp
