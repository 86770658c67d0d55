// Work planning shared by the host code, the GEMM kernels and the host tests (plain C++; the
// host tests build it with g++ alone):
//   1. the split reduction's plan and the CTA-pair kernel's walk over its work units;
//   2. the row-chunk planner of the host-buffer forward pass.
//
// ---------------------------------------------------------------- 1. split reduction
//
// A CTA-pair launch of T output tiles, each reduced over kb_tile blocks of 64, on P resident
// pairs. Tile t covers row block m and column block n of the output (decode_tile_mn: groups of
// group_m row blocks, each swept column by column, alternate groups in reverse, so that the
// tiles running at once share operand rows and columns in L2). Tiles [0, sk_first) are whole units, handed out round robin
// (pair p: p, p + P, ...).
// The sk_iters = (T - sk_first) * kb_tile reduction blocks of the remaining tiles, in tile
// order, are cut into P contiguous shares [floor(S p / P), floor(S (p + 1) / P)) that every
// role of a pair walks in order. A pair whose share starts inside a tile writes its partial sum
// for the owner of that tile: the pair that holds the tile's first block, last in its share.
//
// ---------------------------------------------------------------- 2. host-buffer chunks
//
// Token rows are independent, so a forward pass on host buffers can stream: the copy of chunk
// c + 1 in (and of chunk c - 1 out) overlaps the GEMMs of chunk c. Two effects pull the chunk
// sizes apart. The copy of the first chunk in and of the last chunk out cannot overlap any
// compute, which favours small end chunks. Each chunk's GEMMs run in rounds of tiles over the
// GPU's tile slots (CTA pairs or SMs), and a chunk whose tile count is just above a multiple
// of the slots pays for a nearly empty round, which favours chunk sizes that fill whole rounds.
// The planner scores every split of the rows into at most `max_chunks` chunks of whole
// 256-row blocks under a pipeline model and keeps the fastest.
//
// The model: one copy stream in, one copy stream out, one compute stream.
//   in_c   = in_{c-1} + X bytes of chunk c / bandwidth in
//   comp_c = max(comp_{c-1}, in_c) + sum over both GEMMs of (rounds(chunk c) * round time
//            + a fixed cost per launch)
//   out_c  = max(out_{c-1}, comp_c) + Z bytes of chunk c / bandwidth out
// and the pass ends at max(comp_last, out_last).
//
// ---------------------------------------------------------------- 3. device rates
//
// Both planners weigh the time of a round of tiles against DRAM reads or host-link copies.
// The rates come from the device a context runs on (device_rates), so that a part with
// another SM count, clock or memory system plans from its own round times.
#pragma once

#include <cstdint>
#include <vector>

#if defined(__CUDACC__)
#define TPMLP_HD __host__ __device__ __forceinline__
#else
#define TPMLP_HD inline
#endif

namespace tpmlp {

// Tile t of a launch of m_blocks x n_blocks tiles: groups of group_m row blocks, each swept
// column by column, every second group in reverse column order ("snake"), so that a wave of
// tiles that straddles two groups reads the same column blocks in both. Interleaved A/B
// against all groups sweeping forward (second GEMM, bit-identical where no tile is split):
// 587.5 -> 582.5 us at 7b, 2902 -> 2887 us at GPT-3.
TPMLP_HD void decode_tile_mn(int group_m, int m_blocks, int n_blocks, int t, int& m_blk,
                             int& n_blk) {
    const int per_group = group_m * n_blocks;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int gm = m_blocks - first_m < group_m ? m_blocks - first_m : group_m;
    const int local = t - g * per_group;
    m_blk = first_m + local % gm;
    n_blk = local / gm;
    if (g & 1) n_blk = n_blocks - 1 - n_blk;
}

struct WorkCursor {
    int t;                // next whole tile of this pair
    long long it, it_end; // this pair's share of the split blocks
};

TPMLP_HD WorkCursor work_begin(int sk_iters, int pair, int num_pairs) {
    WorkCursor c;
    c.t = pair;
    c.it = static_cast<long long>(sk_iters) * pair / num_pairs;
    c.it_end = static_cast<long long>(sk_iters) * (pair + 1) / num_pairs;
    return c;
}

// The next work unit of a pair: tile `tile`, reduction blocks [kb0, kb1). False when done.
TPMLP_HD bool work_next(int sk_first, int kb_tile, int num_pairs, WorkCursor& c, int& tile,
                        int& kb0, int& kb1) {
    if (c.t < sk_first) {
        tile = c.t;
        kb0 = 0;
        kb1 = kb_tile;
        c.t += num_pairs;
        return true;
    }
    if (c.it < c.it_end) {
        const long long rel = c.it / kb_tile;
        kb0 = static_cast<int>(c.it - rel * kb_tile);
        const long long left = c.it_end - c.it;
        kb1 = static_cast<int>(kb0 + left < kb_tile ? kb0 + left : kb_tile);
        tile = sk_first + static_cast<int>(rel);
        c.it += kb1 - kb0;
        return true;
    }
    return false;
}

// The pair whose share holds split block i.
TPMLP_HD int work_pair_of(int sk_iters, int num_pairs, long long i) {
    const long long S = sk_iters;
    return static_cast<int>(((i + 1) * num_pairs + S - 1) / S - 1);
}

// Which tiles of a launch are split (sk_first; sk_first == num_tiles: none). Three cases:
//  - A launch of between one and two waves (pairs < T, the second wave at most tail_pct %
//    full) is split entirely, provided each tile has at least min_blocks reduction blocks and
//    the operands (A rows of every tile row and B rows of every tile column, kb_tile blocks of
//    64 bf16 deep) fit in max_operand_bytes: the pairs of a wave no longer walk the reduction
//    in step, so the operands must stay in L2.
//  - A longer launch keeps its whole waves and splits only the last R = T mod P tiles, when
//    that is modelled to take under tail_gain of a round: the R tiles' work spread over all
//    pairs (R / P of a round) plus one read of their operand rows and columns from DRAM,
//    against a round of whole tiles. Their shares must be non-empty (R * kb_tile >= P).
//  - A launch of fewer tiles than pairs (a few hundred token rows) runs each tile's reduction
//    on `parts` = min(max_parts, pairs / T, kb_tile / min_part_blocks) pairs, T * parts pairs
//    in all, when parts >= 2 (shorter shares cost more in partial sums than they save):
//    every share then lies inside one tile, so a tile is summed from exactly `parts` partial
//    sums. Share j of every tile covers the same reduction blocks, so tiles that share an
//    operand read it in step, as whole tiles do, and no L2 limit applies.
// A round is 2 * 256 * 256 * 64 * kb_tile FLOP at pair_flops.
struct SplitPlan {
    int sk_first;
    int sk_iters;
    int pairs;   // pairs to launch when the plan says so (fewer tiles than pairs); 0: unchanged
};

struct SplitLaunch {
    int num_tiles, pairs, kb_tile;
    int m_blocks, n_blocks, group_m;
    int tile_rows, tile_cols;   // A rows per row block, B rows per column block
};

struct SplitRule {
    int tail_pct;               // whole split: the second wave at most this full
    int min_blocks;             // ... each tile has at least this many reduction blocks
    double max_operand_bytes;   // ... and the operands fit in this much L2
    double pair_flops;          // tail split: FLOP/s of one CTA pair
    double dram_Bps;            // ... DRAM bandwidth for the tail's operands
    double tail_gain;           // ... split when the modelled tail is below this share of a round
    int max_parts;              // fewer tiles than pairs: at most this many pairs per tile
    int min_part_blocks;        // ... each with at least this many reduction blocks
};

// The last `rem` tiles of a launch (kb_tile blocks deep, spanning `rows` distinct row blocks of
// tile_rows and `cols` distinct column blocks of tile_cols) are worth spreading over all `pairs`
// pairs when rem / pairs of a round plus one DRAM read of their operand rows and columns takes
// under tail_gain of a round of whole tiles, and every pair gets a non-empty share.
inline bool tail_split_pays(int rem, int kb_tile, int pairs, int rows, int cols, int tile_rows,
                            int tile_cols, const SplitRule& rule) {
    if (rem <= 0 || pairs <= 0 || kb_tile < rule.min_blocks) return false;
    if (static_cast<long long>(rem) * kb_tile < pairs) return false;
    const double block_bytes = static_cast<double>(kb_tile) * 64 * 2.0;  // one row, all K
    const double round_s = 2.0 * 256 * 256 * 64 * kb_tile / rule.pair_flops;
    const double tail_bytes =
        (static_cast<double>(rows) * tile_rows + static_cast<double>(cols) * tile_cols) * block_bytes;
    const double tail_s = round_s * rem / pairs + tail_bytes / rule.dram_Bps;
    return tail_s < rule.tail_gain * round_s;
}

inline SplitPlan plan_split_tiles(const SplitLaunch& L, const SplitRule& rule) {
    SplitPlan p{L.num_tiles, 0, 0};
    if (L.pairs <= 0 || L.num_tiles <= 0 || L.kb_tile < rule.min_blocks) return p;
    const int waves = L.num_tiles / L.pairs, rem = L.num_tiles % L.pairs;
    const double block_bytes = static_cast<double>(L.kb_tile) * 64 * 2.0;  // one row, all K
    if (waves == 0) {
        int parts = L.pairs / L.num_tiles;
        if (parts > rule.max_parts) parts = rule.max_parts;
        if (rule.min_part_blocks > 0 && parts > L.kb_tile / rule.min_part_blocks)
            parts = L.kb_tile / rule.min_part_blocks;
        if (parts < 2 || L.kb_tile < parts) return p;
        p.sk_first = 0;
        p.sk_iters = L.num_tiles * L.kb_tile;
        p.pairs = L.num_tiles * parts;
        return p;
    }
    if (rem == 0) return p;
    if (waves == 1) {
        if (rem * 100 > L.pairs * rule.tail_pct) return p;
        const double operand_bytes =
            (static_cast<double>(L.m_blocks) * L.tile_rows +
             static_cast<double>(L.n_blocks) * L.tile_cols) * block_bytes;
        if (operand_bytes > rule.max_operand_bytes) return p;
        p.sk_first = 0;
        p.sk_iters = L.num_tiles * L.kb_tile;
        return p;
    }
    // the distinct row and column blocks of the last rem tiles
    const int first = L.num_tiles - rem;
    int m_lo = 1 << 30, m_hi = -1, n_cnt = 0, n_prev = -1;
    for (int t = first; t < L.num_tiles; ++t) {
        int m, n;
        decode_tile_mn(L.group_m, L.m_blocks, L.n_blocks, t, m, n);
        m_lo = m < m_lo ? m : m_lo;
        m_hi = m > m_hi ? m : m_hi;
        if (n != n_prev) ++n_cnt;  // the tail walks whole columns of one row group
        n_prev = n;
    }
    if (!tail_split_pays(rem, L.kb_tile, L.pairs, m_hi - m_lo + 1, n_cnt, L.tile_rows, L.tile_cols,
                         rule))
        return p;
    p.sk_first = first;
    p.sk_iters = rem * L.kb_tile;
    return p;
}

// ---------------------------------------------------------------- tall units
//
// The second GEMM of a deep reduction runs most of its output as 512 x 256 tall units (two
// 256 x 256 halves sharing each B tile; GemmArgs::tall_units) over the whole 512-row blocks,
// tall_m_blocks = floor(M / 512) of them: as many whole waves of units as there are,
// `tall_units` = floor(T / P) * P of the T = tall_m_blocks * n_blocks. The launch's ordinary
// tiles then cover the rest, in this order:
//   tiles [0, tall_rest):  the 256-row halves of the remaining units (tall_rest = 2 (T -
//                          tall_units); tile t = half t % 2 of unit tall_units + t / 2);
//   tiles [tall_rest, ..): the 256-row blocks below the last whole 512 rows (0, 1 or 2 of
//                          them), column by column.
// They run as whole waves, then a last partial wave that may be split over all pairs as a tail.
// Tall units are used only when they take no more rounds of tiles than ordinary tiles alone
// (a unit counting two rounds).
struct TallPlan {
    int tall_units;     // 0: no tall units (launch the ordinary kernel)
    int tall_m_blocks;  // floor(M / 512)
    int tall_rest;      // ordinary tiles that are halves of the remaining units
    int tiles;          // all ordinary tiles after the units
    int tail_first;     // their last, partial wave: tiles [tail_first, tiles) ...
    int rows, cols;     // ... spanning this many 256-row and 256-column blocks
};

// The 256-row block and column block of ordinary tile t of a launch with tall units.
TPMLP_HD void decode_tall_rest(int group_m, int tall_m_blocks, int tall_units, int tall_rest,
                               int m_blocks, int n_blocks, int t, int& m_blk, int& n_blk) {
    if (t < tall_rest) {
        int tm;
        decode_tile_mn(group_m, tall_m_blocks, n_blocks, tall_units + (t >> 1), tm, n_blk);
        m_blk = 2 * tm + (t & 1);
    } else {
        const int left = m_blocks - 2 * tall_m_blocks;  // 1 or 2 row blocks below the units
        const int i = t - tall_rest;
        m_blk = 2 * tall_m_blocks + i % left;
        n_blk = i / left;
    }
}

inline TallPlan plan_tall_units(int M, int n_blocks, int group_m, int pairs) {
    TallPlan p{0, M / 512, 0, 0, 0, 0, 0};
    const int m_blocks = (M + 255) / 256;
    const int T = p.tall_m_blocks * n_blocks;
    if (pairs <= 0 || T < pairs) return p;
    const int units = T / pairs * pairs;
    const int rest = 2 * (T - units);
    const int tiles = rest + (m_blocks - 2 * p.tall_m_blocks) * n_blocks;
    const int rounds_tiles = (m_blocks * n_blocks + pairs - 1) / pairs;
    const int rounds_tall = 2 * units / pairs + (tiles + pairs - 1) / pairs;
    if (rounds_tall > rounds_tiles) return p;
    p.tall_units = units;
    p.tall_rest = rest;
    p.tiles = tiles;
    p.tail_first = tiles / pairs * pairs;
    int m_lo = 1 << 30, m_hi = -1, n_cnt = 0, n_prev = -1;
    for (int t = p.tail_first; t < p.tiles; ++t) {
        int m, n;
        decode_tall_rest(group_m, p.tall_m_blocks, p.tall_units, p.tall_rest, m_blocks, n_blocks,
                         t, m, n);
        m_lo = m < m_lo ? m : m_lo;
        m_hi = m > m_hi ? m : m_hi;
        if (n != n_prev) ++n_cnt;
        n_prev = n;
    }
    p.rows = m_hi >= m_lo ? m_hi - m_lo + 1 : 0;
    p.cols = n_cnt;
    return p;
}

// DRAM reads of a launch's tall units under a round model: each round of `pairs` units (and
// then the remaining units, whose halves run as tiles, as one more round) loads the union of
// its units' 512-row blocks of A and 256-column panels of B once, and L2 keeps nothing from
// one round to the next. Counted in B panels: a 512-row block of A is two of them. At 7b
// (16 x 16 units on 76 pairs) it gives the second GEMM's DRAM reads that ncu measured for
// row groups of 1, 2, 4 and 8, to the MB (0.856, 0.889, 0.856 and 0.931 GB).
inline long long tall_round_panels(int group_m, int tall_m_blocks, int n_blocks, int pairs) {
    const int T = tall_m_blocks * n_blocks;
    if (pairs <= 0 || T <= 0) return 0;
    const int units = T / pairs * pairs;
    std::vector<int> m_seen(tall_m_blocks, -1), n_seen(n_blocks, -1);
    long long total = 0;
    int round = -1, rows = 0, cols = 0;
    for (int u = 0; u < T; ++u) {
        const int r = u < units ? u / pairs : units / pairs;
        if (r != round) {
            total += 2LL * rows + cols;
            rows = cols = 0;
            round = r;
        }
        int m, n;
        decode_tile_mn(group_m, tall_m_blocks, n_blocks, u, m, n);
        if (m_seen[m] != r) {
            m_seen[m] = r;
            ++rows;
        }
        if (n_seen[n] != r) {
            n_seen[n] = r;
            ++cols;
        }
    }
    return total + 2LL * rows + cols;
}

// Row groups the tall units may sweep by (whole 512-row blocks), in order of preference.
constexpr int kTallGroups[5] = {8, 4, 16, 2, 1};

// The row group whose rounds read the least under tall_round_panels (the first of kTallGroups
// on a tie). Interleaved A/B with groups of 8, 4, 2 and 1 (bit-identical outputs): 7b 577.5,
// 575.1, 577.8 and 573.1 us per second GEMM, GPT-3 2596, 2610, 2633 and 2649 us, M = 16384
// at H = 4096 1174, 1171, 1177 and 1170 us, each within 1 % of the group this picks.
inline int pick_tall_group(int tall_m_blocks, int n_blocks, int pairs) {
    int best = kTallGroups[0];
    long long best_bytes = -1;
    for (int g : kTallGroups) {
        if (g > tall_m_blocks && g != kTallGroups[0]) continue;  // same order as the whole
        const long long b = tall_round_panels(g, tall_m_blocks, n_blocks, pairs);
        if (best_bytes < 0 || b < best_bytes) {
            best = g;
            best_bytes = b;
        }
    }
    return best;
}

// ---------------------------------------------------------------- device rates
//
//   gemm_flops  dense bf16 rate the GEMMs hold: SMs x 8192 FLOP per SM per clock (one
//               tcgen05 kind::f16 MMA of 128 x 256 x 16 per SM every 128 cycles) x the
//               maximum SM clock x kGemmClockShare, the share of that the GEMMs keep under
//               the board's power cap (a cuBLAS bf16 loop: 1.73 PFLOP/s over 152 SMs at a
//               2.07 GHz maximum, 0.67 of it);
//   dram_Bps    HBM bandwidth a stream of reads reaches: two transfers per memory clock x
//               the bus width x kDramShare (a device-to-device copy moves 6.75 TB/s against
//               the 8.18 TB/s this gives for 8192 bits at 3.996 GHz: 0.8);
//   copy_Bps    page-locked host <-> device copies per direction, with copies both ways at
//               once. No device attribute gives it: 168 GB/s, measured over NVLink-C2C with
//               16-128 MB copies (205 GB/s one way alone).
// An attribute the device does not report (0) takes the value of a GB300 (152 SMs, 2.07 GHz,
// 3.996 GHz x 8192 bits).
struct DeviceRates {
    double gemm_flops;
    double dram_Bps;
    double copy_Bps;
};

constexpr double kGemmFlopsPerSmClock = 8192.0;
constexpr double kGemmClockShare = 0.67;
constexpr double kDramShare = 0.8;
constexpr double kHostCopyBps = 168e9;

inline DeviceRates device_rates(int num_sms, double sm_clock_khz, double mem_clock_khz,
                                int mem_bus_bits) {
    if (num_sms <= 0) num_sms = 152;
    if (!(sm_clock_khz > 0)) sm_clock_khz = 2070000.0;
    if (!(mem_clock_khz > 0)) mem_clock_khz = 3996000.0;
    if (mem_bus_bits <= 0) mem_bus_bits = 8192;
    DeviceRates r;
    r.gemm_flops = num_sms * kGemmFlopsPerSmClock * sm_clock_khz * 1e3 * kGemmClockShare;
    r.dram_Bps = 2.0 * mem_clock_khz * 1e3 * (mem_bus_bits / 8.0) * kDramShare;
    r.copy_Bps = kHostCopyBps;
    return r;
}

// The split rule of a device with `pairs` CTA pairs (tpmlp_gemm_pair_kernel): the thresholds
// are the measured ones (see plan_split_tiles); the tail model's rates scale with the device.
inline SplitRule split_rule(const DeviceRates& r, int pairs) {
    SplitRule s{};
    s.tail_pct = 85;              // whole split: the second wave at most 85 % full
    s.min_blocks = 16;            // ... tiles at least 16 blocks deep
    s.max_operand_bytes = 64.0 * (1 << 20);  // ... operands within 64 MiB of L2
    s.pair_flops = r.gemm_flops / (pairs > 0 ? pairs : 1);
    s.dram_Bps = r.dram_Bps;
    s.tail_gain = 0.5;            // tail split: under half a round of whole tiles
    s.max_parts = 4;              // fewer tiles than pairs: at most 4 pairs per tile
    s.min_part_blocks = 32;       // ... of at least 32 blocks each
    return s;
}

struct ChunkGemm {
    int64_t tile_rows;   // token rows per output tile (256 on CTA pairs, 128 on one SM)
    int64_t col_tiles;   // output tiles per row block
    int64_t slots;       // tiles that run at once (resident CTA pairs or SMs)
    double tile_s;       // seconds per round of tiles
    double launch_s;     // fixed seconds per launch (set-up, first wave's ramp, last wave's drain)
};

// The fixed cost of one GEMM launch in the chunk model. Host-buffer forward passes timed with
// plans of at most 1, 2, 3 and 4 chunks were fastest with 3 chunks at GPT-3, 4 at 7b and 2 at
// GPT-2; without this cost the model preferred 4 chunks everywhere. Interleaved A/B of the
// planner with 0, 10 and 20 us: GPT-3 5.936 / 5.899 / 5.874 ms, 7b 1.405 / 1.391 / 1.409 ms,
// GPT-2 0.203 / 0.187 / 0.204 ms.
#ifndef TPMLP_CHUNK_LAUNCH_S
#define TPMLP_CHUNK_LAUNCH_S 10e-6
#endif
constexpr double kChunkLaunchS = TPMLP_CHUNK_LAUNCH_S;

struct ChunkModel {
    ChunkGemm g[2];
    double x_row_bytes, z_row_bytes;
    double copy_Bps;   // copy bandwidth per direction, with copies in and out running together
};

constexpr int64_t kChunkBlockRows = 256;

inline int64_t ceil_div_i64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Modelled seconds of a pass split into `n` chunks of rows[0..n).
inline double simulate_chunks(const ChunkModel& m, const int64_t* rows, int n) {
    double in = 0.0, comp = 0.0, out = 0.0;
    for (int i = 0; i < n; ++i) {
        in += static_cast<double>(rows[i]) * m.x_row_bytes / m.copy_Bps;
        double t = in > comp ? in : comp;
        for (const ChunkGemm& g : m.g) {
            const int64_t tiles = ceil_div_i64(rows[i], g.tile_rows) * g.col_tiles;
            t += static_cast<double>(ceil_div_i64(tiles, g.slots)) * g.tile_s + g.launch_s;
        }
        comp = t;
        out = (out > comp ? out : comp) + static_cast<double>(rows[i]) * m.z_row_bytes / m.copy_Bps;
    }
    return comp > out ? comp : out;
}

// Best split of M rows into at most max_chunks (<= 8) chunks whose sizes are multiples of
// `granule` blocks of 256 rows (the last chunk takes the remainder). The granule grows with M
// so that at most max_granules of them are enumerated. Writes the chunk row counts to rows[]
// and returns their number (>= 1; 0 rows -> 0 chunks).
inline int plan_chunks(const ChunkModel& m, int64_t M, int max_chunks, int64_t max_granules,
                       int64_t* rows) {
    if (M <= 0) return 0;
    if (max_chunks < 1) max_chunks = 1;
    if (max_chunks > 8) max_chunks = 8;
    const int64_t blocks = ceil_div_i64(M, kChunkBlockRows);
    const int64_t granule = ceil_div_i64(blocks, max_granules > 0 ? max_granules : 1);
    const int64_t G = ceil_div_i64(blocks, granule);  // granules; the last may be short
    auto rows_of = [&](int64_t g0, int64_t g1) {     // rows of granules [g0, g1)
        const int64_t r0 = g0 * granule * kChunkBlockRows;
        int64_t r1 = g1 * granule * kChunkBlockRows;
        if (r1 > M) r1 = M;
        return r1 - r0;
    };
    int best_n = 1;
    int64_t best_rows[8] = {M};
    double best_t = simulate_chunks(m, best_rows, 1);
    // enumerate cut points 0 < c_1 < ... < c_{n-1} < G in granules
    int64_t cut[8];
    int64_t cand[8];
    for (int n = 2; n <= max_chunks && n <= G; ++n) {
        for (int i = 0; i < n - 1; ++i) cut[i] = i + 1;
        for (;;) {
            int64_t prev = 0;
            for (int i = 0; i < n - 1; ++i) {
                cand[i] = rows_of(prev, cut[i]);
                prev = cut[i];
            }
            cand[n - 1] = rows_of(prev, G);
            const double t = simulate_chunks(m, cand, n);
            if (t < best_t * (1.0 - 1e-9)) {  // ties keep the earlier (fewer chunks) plan
                best_t = t;
                best_n = n;
                for (int i = 0; i < n; ++i) best_rows[i] = cand[i];
            }
            // next combination of n - 1 cuts from {1 .. G-1}
            int i = n - 2;
            while (i >= 0 && cut[i] == G - 1 - (n - 2 - i)) --i;
            if (i < 0) break;
            ++cut[i];
            for (int j = i + 1; j < n - 1; ++j) cut[j] = cut[j - 1] + 1;
        }
    }
    for (int i = 0; i < best_n; ++i) rows[i] = best_rows[i];
    return best_n;
}

}  // namespace tpmlp
