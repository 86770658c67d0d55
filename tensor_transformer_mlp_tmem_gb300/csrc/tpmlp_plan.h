// Work planning shared by the host code, the GEMM kernels and the host tests (plain C++; the
// host tests build it with g++ alone):
//   1. the split reduction's plan and the CTA-pair kernel's walk over its work units;
//   2. the row-chunk planner of the host-buffer forward pass.
//
// ---------------------------------------------------------------- 1. split reduction
//
// A CTA-pair launch of T output tiles, each reduced over kb_tile blocks of 64, on P resident
// pairs. Tiles [0, sk_first) are whole units, handed out round robin (pair p: p, p + P, ...).
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
//   comp_c = max(comp_{c-1}, in_c) + sum over both GEMMs of rounds(chunk c) * round time
//   out_c  = max(out_{c-1}, comp_c) + Z bytes of chunk c / bandwidth out
// and the pass ends at max(comp_last, out_last).
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define TPMLP_HD __host__ __device__ __forceinline__
#else
#define TPMLP_HD inline
#endif

namespace tpmlp {

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

// Which tiles of a launch are split (sk_first; sk_first == num_tiles: none). A launch of between
// one and two waves (pairs < T, and the second wave at most tail_pct % full) is split
// entirely, provided each tile has at least min_blocks reduction blocks and the operands
// (A rows and B rows of every tile row and column, kb_tile blocks of 64 bf16 deep) fit in
// max_operand_bytes. Longer launches keep whole tiles.
struct SplitPlan {
    int sk_first;
    int sk_iters;
};

inline SplitPlan plan_split_tiles(int num_tiles, int pairs, int kb_tile, int m_blocks, int n_blocks,
                                  int tile_rows, int tail_pct, int min_blocks,
                                  double max_operand_bytes) {
    SplitPlan p{num_tiles, 0};
    if (pairs <= 0 || kb_tile <= 0) return p;
    const int waves = num_tiles / pairs, rem = num_tiles % pairs;
    if (waves != 1 || rem == 0 || rem * 100 > pairs * tail_pct) return p;
    const double operand_bytes =
        static_cast<double>(m_blocks + n_blocks) * tile_rows * kb_tile * 64 * 2.0;
    if (kb_tile < min_blocks || operand_bytes > max_operand_bytes) return p;
    p.sk_first = 0;
    p.sk_iters = num_tiles * kb_tile;
    return p;
}

struct ChunkGemm {
    int64_t tile_rows;   // token rows per output tile (256 on CTA pairs, 128 on one SM)
    int64_t col_tiles;   // output tiles per row block
    int64_t slots;       // tiles that run at once (resident CTA pairs or SMs)
    double tile_s;       // seconds per round of tiles
};

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
            t += static_cast<double>(ceil_div_i64(tiles, g.slots)) * g.tile_s;
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
