// Row-chunk planner of the host-buffer forward pass (plain C++, no CUDA: the host tests build
// it alone).
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

namespace tpmlp {

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
