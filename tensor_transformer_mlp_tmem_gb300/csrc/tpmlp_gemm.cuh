// The two GEMMs of the tensor-parallel MLP block, as one persistent, warp-specialised
// sm_103a kernel template:
//
//   GEMM1 (column-parallel layer, every shard i):  Y[:, i f + j] = GeLU(X W1_i + b1_i)[:, j]
//   GEMM2 (row-parallel layer + the sum over shards): Z = b2 + sum_i Y_i W2_i
//
// (千亿参数模型如何拆分到多张GPU上训练, "方案一"/"方案二"; 大模型分布式并行策略详解 §4.1.)
//
// Per CTA (one per SM, looping over output tiles of kBM x BN):
//   warp 0      TMA producer: streams kBM x 64 tiles of A and BN x 64 tiles of B (both
//               K-major, 128-byte swizzled) into a STAGES-deep shared-memory ring.
//   warp 1      allocates tensor memory (2 x BN fp32 columns: two accumulators) and, from
//               one lane, issues tcgen05.mma (M = 128, N = BN, K = 16 per instruction).
//   warps 2..   epilogue (4 or 8 warps): tcgen05.ld of the finished accumulator (each warp
//               owns the 32 TMEM lanes = output rows its warp rank may access; with 8 warps
//               two share a lane quadrant and split its columns), bias, GeLU (GEMM1),
//               conversion and stores. The accumulator is handed back to the MMA warp as
//               soon as it has been read, so the next tile's MMAs overlap this epilogue.
//
// GEMM2's reduction runs shard-major: shard 0's f/64 blocks, then shard 1's, ... all into
// the SAME fp32 accumulator. That accumulation is the on-chip replacement for the pages'
// All-Reduce of the k partial outputs (AI大模型分布式训练 §2.2 sums the RowParallelLinear
// partials with dist.all_reduce): no partial ever leaves tensor memory.
//
// Every wait is bounded (see ptx::mbar_wait); a CTA that gives up records a code in the
// device status word, drains its in-flight copies and MMAs, frees its tensor memory and
// returns.
#pragma once

#include <cuda_bf16.h>

#include "sm103_ptx.cuh"
#include "tpmlp_plan.h"

namespace tpmlp {

constexpr int kBM = 128;        // output rows per tile = TMEM lanes
constexpr int kBK = 64;         // reduction depth per stage: one 128-byte swizzle row of bf16
constexpr int kUmmaK = 16;      // reduction depth of one kind::f16 MMA
// Epilogue warps: 4 (one per TMEM lane quadrant) or 8 (two per quadrant, each draining half
// of the accumulator's columns).
#ifndef TPMLP_EPI_WARPS
#define TPMLP_EPI_WARPS 8
#endif
constexpr int kEpiWarps = TPMLP_EPI_WARPS;
constexpr int kEpiParts = kEpiWarps / 4;  // column parts per lane quadrant
constexpr int kNumThreads = 64 + 32 * kEpiWarps;
static_assert(kEpiWarps == 4 || kEpiWarps == 8, "epilogue warps");

// kGemm1: Y = GeLU(acc + b1).  kGemm1Gated: the accumulator's column halves hold the gate and
// the up projection of the same outputs, Y = SiLU(gate + bg) * (up + bu).  kGemm2: Z = acc + b2.
// kGemm2Residual: Z = R + (acc + b2), R the layer's input (the residual add after the block).
// kGemm1Linear: the column-parallel tiling of kGemm1 without the activation (out = acc + b).
// Backward: kGemm1Train writes Y = GeLU(acc + b1) and the pre-activation A = acc + b1;
// kBwdDA: dA = acc * GeLU'(A) (aux = the saved A); kWeightGrad: plain fp32 acc (no bias), with
// both operands M-contiguous (the reduction runs over tokens).
// Gated backward: kGemm1GatedTrain is kGemm1Gated that also writes the pre-activations
// G = gate + bg and U = up + bu (bf16) to out2; kBwdGated takes acc = dY and the saved G, U
// (aux) and writes dG = dY U SiLU'(G) and dU = dY SiLU(G).
enum class Mode : int {
    kGemm1 = 1, kGemm2 = 2, kGemm1Gated = 3, kGemm2Residual = 4, kGemm1Linear = 5,
    kGemm1Train = 6, kBwdDA = 7, kWeightGrad = 8, kGemm1GatedTrain = 9, kBwdGated = 10
};

// Modes whose B operand is the column-sharded weight (tiles inside one shard, K = H).
__host__ __device__ constexpr bool is_gemm1(Mode m) {
    return m == Mode::kGemm1 || m == Mode::kGemm1Gated || m == Mode::kGemm1Linear ||
           m == Mode::kGemm1Train || m == Mode::kBwdDA || m == Mode::kGemm1GatedTrain ||
           m == Mode::kBwdGated;
}

// Modes whose accumulator holds the gate and up projections of the same outputs.
__host__ __device__ constexpr bool is_gated(Mode m) {
    return m == Mode::kGemm1Gated || m == Mode::kGemm1GatedTrain;
}

// Modes that add a bias in the epilogue.
__host__ __device__ constexpr bool has_bias(Mode m) {
    return m != Mode::kBwdDA && m != Mode::kWeightGrad && m != Mode::kBwdGated;
}

// Wait sites recorded in the status word when a bounded wait gives up: (mode << 8) | site.
enum : int {
    kSiteProducer = 1, kSiteMmaAccum = 2, kSiteMmaFull = 3, kSiteEpilogue = 4, kSiteSplitCount = 5
};

struct GemmArgs {
    int M;          // valid output rows (token rows)
    int ldo;        // output columns = row pitch of `out` in elements
    int f;          // shard width
    int k;          // shard count
    int kb_tile;    // 64-deep reduction blocks per output tile
    int kb_shard;   // 64-deep reduction blocks per shard (GEMM2)
    int m_blocks;   // ceil(M / kBM)
    int n_blocks;   // ldo / BN
    int num_tiles;  // m_blocks * n_blocks
    int group_m;    // tile rasterisation: this many row blocks share a column sweep
    const float* bias;  // [ldo] fp32
    void* out;          // [M][ldo] bf16 or fp32
    const void* residual;  // kGemm2Residual: [M][ldo] bf16 added to the output (may equal out);
                           // kBwdDA: the saved pre-activation A [M][ldo] bf16
    void* out2;            // kGemm1Train: the pre-activation A [M][ldo] bf16;
                           // kGemm1GatedTrain: G and U [M][ldo2] bf16 (U at column half + j)
    int ldo2;              // row pitch of out2 in elements (kGemm1GatedTrain)
    int half;              // kGemm1GatedTrain: U's column offset in out2; kBwdGated: dU's and
                           // U's column offset in out and residual (both of row pitch ldo)
    int k2;                // second-GEMM reduction: shards [0, k2) read B from the first map,
                           // shards [k2, k) from the second (shard index i - k2); k2 = k: one map
    int* status;        // device status word
    // Split reduction (CTA-pair kernel only; tpmlp_plan.h). Tiles [0, sk_first) are whole
    // units handed out round robin; the sk_iters = (num_tiles - sk_first) * kb_tile reduction
    // blocks of the remaining tiles are divided evenly among the pairs, in tile order. Every
    // pair holding part of a split tile writes its fp32 partial sum to one of its two slots
    // and counts itself in; the last to arrive sums all of them, in pair order, and runs the
    // epilogue. Nothing waits on another CTA.
    int sk_first;          // == num_tiles: no split
    int sk_iters;
    float* sk_partial;     // [pairs][2: first / last unit][2 CTAs][256 columns][128 rows] fp32
    uint32_t* sk_count;    // [split tiles][2 CTAs][epilogue warps] epoch-tagged arrivals
    uint32_t sk_epoch;     // new for every launch that splits
    int b_blocked;         // CTA-pair second GEMM: B is the packed operand in 16 KB blocks
                           // (2-D map of 128-byte rows; see transpose_blocked_bf16_kernel)
    // Tall units (CTA-pair kernel, TALL instantiation): the whole 512-row blocks of the output,
    // tall_m_blocks = floor(M / 512) of them, are also cut into 512 x 256 units of two 256-row
    // halves, numbered like tiles. Units [0, tall_units) are computed whole, round robin over
    // the pairs; the tiles of the launch (num_tiles, sk_*) then cover the rest: the halves of
    // the remaining units (tiles [0, tall_rest)) and the row blocks below the last whole 512
    // rows (tpmlp_plan.h, decode_tall_rest).
    int tall_units;        // 0: no tall units
    int tall_m_blocks;
    int tall_rest;
    // 1: a unit of an odd round (unit / pairs odd) sweeps its reduction blocks from the last
    // to the first, so that it starts on the operand blocks the round before it loaded last,
    // which are still in L2. Its sums then run in the opposite order (last bits may differ).
    int tall_serpentine;
};

constexpr int kSkSlotFloats = 128 * 256;  // one CTA's half of a 256 x 256 accumulator

// The accumulator columns one epilogue warp drains, 32 at a time: [c0, c0 + kCols) with
// c0 = part * kCols, and in the gated layer also the same columns of the up half (+ G).
template <Mode MODE, int WIDTH, typename Fn>
__device__ __forceinline__ void for_each_warp_slice(int part, Fn&& fn) {
    if constexpr (is_gated(MODE)) {
        constexpr int G = WIDTH / 2, kCols = G / kEpiParts;
#pragma unroll 1
        for (int c = part * kCols; c < (part + 1) * kCols; c += 32) {
            fn(c);
            fn(G + c);
        }
    } else {
        constexpr int kCols = WIDTH / kEpiParts;
#pragma unroll 1
        for (int c = part * kCols; c < (part + 1) * kCols; c += 32) fn(c);
    }
}

// Split units. A slot holds one CTA's 128 accumulator rows x 256 columns in groups of four
// columns: element (r, c) at (c / 4) * 512 + r * 4 + c % 4, so that each lane moves 16 bytes
// per access and a warp's 32 lanes cover 512 contiguous bytes. Pair p's slots: p * 2 + 0 for
// the unit that starts its share inside a tile, p * 2 + 1 for the unit that holds a tile's
// first blocks (a pair has at most one of each).
__device__ __forceinline__ float* split_slot(float* partial, int pair, int which, uint32_t rank) {
    return partial + ((static_cast<size_t>(pair) * 2 + which) * 2 + rank) * kSkSlotFloats;
}

__device__ __forceinline__ size_t slot_index(int c, int lrow) {
    return static_cast<size_t>(c >> 2) * 512 + static_cast<size_t>(lrow) * 4 + (c & 3);
}

// This warp's share of its accumulator -> its slot.
template <Mode MODE, int WIDTH>
__device__ __forceinline__ void save_partial(uint32_t taddr, int part, float* slot, int lrow) {
    for_each_warp_slice<MODE, WIDTH>(part, [&](int c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + c, v);
        ptx::tmem_wait_ld(v);
#pragma unroll
        for (int g = 0; g < 8; ++g)
            __stcg(reinterpret_cast<float4*>(slot + slot_index(c + 4 * g, lrow)),
                   make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                               __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3])));
    });
}

// The first pair's finish: its own part (the first in pair order) plus the partials of pairs
// p_first + 1 .. p_last (slot 0 each), added in that order into its accumulator.
template <Mode MODE, int WIDTH>
__device__ __forceinline__ void fold_partials(uint32_t taddr, int part, float* partial,
                                              uint32_t rank, int p_first, int p_last, int lrow) {
    for_each_warp_slice<MODE, WIDTH>(part, [&](int c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + c, v);
        ptx::tmem_wait_ld(v);
#pragma unroll 1
        for (int p = p_first + 1; p <= p_last; ++p) {
            const float* slot = split_slot(partial, p, 0, rank);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const float4 q = __ldcg(reinterpret_cast<const float4*>(slot + slot_index(c + 4 * g, lrow)));
                v[4 * g] = __float_as_uint(__uint_as_float(v[4 * g]) + q.x);
                v[4 * g + 1] = __float_as_uint(__uint_as_float(v[4 * g + 1]) + q.y);
                v[4 * g + 2] = __float_as_uint(__uint_as_float(v[4 * g + 2]) + q.z);
                v[4 * g + 3] = __float_as_uint(__uint_as_float(v[4 * g + 3]) + q.w);
            }
        }
        ptx::tmem_st_32x32b_x32_wait(taddr + c, v);
    });
}

// Any other pair's finish (the first pair handed the tile over): the same sum in pair order
// p_first .. p_last (the first pair's part from its slot 1, the others' from slot 0, this
// pair's own from its accumulator), written back into this warp's share of the accumulator,
// 16 columns at a time (three arrays of them are live).
template <Mode MODE, int WIDTH>
__device__ __forceinline__ void reduce_partials(uint32_t taddr, int part, float* partial,
                                                uint32_t rank, int p_first, int p_last, int self,
                                                int lrow) {
    for_each_warp_slice<MODE, WIDTH>(part, [&](int c) {
#pragma unroll 1
        for (int h = c; h < c + 32; h += 16) {
            uint32_t own[16];
            float sum[16];
            ptx::tmem_ld_32x32b_x16_wait(taddr + h, own);
#pragma unroll 1
            for (int p = p_first; p <= p_last; ++p) {
                float x[16];
                if (p == self) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) x[j] = __uint_as_float(own[j]);
                } else {
                    const float* slot = split_slot(partial, p, p == p_first ? 1 : 0, rank);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const float4 q = __ldcg(reinterpret_cast<const float4*>(slot + slot_index(h + 4 * g, lrow)));
                        x[4 * g] = q.x;
                        x[4 * g + 1] = q.y;
                        x[4 * g + 2] = q.z;
                        x[4 * g + 3] = q.w;
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) sum[j] = p == p_first ? x[j] : sum[j] + x[j];
            }
            uint32_t out[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) out[j] = __float_as_uint(sum[j]);
            ptx::tmem_st_32x32b_x16_wait(taddr + h, out);
        }
    });
}

// Shared-memory matrix descriptor for a K-major operand tile stored as rows of 64 bf16
// (128 bytes) with the 128-byte swizzle, 8-row swizzle atoms 1024 bytes apart (the layout
// TMA writes with CU_TENSOR_MAP_SWIZZLE_128B and a 64-element inner box).
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4 (not used for swizzled K-major; 1)
//   bits 32-45  stride-dimension byte offset >> 4 (1024 B between 8-row groups)
//   bits 46-47  descriptor version (1 for tcgen05)
//   bits 49-51  base offset (0: atoms are 1024-byte aligned)
//   bits 61-63  swizzle mode (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Descriptor for an MN-major operand tile (M- or N-index contiguous): TMA boxes of 64 (MN)
// x 64 (K) bf16, each 8 KB, placed one after another along MN. In a box a K row is 128 bytes
// of 64 consecutive MN elements, 128-byte swizzled in groups of 8 rows.
//   leading-dimension byte offset: 8192 B between consecutive 64-wide MN blocks
//   stride-dimension byte offset:  1024 B between consecutive 8-row K groups
__device__ __forceinline__ uint64_t sdesc_mn128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
           (static_cast<uint64_t>(8192 >> 4) << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
           (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9 and
// 10-12 = 1), A / B major-ness in bits 15 / 16 (0 = K-major, 1 = MN-major), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool mn_major = false) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (mn_major ? (1u << 15) | (1u << 16) : 0u) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

template <int BN, int STAGES>
struct GemmSmem {
    static constexpr uint32_t kABytes = kBM * kBK * 2;
    static constexpr uint32_t kBBytes = BN * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kCtrlBytes = 8 * (2 * STAGES + 5) + 8;
    static constexpr uint32_t kEpiOffset = STAGES * kStageBytes + (kCtrlBytes + 127) / 128 * 128;
    static constexpr uint32_t kTotal = 1024 /*alignment slack*/ + kEpiOffset + kEpiWarps * 2048;  // + epilogue staging
    static_assert(kTotal <= 232448, "dynamic shared memory per CTA");
    static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators; power of two >= 32
};

// 2^x and 1/x on the special-function unit (PTX ex2.approx.ftz.f32: relative error near
// 2^-22; rcp.approx.ftz.f32: within one ulp).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Standard normal lower tail Phi(-|a|) = erfc(|a| / sqrt 2) / 2 without a branch, in the form
// erfc(z) = t exp(-z^2 + P(t)), t = 1 / (1 + z/2) (Press et al., Numerical Recipes in C,
// 2nd ed., section 6.2), with a degree-7 P refitted to minimax relative error and carried to
// base 2 with the factor 1/2 folded in (fit_phi.py writes the coefficients):
//   Phi(-|a|) = t * 2^(P2(t) - a^2 log2(e) / 2).
// Relative error below 1e-5 over the fp32 range, more than two orders of magnitude under a
// bf16 step. normal_tail_t gives t, normal_tail_exp the power of two.
constexpr int kPhiDegree = 7;
// P2's coefficients, highest degree first.
__device__ constexpr float kPhiP2[kPhiDegree + 1] = {
    -2.294616550e-01f, 9.304409623e-01f, -1.215087414e+00f, 3.299344182e-01f,
    1.498845778e-02f, 5.527308583e-01f, 1.442202449e+00f, -2.825744629e+00f};
constexpr float kHalfLog2e = 0.72134752044448170f;  // log2(e) / 2

__device__ __forceinline__ float normal_tail_t(float a) {
    return rcp_approx(fmaf(fabsf(a), 0.35355339059327376f, 1.0f));
}
__device__ __forceinline__ float normal_tail_exp(float a, float t) {
    float p = kPhiP2[0];
#pragma unroll
    for (int i = 1; i <= kPhiDegree; ++i) p = fmaf(p, t, kPhiP2[i]);
    return ex2_approx(fmaf(a * a, -kHalfLog2e, p));
}
__device__ __forceinline__ float normal_lower_tail(float a) {
    const float t = normal_tail_t(a);
    return t * normal_tail_exp(a, t);
}

// Packed fp32x2 arithmetic: two IEEE fp32 operations per instruction, each half rounded
// exactly like the scalar operation.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_splat(float v) { return f2_pack(v, v); }

// GeLU in its erf form, a * Phi(a) = a/2 * (1 + erf(a / sqrt 2)), written through the lower
// tail as max(a, 0) - |a| Phi(-|a|) (for a >= 0 by Phi(a) = 1 - Phi(-a)): no select, and the
// tail's factor t is multiplied into |a| before the power of two. Two values at a time: the
// polynomial and the exponent run as packed fp32x2 operations, the reciprocal, exp2, |a| t
// and the max per value, so the results equal those of the scalar formula bit for bit.
// Per value about ten instructions, bias add excluded (the epilogue is bound by instruction
// issue at short reductions).
__device__ __forceinline__ void gelu_erf2(float& a0, float& a1) {
    const float t0 = normal_tail_t(a0), t1 = normal_tail_t(a1);
    const uint64_t T = f2_pack(t0, t1);
    uint64_t P = f2_splat(kPhiP2[0]);
#pragma unroll
    for (int i = 1; i <= kPhiDegree; ++i) P = f2_fma(P, T, f2_splat(kPhiP2[i]));
    const uint64_t A = f2_pack(a0, a1);
    float e0, e1;
    f2_unpack(f2_fma(f2_mul(A, A), f2_splat(-kHalfLog2e), P), e0, e1);
    const uint64_t X = f2_pack(ex2_approx(e0), ex2_approx(e1));
    const uint64_t S = f2_pack(-(fabsf(a0) * t0), -(fabsf(a1) * t1));
    f2_unpack(f2_fma(S, X, f2_pack(fmaxf(a0, 0.0f), fmaxf(a1, 0.0f))), a0, a1);
}

// GeLU'(a) = Phi(a) + a phi(a), phi(a) = 2^(-a^2 log2(e) / 2) / sqrt(2 pi) the normal density.
__device__ __forceinline__ float gelu_grad(float a) {
    const float q = normal_lower_tail(a);
    return (a < 0.0f ? q : 1.0f - q) +
           a * 0.39894228040143267794f * ex2_approx(a * a * -kHalfLog2e);
}

// SiLU(a) = a * sigma(a) = a / (1 + e^-a) = a * 1 / (1 + 2^(-a log2 e)).
__device__ __forceinline__ float silu(float a) {
    return a * rcp_approx(1.0f + ex2_approx(a * -1.44269504088896341f));
}

// SiLU(g) * u on two values at once, bit-identical to the scalar silu(g) * u: the products and
// the sum run as packed fp32x2 operations, exp2 and the reciprocal per value.
__device__ __forceinline__ void swiglu2(float& g0, float& g1, float u0, float u1) {
    const uint64_t G = f2_pack(g0, g1);
    float e0, e1;
    f2_unpack(f2_mul(G, f2_splat(-1.44269504088896341f)), e0, e1);
    float d0, d1;
    f2_unpack(f2_add(f2_splat(1.0f), f2_pack(ex2_approx(e0), ex2_approx(e1))), d0, d1);
    const uint64_t S = f2_mul(G, f2_pack(rcp_approx(d0), rcp_approx(d1)));
    f2_unpack(f2_mul(S, f2_pack(u0, u1)), g0, g1);
}

// SiLU'(a) = sigma(a) (1 + a (1 - sigma(a))).
__device__ __forceinline__ float silu_grad(float a) {
    const float s = rcp_approx(1.0f + ex2_approx(a * -1.44269504088896341f));
    return s * fmaf(a, 1.0f - s, 1.0f);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&p);
}

// Per-warp shared-memory staging for bf16 output slices (32 rows x 32 columns = 2 KB).
constexpr uint32_t kStageSliceBytes = 32 * 64;

// Store a warp's 32 rows x 32 bf16 columns (lane i holds row row0 + i as 16 packed words)
// through the warp's 2 KB staging buffer, so that each global store writes eight whole
// 64-byte row segments (four lanes per row) instead of 32 scattered 16-byte pieces. In the
// buffer, 16-byte chunk c of row r sits at position c ^ ((r >> 1) & 3): both the row-wise
// writes and the segment-wise reads touch 32 distinct banks per quarter warp.
__device__ __forceinline__ void store_rows_coalesced(const uint32_t (&p)[16], uint32_t stage,
                                                     __nv_bfloat16* out, int row0, int M, int ldo,
                                                     int col) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t a = stage + lane * 64 + 16 * (c ^ ((lane >> 1) & 3));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(p[4 * c]),
                     "r"(p[4 * c + 1]), "r"(p[4 * c + 2]), "r"(p[4 * c + 3])
                     : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = 8 * j + (lane >> 2), c = lane & 3;
        const uint32_t a = stage + r * 64 + 16 * (c ^ ((r >> 1) & 3));
        uint4 v;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(a)
                     : "memory");
        if (row0 + r < M)
            *reinterpret_cast<uint4*>(out + static_cast<size_t>(row0 + r) * ldo + col + 8 * c) = v;
    }
    __syncwarp();  // the buffer is free again
}

__device__ __forceinline__ void pack_slice(const float (&x)[32], uint32_t (&p)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
}

// One 32-column slice of the warp's 32 output rows (this lane: `row`): + bias, (GeLU),
// (+ residual), convert, store. All lanes of the warp call it together.
template <Mode MODE, bool OUT_F32>
__device__ __forceinline__ void epilogue_slice(const uint32_t (&v)[32], const float* __restrict__ bias,
                                               void* out, int row, int M, int ldo, int col,
                                               const void* residual, void* out2, uint32_t stage) {
    const int row0 = row - static_cast<int>(threadIdx.x & 31);
    float x[32];
    if constexpr (!has_bias(MODE)) {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);  // no bias
    } else {
        const float4* b4 = reinterpret_cast<const float4*>(bias + col);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 bb = __ldg(b4 + j);
            f2_unpack(f2_add(f2_pack(__uint_as_float(v[4 * j + 0]), __uint_as_float(v[4 * j + 1])),
                             f2_pack(bb.x, bb.y)),
                      x[4 * j + 0], x[4 * j + 1]);
            f2_unpack(f2_add(f2_pack(__uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])),
                             f2_pack(bb.z, bb.w)),
                      x[4 * j + 2], x[4 * j + 3]);
        }
    }
    if constexpr (MODE == Mode::kGemm1Train) {
        // save the pre-activation for the backward pass, then apply GeLU
        uint32_t p[16];
        pack_slice(x, p);
        store_rows_coalesced(p, stage, static_cast<__nv_bfloat16*>(out2), row0, M, ldo, col);
    }
    if constexpr (MODE == Mode::kGemm1 || MODE == Mode::kGemm1Train) {
#pragma unroll
        for (int j = 0; j < 16; ++j) gelu_erf2(x[2 * j], x[2 * j + 1]);
    }
    if constexpr (MODE == Mode::kBwdDA) {
        // dA = dY * GeLU'(A), A the saved (bf16) pre-activation
        if (row < M) {
            const uint4* a4 = reinterpret_cast<const uint4*>(
                static_cast<const __nv_bfloat16*>(residual) + static_cast<size_t>(row) * ldo + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 u = a4[j];
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    x[8 * j + 2 * i] *= gelu_grad(__uint_as_float(w[i] << 16));
                    x[8 * j + 2 * i + 1] *= gelu_grad(__uint_as_float(w[i] & 0xFFFF0000u));
                }
            }
        }
    }
    if constexpr (MODE == Mode::kGemm2Residual) {
        // read before the store below: the output may be the residual buffer itself
        if (row < M) {
            const uint4* r4 = reinterpret_cast<const uint4*>(
                static_cast<const __nv_bfloat16*>(residual) + static_cast<size_t>(row) * ldo + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 u = r4[j];
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    x[8 * j + 2 * i] += __uint_as_float(w[i] << 16);
                    x[8 * j + 2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
                }
            }
        }
        // every lane of the warp has read its residual row before any lane stores below
        __syncwarp();
    }
    if constexpr (OUT_F32) {
        if (row < M) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) +
                                                    static_cast<size_t>(row) * ldo + col);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
        }
    } else {
        uint32_t p[16];
        pack_slice(x, p);
        store_rows_coalesced(p, stage, static_cast<__nv_bfloat16*>(out), row0, M, ldo, col);
    }
}

// One 32-column slice of the warp's 32 output rows of the gated first layer: the gate values g
// and the up values u of the same 32 outputs; Y = SiLU(g + bias_g) * (u + bias_u), bf16.
// TRAIN: also keep the pre-activations for the backward pass, G = g + bias_g at out2[row][col]
// and U = u + bias_u at out2[row][half + col] (bf16, row pitch ldo2).
template <bool TRAIN>
__device__ __forceinline__ void epilogue_gated_slice(const uint32_t (&g)[32], const uint32_t (&u)[32],
                                                     const float* __restrict__ bias_g,
                                                     const float* __restrict__ bias_u,
                                                     const GemmArgs& args, int row, int col,
                                                     uint32_t stage) {
    const int row0 = row - static_cast<int>(threadIdx.x & 31);
    float gv[32], uv[32];
    const float4* bg4 = reinterpret_cast<const float4*>(bias_g);
    const float4* bu4 = reinterpret_cast<const float4*>(bias_u);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 bg = __ldg(bg4 + j);
        const float4 bu = __ldg(bu4 + j);
        const float bgv[4] = {bg.x, bg.y, bg.z, bg.w}, buv[4] = {bu.x, bu.y, bu.z, bu.w};
#pragma unroll
        for (int h = 0; h < 4; h += 2) {
            const int e = 4 * j + h;
            f2_unpack(f2_add(f2_pack(__uint_as_float(g[e]), __uint_as_float(g[e + 1])),
                             f2_pack(bgv[h], bgv[h + 1])),
                      gv[e], gv[e + 1]);
            f2_unpack(f2_add(f2_pack(__uint_as_float(u[e]), __uint_as_float(u[e + 1])),
                             f2_pack(buv[h], buv[h + 1])),
                      uv[e], uv[e + 1]);
        }
    }
    uint32_t p[16];
    if constexpr (TRAIN) {
        __nv_bfloat16* a_save = static_cast<__nv_bfloat16*>(args.out2);
        pack_slice(gv, p);
        store_rows_coalesced(p, stage, a_save, row0, args.M, args.ldo2, col);
        pack_slice(uv, p);
        store_rows_coalesced(p, stage, a_save, row0, args.M, args.ldo2, args.half + col);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) swiglu2(gv[2 * j], gv[2 * j + 1], uv[2 * j], uv[2 * j + 1]);
    pack_slice(gv, p);
    store_rows_coalesced(p, stage, static_cast<__nv_bfloat16*>(args.out), row0, args.M, args.ldo,
                         col);
}

// One 32-column slice of the gated backward's first GEMM: v = dY for outputs [col, col + 32)
// of this lane's row; G and U from the saved pre-activations (aux[row][col], aux[row][half +
// col], row pitch ldo). Writes dG = dY U SiLU'(G) to out[row][col] and dU = dY SiLU(G) to
// out[row][half + col] (bf16, row pitch ldo).
__device__ __forceinline__ void epilogue_bwd_gated_slice(const uint32_t (&v)[32], const GemmArgs& args,
                                                         int row, int col, uint32_t stage) {
    const int row0 = row - static_cast<int>(threadIdx.x & 31);
    float dg[32], du[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) dg[j] = du[j] = __uint_as_float(v[j]);
    if (row < args.M) {
        const __nv_bfloat16* aux = static_cast<const __nv_bfloat16*>(args.residual) +
                                   static_cast<size_t>(row) * args.ldo + col;
        const uint4* g4 = reinterpret_cast<const uint4*>(aux);
        const uint4* u4 = reinterpret_cast<const uint4*>(aux + args.half);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 gq = g4[j], uq = u4[j];
            const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
            const uint32_t uw[4] = {uq.x, uq.y, uq.z, uq.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int e = 8 * j + 2 * i + h;
                    const float gg = __uint_as_float(h ? (gw[i] & 0xFFFF0000u) : (gw[i] << 16));
                    const float uu = __uint_as_float(h ? (uw[i] & 0xFFFF0000u) : (uw[i] << 16));
                    du[e] *= silu(gg);
                    dg[e] *= uu * silu_grad(gg);
                }
            }
        }
    }
    uint32_t p[16];
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
    pack_slice(dg, p);
    store_rows_coalesced(p, stage, out, row0, args.M, args.ldo, col);
    pack_slice(du, p);
    store_rows_coalesced(p, stage, out, row0, args.M, args.ldo, args.half + col);
}

// Drain the accumulator columns [base, base + width) of this warp's 32 rows through the
// epilogue. Releases the accumulator (arrive on `release_bar`, via `arrive`) once the last
// columns are in registers. n0 is the tile's first column in B-row space; for the gated
// layer the first half of the columns is the gate and the second half the up projection of
// outputs [n0 / 2, n0 / 2 + width / 2).
// `part` (0 .. kEpiParts-1) selects which share of the columns this warp drains.
template <Mode MODE, bool OUT_F32, int WIDTH, typename Release>
__device__ __forceinline__ void drain_accumulator(uint32_t taddr, const GemmArgs& args, int row,
                                                  int n0, int part, uint32_t stage,
                                                  Release release) {
    if constexpr (is_gated(MODE)) {
        constexpr int G = WIDTH / 2;
        constexpr int kCols = G / kEpiParts;
        static_assert(kCols % 32 == 0, "gated epilogue slice");
        const int c0 = part * kCols;
#pragma unroll 1
        for (int c = c0; c < c0 + kCols; c += 32) {
            uint32_t g[32], u[32];
            ptx::tmem_ld_32x32b_x32(taddr + c, g);
            ptx::tmem_ld_32x32b_x32(taddr + G + c, u);
            ptx::tmem_wait_ld(g);
            ptx::tmem_wait_ld(u);
            if (c + 32 == c0 + kCols) release();
            epilogue_gated_slice<MODE == Mode::kGemm1GatedTrain>(
                g, u, args.bias + n0 + c, args.bias + n0 + G + c, args, row, n0 / 2 + c, stage);
        }
    } else {
        constexpr int kCols = WIDTH / kEpiParts;
        static_assert(kCols % 32 == 0, "epilogue slice");
        const int c0 = part * kCols;
#pragma unroll 1
        for (int c = c0; c < c0 + kCols; c += 32) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(taddr + c, v);
            ptx::tmem_wait_ld(v);
            if (c + 32 == c0 + kCols) release();
            if constexpr (MODE == Mode::kBwdGated)
                epilogue_bwd_gated_slice(v, args, row, n0 + c, stage);
            else
                epilogue_slice<MODE, OUT_F32>(v, args.bias, args.out, row, args.M, args.ldo,
                                              n0 + c, args.residual, args.out2, stage);
        }
    }
}

// Row block (of kBM or kPairBM rows) and column block of tile t; with tall units, of the
// ordinary tile t after them (see GemmArgs::tall_units).
// A tall unit of the second GEMM (CTA-pair kernel): this warp's share of both accumulators,
// the first half's rows (accumulator at taddr0, this lane's row row0) and the second half's
// (taddr1, row1) over the same output columns, 32 columns at a time with both halves'
// tensor-memory loads in flight together. `release` hands both accumulators back once their
// last columns are in registers.
template <Mode MODE, bool OUT_F32, int WIDTH, typename Release>
__device__ __forceinline__ void drain_tall(uint32_t taddr0, uint32_t taddr1, const GemmArgs& args,
                                           int row0, int row1, int n0, int part, uint32_t stage,
                                           Release release) {
    static_assert(MODE == Mode::kGemm2 || MODE == Mode::kGemm2Residual, "tall units: second GEMM");
    constexpr int kCols = WIDTH / kEpiParts;
    const int c0 = part * kCols;
#pragma unroll 1
    for (int c = c0; c < c0 + kCols; c += 32) {
        uint32_t v0[32], v1[32];
        ptx::tmem_ld_32x32b_x32(taddr0 + c, v0);
        ptx::tmem_ld_32x32b_x32(taddr1 + c, v1);
        ptx::tmem_wait_ld(v0);
        ptx::tmem_wait_ld(v1);
        if (c + 32 == c0 + kCols) release();
        epilogue_slice<MODE, OUT_F32>(v0, args.bias, args.out, row0, args.M, args.ldo, n0 + c,
                                      args.residual, args.out2, stage);
        epilogue_slice<MODE, OUT_F32>(v1, args.bias, args.out, row1, args.M, args.ldo, n0 + c,
                                      args.residual, args.out2, stage);
    }
}

__device__ __forceinline__ void decode_tile(const GemmArgs& a, int t, int& m_blk, int& n_blk) {
    if (a.tall_units > 0)
        decode_tall_rest(a.group_m, a.tall_m_blocks, a.tall_units, a.tall_rest, a.m_blocks,
                         a.n_blocks, t, m_blk, n_blk);
    else
        decode_tile_mn(a.group_m, a.m_blocks, a.n_blocks, t, m_blk, n_blk);
}

// Bring the bias of this warp's columns in tile t (the CTA's first) into L2 while the tile's
// operands stream in. In a short launch after a cold L2, the epilogue's bias loads would
// otherwise wait on DRAM once per 32-column slice; later tiles find the bias in L2.
template <Mode MODE, int WIDTH>
__device__ __forceinline__ void prefetch_tile_bias(const GemmArgs& a, int t, int part) {
    if constexpr (has_bias(MODE)) {
        if (t >= a.num_tiles) return;
        int m_blk, n_blk;
        decode_tile(a, t, m_blk, n_blk);
        constexpr bool kGated = is_gated(MODE);
        constexpr int kCols = (kGated ? WIDTH / 2 : WIDTH) / kEpiParts;  // <= 128: 4 lines
        const int lane = threadIdx.x & 31;
        const int line = lane & 3, half = lane >> 2;  // half 1: the gated layer's up columns
        if (32 * line < kCols && half < (kGated ? 2 : 1)) {
            const float* p = a.bias + n_blk * WIDTH + half * (WIDTH / 2) + part * kCols + 32 * line;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
        }
    }
}

// A: GEMM1 -> X [M][H] (2-D map, box 64 x 128); GEMM2 -> Y [M][F] (2-D map, box 64 x 128).
// B: GEMM1 -> W1p [k][f][H] (3-D map, box 64 x BN x 1); GEMM2 -> W2p [k][H][f] (same box).
// MN: both operands M-/N-contiguous (the weight-gradient GEMMs, reduction over tokens):
// A = 2 TMA boxes of 64 (M) x 64 (K), B = BN/64 boxes of 64 (N) x 64 (K); the maps' inner
// dimension is the output row / column index and the outer one the token.
template <int BN, int STAGES, Mode MODE, bool OUT_F32, bool MN = false>
__global__ void __launch_bounds__(kNumThreads, 1)
    tpmlp_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmB2, const GemmArgs args) {
    using L = GemmSmem<BN, STAGES>;
    constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN, MN);
    constexpr int kCode = static_cast<int>(MODE) << 8;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    // control block after the stage ring
    const uint32_t ctrl = base + STAGES * L::kStageBytes;
    auto full_bar = [&](int s) { return ctrl + 8u * s; };
    auto empty_bar = [&](int s) { return ctrl + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return ctrl + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return ctrl + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = ctrl + 8u * (2 * STAGES + 4);
    uint32_t* const tmem_holder =
        reinterpret_cast<uint32_t*>(base_ptr + STAGES * L::kStageBytes + 8 * (2 * STAGES + 5));
    volatile uint32_t* const abort_flag = tmem_holder + 1;

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 5, 0);
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), kEpiWarps);
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
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), L::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // The set-up above overlaps the previous kernel's tail; global memory only from here on.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < args.num_tiles; t += gridDim.x) {
                int m_blk, n_blk;
                decode_tile(args, t, m_blk, n_blk);
                const int m0 = m_blk * kBM;
                const int n0 = n_blk * BN;
                const int shard1 = is_gemm1(MODE) ? n0 / args.f : 0;
                const int n_in_shard1 = n0 - shard1 * args.f;
                for (int kb = 0; kb < args.kb_tile; ++kb) {
                    if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.status,
                                        kCode | kSiteProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + stage * L::kStageBytes;
                    const uint32_t sb = sa + L::kABytes;
#ifdef TPMLP_TEST_SKIP_STAGE
                    // test builds only: never fill this stage, so the MMA's wait on it runs out
                    if (issued == TPMLP_TEST_SKIP_STAGE) {
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
#endif
                    ptx::mbar_arrive_expect_tx(full_bar(stage), L::kStageBytes);
                    if constexpr (MN) {
#pragma unroll
                        for (int b = 0; b < kBM / 64; ++b)
                            ptx::tma_load_2d(sa + b * 8192, &tmA, full_bar(stage), m0 + 64 * b,
                                             kb * kBK);
#pragma unroll
                        for (int b = 0; b < BN / 64; ++b)
                            ptx::tma_load_2d(sb + b * 8192, &tmB, full_bar(stage), n0 + 64 * b,
                                             kb * kBK);
                    } else if constexpr (is_gemm1(MODE)) {
                        ptx::tma_load_2d(sa, &tmA, full_bar(stage), kb * kBK, m0);
                        ptx::tma_load_3d(sb, &tmB, full_bar(stage), kb * kBK, n_in_shard1, shard1);
                    } else {
                        const int i = kb / args.kb_shard;               // shard of this block
                        const int kk = (kb - i * args.kb_shard) * kBK;  // offset inside shard i
                        const bool second = i >= args.k2;
                        ptx::tma_load_2d(sa, &tmA, full_bar(stage), i * args.f + kk, m0);
                        ptx::tma_load_3d(sb, second ? &tmB2 : &tmB, full_bar(stage), kk, n0,
                                         second ? i - args.k2 : i);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // wait for the copies still in flight before the CTA may exit
                for (uint32_t s = 0; s < STAGES && s < issued; ++s) {
                    const uint32_t last = s + ((issued - 1 - s) / STAGES) * STAGES;
                    ptx::mbar_wait_drain(full_bar(s), (last / STAGES) & 1u);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < args.num_tiles; t += gridDim.x) {
                if (!ptx::mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.status,
                                    kCode | kSiteMmaAccum)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < args.kb_tile; ++kb) {
                    if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag, args.status,
                                        kCode | kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = base + stage * L::kStageBytes;
                    const uint64_t da = MN ? sdesc_mn128(sa) : sdesc_k128(sa);
                    const uint64_t db = MN ? sdesc_mn128(sa + L::kABytes) : sdesc_k128(sa + L::kABytes);
                    // one MMA covers 16 of the stage's 64 K: 32 bytes along a K-major row
                    // (>> 4 = 2), or 16 rows of 128 bytes in an MN-major box (>> 4 = 128)
                    constexpr uint32_t kStep = MN ? 128u : 2u;
#pragma unroll
                    for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                        ptx::mma_bf16_ss(d_tmem, da + kStep * kk, db + kStep * kk, kIdesc,
                                         (kb | kk) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(empty_bar(stage));  // stage free once these MMAs finish
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(tfull_bar(acc));  // accumulator complete
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // every MMA this thread issued has completed before tensor memory is released
            ptx::mma_commit(drain_bar);
            ptx::mbar_wait_drain(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lanes [32q, 32q+32) = tile rows this warp may read
        const int part = (warp - 2) >> 2;  // which share of the columns
        uint32_t acc = 0, acc_phase = 0;
        prefetch_tile_bias<MODE, BN>(args, blockIdx.x, part);
        for (int t = blockIdx.x; t < args.num_tiles; t += gridDim.x) {
            int m_blk, n_blk;
            decode_tile(args, t, m_blk, n_blk);
            const int m0 = m_blk * kBM;
            const int n0 = n_blk * BN;
            bool ok = ptx::mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.status,
                                     kCode | kSiteEpilogue);
            if (!__all_sync(0xffffffffu, ok)) break;
            ptx::tc_fence_after();
            const int row = m0 + q * 32 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            const uint32_t empty = tempty_bar(acc);
            const uint32_t stage_buf = base + L::kEpiOffset + (warp - 2) * kStageSliceBytes;
            drain_accumulator<MODE, OUT_F32, BN>(taddr, args, row, n0, part, stage_buf, [&] {
                // all of this warp's accumulator columns are in registers: hand it back
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_relaxed(empty);
            });
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

}  // namespace tpmlp
