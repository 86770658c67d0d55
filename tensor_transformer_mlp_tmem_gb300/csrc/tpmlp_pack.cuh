// The shard packer: lays the weights out the way the GEMM kernel's TMA loads want them.
//
// The pages split the first weight by columns and the second by rows into k equal,
// contiguous pieces (AI大模型分布式训练 §2.1-2.2: W [hidden, ffn] into k pieces of
// [hidden, ffn/k]; the row-parallel weight into [in/k, out]); here every piece is also
// transposed so that its reduction dimension is contiguous (K-major), which is what the
// tensor cores read with the 128-byte swizzle:
//
//   W1 [H][F]  ->  W1p [k][f][H]   W1p[i][j][h] = W1[h][i f + j]   (column shard i, transposed)
//   W2 [F][H]  ->  W2p [k][H][f]   W2p[i][n][j] = W2[i f + j][n]   (row shard i, transposed)
//   b1, b2 (bf16) -> fp32 copies (b1 keeps the shard-major order: slice i = b1[i f, (i+1) f))
//
// Packing is a pure permutation of bits (plus an exact bf16 -> fp32 widening of the biases).
#pragma once

#include <cstdint>

namespace tpmlp {

constexpr int kTransposeTile = 64;

// out[b][c][r] = in[b][r][c] for a batch of R x C bf16 matrices (bit copies).
__global__ void __launch_bounds__(256)
    transpose_bf16_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, int R, int C,
                          long long in_batch_stride, long long out_batch_stride) {
    __shared__ uint16_t tile[kTransposeTile][kTransposeTile + 2];
    const long long b = blockIdx.z;
    const int r0 = blockIdx.y * kTransposeTile;
    const int c0 = blockIdx.x * kTransposeTile;
    const uint16_t* src = in + b * in_batch_stride;
    uint16_t* dst = out + b * out_batch_stride;
    const int tx = threadIdx.x;  // 0..63
    for (int i = threadIdx.y; i < kTransposeTile; i += blockDim.y) {
        const int r = r0 + i, c = c0 + tx;
        if (r < R && c < C) tile[i][tx] = src[static_cast<size_t>(r) * C + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < kTransposeTile; i += blockDim.y) {
        const int c = c0 + i, r = r0 + tx;
        if (c < C && r < R) dst[static_cast<size_t>(c) * R + r] = tile[tx][i];
    }
}

// W2 [F][H] -> the second GEMM's operand in 16 KB blocks: for shard i, output row n and
// reduction index j (0 <= j < f), element W2[i f + j][n] sits at
//   ((i * (H / 128) + n / 128) * (f / 64) + j / 64) * 8192 + (n % 128) * 64 + j % 64,
// so the 128 rows x 64 columns that one TMA box of the CTA-pair kernel reads are contiguous.
__global__ void __launch_bounds__(256)
    transpose_blocked_bf16_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out,
                                  int f, int H) {
    __shared__ uint16_t tile[kTransposeTile][kTransposeTile + 2];
    const int i = blockIdx.z;
    const int r0 = blockIdx.y * kTransposeTile;  // j
    const int c0 = blockIdx.x * kTransposeTile;  // n
    const uint16_t* src = in + static_cast<size_t>(i) * f * H;
    const int tx = threadIdx.x;
    for (int y = threadIdx.y; y < kTransposeTile; y += blockDim.y) {
        const int r = r0 + y, c = c0 + tx;
        if (r < f && c < H) tile[y][tx] = src[static_cast<size_t>(r) * H + c];
    }
    __syncthreads();
    for (int y = threadIdx.y; y < kTransposeTile; y += blockDim.y) {
        const int n = c0 + y, j = r0 + tx;
        if (n < H && j < f) {
            const size_t blk = (static_cast<size_t>(i) * (H / 128) + n / 128) * (f / 64) + j / 64;
            out[blk * 8192 + (n % 128) * 64 + j % 64] = tile[tx][y];
        }
    }
}

// Gated first layer: the gate and the up projection are packed into one K-major operand whose
// rows alternate in blocks of G: for output column j (0 <= j < F) of part p (0 = gate,
// 1 = up), the packed row is (j / G) * 2G + p * G + (j % G). With G dividing the shard width
// f, shard i's 2f packed rows are [2 i f, 2 (i+1) f) and every 2G-row tile holds the gate and
// the up columns of the same G outputs.
//   out[(j / G) * 2G + p * G + (j % G)][r] = in[r][j]      (in: [R][C] bf16, out rows of R)
__global__ void __launch_bounds__(256)
    transpose_interleave_bf16_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out,
                                     int R, int C, int G, int part) {
    __shared__ uint16_t tile[kTransposeTile][kTransposeTile + 2];
    const int r0 = blockIdx.y * kTransposeTile;
    const int c0 = blockIdx.x * kTransposeTile;
    const int tx = threadIdx.x;  // 0..63
    for (int i = threadIdx.y; i < kTransposeTile; i += blockDim.y) {
        const int r = r0 + i, c = c0 + tx;
        if (r < R && c < C) tile[i][tx] = in[static_cast<size_t>(r) * C + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < kTransposeTile; i += blockDim.y) {
        const int j = c0 + i, r = r0 + tx;
        if (j < C && r < R) {
            const size_t row = static_cast<size_t>(j / G) * 2 * G + static_cast<size_t>(part) * G + j % G;
            out[row * R + r] = tile[tx][i];
        }
    }
}

// The biases of the gated layer in the same interleaved order (widened to fp32).
__global__ void interleave_bias_kernel(const uint16_t* __restrict__ in, float* __restrict__ out,
                                       int C, int G, int part) {
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < C; j += gridDim.x * blockDim.x)
        out[static_cast<size_t>(j / G) * 2 * G + static_cast<size_t>(part) * G + j % G] =
            __uint_as_float(static_cast<uint32_t>(in[j]) << 16);
}

__global__ void bf16_to_f32_kernel(const uint16_t* __restrict__ in, float* __restrict__ out,
                                   long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        out[i] = __uint_as_float(static_cast<uint32_t>(in[i]) << 16);
}

}  // namespace tpmlp
