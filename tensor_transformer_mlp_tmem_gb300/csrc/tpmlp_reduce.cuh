// Column sums of a bf16 matrix (the bias gradients of the backward pass: db = sum over the
// token rows of the output gradient), deterministic: a fixed split of the rows into partial
// sums, then the partials added in split order.
#pragma once

#include <cstdint>

namespace tpmlp {

constexpr int kColsumThreads = 256;  // 8 eight-column chunks x 32 row lanes = 64 columns

// partial[s][c] = sum of in[r][c] over the rows r of split s (rows_per_split rows each);
// in has row pitch ld elements.
__global__ void __launch_bounds__(kColsumThreads)
    colsum_partial_kernel(const uint16_t* __restrict__ in, int M, int C, int ld,
                          int rows_per_split, float* __restrict__ partial) {
    __shared__ float red[32][65];
    const int chunk = threadIdx.x & 7;
    const int lane_row = threadIdx.x >> 3;
    const int c0 = blockIdx.x * 64 + chunk * 8;
    const int r_begin = blockIdx.y * rows_per_split;
    const int r_end = min(M, r_begin + rows_per_split);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int r = r_begin + lane_row; r < r_end; r += 32) {
        const uint4 u = *reinterpret_cast<const uint4*>(in + static_cast<size_t>(r) * ld + c0);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] += __uint_as_float(w[i] << 16);
            acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) red[lane_row][chunk * 8 + i] = acc[i];
    __syncthreads();
    if (threadIdx.x < 64) {
        float t = 0.f;
        for (int l = 0; l < 32; ++l) t += red[l][threadIdx.x];
        partial[static_cast<size_t>(blockIdx.y) * C + blockIdx.x * 64 + threadIdx.x] = t;
    }
}

// out[c] = sum over s of partial[s][c], in split order.
__global__ void colsum_final_kernel(const float* __restrict__ partial, int splits, int C,
                                    float* __restrict__ out) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= C) return;
    float t = 0.f;
    for (int s = 0; s < splits; ++s) t += partial[static_cast<size_t>(s) * C + c];
    out[c] = t;
}

}  // namespace tpmlp
