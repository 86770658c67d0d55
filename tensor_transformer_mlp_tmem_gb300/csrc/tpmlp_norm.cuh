// LayerNorm of each token's hidden vector: the step in front of the block in a Transformer
// layer. LayerNorm needs the whole hidden vector of a token (大模型分布式并行策略详解 §4.2);
// tokens are independent, which is what lets sequence parallelism split it along the tokens
// (AI大模型分布式训练 §4.2). On one GPU every token is a CTA.
//
//   Xn[m, h] = (X[m, h] - mu_m) * rsqrt(var_m + eps) * gamma[h] + beta[h]
//   mu_m = mean_h X[m, h],  var_m = mean_h (X[m, h] - mu_m)^2  (biased)
//
// One CTA of 256 threads per token row; the row stays in registers (two passes over them:
// mean, then the centred sum of squares), fp32 statistics, bf16 output. Memory-bound: one
// read of X and one write of Xn.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace tpmlp {

constexpr int kNormMaxH = 16384;

// Sum over the CTA; every thread gets the total. `red` holds one float per warp.
template <int THREADS>
__device__ __forceinline__ float norm_block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if constexpr (THREADS == 32) {
        return v;
    } else {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        __syncthreads();  // the previous use of `red` is finished
        if (lane == 0) red[warp] = v;
        __syncthreads();
        float t = lane < THREADS / 32 ? red[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        return t;
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One CTA of THREADS threads per token row; each thread keeps NC 16-byte chunks (8 bf16) of
// the row in registers, packed. Small CTAs keep many rows in flight per SM.
template <int THREADS, int NC>
__global__ void __launch_bounds__(THREADS)
    layernorm_kernel(const uint16_t* __restrict__ X, const float* __restrict__ gamma,
                     const float* __restrict__ beta, float eps, uint16_t* __restrict__ Xn,
                     int H) {
    __shared__ float red[THREADS / 32 > 0 ? THREADS / 32 : 1];
    const size_t row = blockIdx.x;
    const uint4* x4 = reinterpret_cast<const uint4*>(X + row * H);
    uint4* y4 = reinterpret_cast<uint4*>(Xn + row * H);
    const int chunks = H / 8;

    uint4 q[NC];
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int idx = c * THREADS + threadIdx.x;
        q[c] = idx < chunks ? x4[idx] : make_uint4(0, 0, 0, 0);  // zeros add nothing
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint32_t w[4] = {q[c].x, q[c].y, q[c].z, q[c].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) s += bf16_lo(w[i]) + bf16_hi(w[i]);
    }
    const float mean = norm_block_sum<THREADS>(s, red) / static_cast<float>(H);
    float ss = 0.0f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        if (c * THREADS + static_cast<int>(threadIdx.x) < chunks) {
            const uint32_t w[4] = {q[c].x, q[c].y, q[c].z, q[c].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float d0 = bf16_lo(w[i]) - mean, d1 = bf16_hi(w[i]) - mean;
                ss += d0 * d0 + d1 * d1;
            }
        }
    }
    const float rstd = rsqrtf(norm_block_sum<THREADS>(ss, red) / static_cast<float>(H) + eps);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int idx = c * THREADS + threadIdx.x;
        if (idx < chunks) {
            const float4* g4 = reinterpret_cast<const float4*>(gamma + 8 * idx);
            const float4* b4 = reinterpret_cast<const float4*>(beta + 8 * idx);
            const float4 g0 = __ldg(g4), g1 = __ldg(g4 + 1), b0 = __ldg(b4), b1 = __ldg(b4 + 1);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            const uint32_t w[4] = {q[c].x, q[c].y, q[c].z, q[c].w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float lo = (bf16_lo(w[i]) - mean) * rstd * g[2 * i] + b[2 * i];
                const float hi = (bf16_hi(w[i]) - mean) * rstd * g[2 * i + 1] + b[2 * i + 1];
                __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
                o[i] = *reinterpret_cast<uint32_t*>(&p);
            }
            y4[idx] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

}  // namespace tpmlp
