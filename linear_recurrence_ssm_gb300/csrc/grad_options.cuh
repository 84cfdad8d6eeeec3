// grad_options.cuh -- the elementwise steps of the gradients of the scans'
// options, shared by the diagonal (diag_bwd_ex.cu) and chunked
// (ssd_bwd_ex.cu) scans: with v = dt + dt_bias, s = softplus(v) (or v),
// dte = clamp(s, lo, hi) (or s), u the scan's output before the gate and
// y = u silu(z):
//   dte and the chain factor f = [lo <= s <= hi] sig(v)
//   g = dy silu(z) (the upstream gradient of the scan), dz = dy u silu'(z)
//   ddt = d dte f and ddt_bias[c] = sum over (b, t) of ddt, in a fixed order
// (c the channel of the bias: the diagonal scan's ED, the chunked scan's H).
#pragma once

#include "ssm_common.cuh"

#include <algorithm>

namespace ssm {
namespace grad_opts {
namespace {   // each translation unit keeps its own copy of these kernels

constexpr int kThreads = 256;

__device__ __forceinline__ float sigmoid_exact(float v) { return 1.0f / (1.0f + expf(-v)); }

// dte and the chain factor f of every (b, t, h).
template <typename Tin>
__global__ void prep_kernel(const Tin *__restrict__ dt, const float *__restrict__ bias, int softplus,
                            int limit, float lo, float hi, float *__restrict__ dte,
                            float *__restrict__ chain, int64_t n, int H) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x) {
        const float v = to_f32(dt[i]) + (bias ? bias[i % H] : 0.0f);
        float s = v, f = 1.0f;
        if (softplus) {
            s = v > 20.0f ? v : log1pf(expf(v));
            f = sigmoid_exact(v);
        }
        if (limit) {
            if (s < lo || s > hi) f = 0.0f;   // clamped: no gradient
            s = fminf(fmaxf(s, lo), hi);
        }
        dte[i] = s;
        chain[i] = f;
    }
}

// Exact widening of bf16 to fp32.
__global__ void widen_kernel(const __nv_bfloat16 *__restrict__ src, float *__restrict__ dst,
                             int64_t n) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x)
        dst[i] = __bfloat162float(src[i]);
}

// g = dy silu(z) and dz = dy u silu'(z), silu'(z) = sig(z) (1 + z (1 - sig(z))).
template <typename Tin>
__global__ void gate_kernel(const float *__restrict__ dy, const Tin *__restrict__ z,
                            const float *__restrict__ u, float *__restrict__ g, float *__restrict__ dz,
                            int64_t n) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x) {
        const float zv = to_f32(z[i]);
        const float sg = sigmoid_exact(zv);
        g[i] = dy[i] * zv * sg;
        if (dz) dz[i] = dy[i] * u[i] * sg * (1.0f + zv * (1.0f - sg));
    }
}

// ddt *= f, then ddt_bias[h] = sum over (b, t) of ddt: one CTA per head,
// the sum formed in a fixed order (so reruns give the same bits).
__global__ void chain_bias_kernel(float *__restrict__ ddt, const float *__restrict__ chain,
                                  float *__restrict__ ddt_bias, int64_t rows, int H) {
    __shared__ float part[kThreads];
    const int h = blockIdx.x;
    float acc = 0.0f;
    for (int64_t r = threadIdx.x; r < rows; r += kThreads) {
        const int64_t i = r * H + h;
        const float v = ddt[i] * chain[i];
        ddt[i] = v;
        acc += v;
    }
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int s = kThreads / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) part[threadIdx.x] += part[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0 && ddt_bias) ddt_bias[h] = part[0];
}

inline unsigned grid_for(int64_t n) {
    return unsigned(std::min<int64_t>((n + kThreads - 1) / kThreads, 4096));
}

}  // namespace
}  // namespace grad_opts
}  // namespace ssm
