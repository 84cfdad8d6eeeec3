// ssm_common.cuh -- small device helpers shared by the scan kernels
// (asynchronous copies, bf16 unpacking, exp2 on the MUFU pipe).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/ssm_scan.h"

#define SSM_LOG2E 1.4426950408889634f

namespace ssm {

// ---- options of the scans (host and device) -------------------------------
// delta <- clamp(softplus(delta + dt_bias)), y <- y * silu(z), initial and
// final states; null pointers / zero flags mean "not used".  The public
// ssm_scan_options_t is copied into this form by the entry points.
struct ScanOpts {
    const float *dt_bias;   // (ED) diagonal / (H) SSD
    const void *z;          // x-shaped gate, element type of x
    const float *h0;        // initial state, fp32
    float *h_final;         // final state out, fp32
    float dt_min, dt_max;
    int dt_softplus, dt_limit;
    int ngroups;            // SSD: groups of B, C (0 or 1 = one group)
    // internal (gradients of the diagonal scan): the forward pass keeps the
    // state entering every 16-step segment, ckpt[(k * Bs * ED + c) * 16 + n],
    // and may skip writing y
    float *ckpt;
    int no_y;
};

// ---- element conversion ---------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
// Four consecutive elements (8-byte aligned for bf16, 16-byte for fp32).
__device__ __forceinline__ float4 to_f32x4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 to_f32x4(const __nv_bfloat16 *p) {
    // a bf16 is the high half of the fp32 with the same bits
    const uint2 w = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}

// exp2 on the special-function unit (MUFU.EX2); relative error ~2^-22,
// subnormal results flushed to zero.
__device__ __forceinline__ float ex2(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// softplus(d) = log(1 + e^d) on the special-function unit.  Above 20 the
// correction term is below fp32 resolution; far below 0 the result (~e^d)
// may flush to 0, an absolute error under 1e-8.
__device__ __forceinline__ float softplus_fast(float d) {
    return d > 20.0f ? d : __logf(1.0f + __expf(d));
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z); the fast division returns 0 once
// the denominator is huge (z -> -inf), the function's limit.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// ---- cp.async (Ampere-style asynchronous global -> shared copies) ---------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte copy; `src_bytes` < 16 zero-fills the rest (0 = pure zero fill).
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem_dst)),
                 "l"(gsrc), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

}  // namespace ssm
