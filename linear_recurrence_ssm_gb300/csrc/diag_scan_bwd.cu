// diag_scan_bwd.cu -- gradients of the diagonal selective scan (N <= 16).
//
// Forward: h_t = a_t h_{t-1} + delta_t B_t x_t with a_t[n] = exp(delta_t A[e,n]),
// y_t = C_t . h_t + D[e] x_t.  Given dy, the adjoint of the state runs
// backwards in time,
//     g_t[n] = dy_t C_t[n] + a_{t+1}[n] g_{t+1}[n],    g_L = 0,
// and every input gradient is a sum over (t, n) of g_t with quantities of
// the forward pass (h_{t-1}, a_t): see the formulas at diag_bwd_kernel.
//
// Two passes.  The first re-runs the forward recurrence and keeps the state
// entering every kSeg-step segment (checkpoints).  The second walks the
// segments from the last to the first: it re-runs a segment forward from its
// checkpoint into shared memory (the entering state of each step), then
// walks the segment backwards carrying g.  Gradients of the per-channel
// parameters (A, D) are summed in registers and added once per thread;
// gradients of B and C are sums over the channels of one batch row: each
// warp reduces its 32 channels through shared memory and adds one value per
// (t, n) to global memory with an atomic add.
#include "ssm_common.cuh"

namespace ssm {
namespace diag_bwd {

constexpr int kNP = 16;       // states (padded)
constexpr int kSeg = 16;      // steps per checkpointed segment
constexpr int kCh = 64;       // channels per CTA (two warps)

// State entering segment k of channel c: ckpt[(k * nch + c) * 16 + n].
template <typename Tin>
__global__ void __launch_bounds__(kCh)
diag_ckpt_kernel(const Tin *__restrict__ x, const Tin *__restrict__ dlt,
                 const float *__restrict__ A, const Tin *__restrict__ Bm, float *__restrict__ ckpt,
                 int Bs, int L, int ED, int N) {
    const int64_t b = blockIdx.y;
    const int e = blockIdx.x * kCh + threadIdx.x;
    if (e >= ED) return;
    const int64_t c = b * ED + e;
    const int64_t nch = int64_t(Bs) * ED;
    float A2[kNP], h[kNP];
#pragma unroll
    for (int n = 0; n < kNP; ++n) {
        A2[n] = n < N ? A[int64_t(e) * N + n] * SSM_LOG2E : 0.0f;
        h[n] = 0.0f;
    }
    for (int t = 0; t < L; ++t) {
        if (t % kSeg == 0) {
            float4 *dst = reinterpret_cast<float4 *>(ckpt + ((int64_t(t / kSeg) * nch + c) * kNP));
#pragma unroll
            for (int q = 0; q < kNP / 4; ++q)
                dst[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
        }
        const int64_t i = (b * L + t) * ED + e;
        const float dl = to_f32(dlt[i]), dlx = dl * to_f32(x[i]);
        const Tin *br = Bm + (b * L + t) * N;
#pragma unroll
        for (int n = 0; n < kNP; ++n) {
            const float bv = n < N ? to_f32(br[n]) : 0.0f;
            h[n] = fmaf(ex2(dl * A2[n]), h[n], dlx * bv);
        }
    }
}

// Reverse pass.  Per step t (thread = channel e of batch row b), with
// hp = h_{t-1} and g = g_t:
//   dx_t     = sum_n g[n] delta_t B_t[n] + D[e] dy_t
//   ddelta_t = sum_n g[n] (A[e,n] a_t[n] hp[n] + B_t[n] x_t)
//   dA[e,n] += g[n] delta_t a_t[n] hp[n]
//   dB_t[n] += g[n] delta_t x_t        (summed over the channels e)
//   dC_t[n] += dy_t h_t[n]             (summed over the channels e)
//   dD[e]   += dy_t x_t
template <typename Tin>
__global__ void __launch_bounds__(kCh)
diag_bwd_kernel(const Tin *__restrict__ x, const Tin *__restrict__ dlt, const float *__restrict__ A,
                const Tin *__restrict__ Bm, const Tin *__restrict__ Cm, const float *__restrict__ D,
                const float *__restrict__ dy, const float *__restrict__ ckpt,
                float *__restrict__ dx, float *__restrict__ ddelta, float *__restrict__ dA,
                float *__restrict__ dB, float *__restrict__ dC, float *__restrict__ dD, int Bs,
                int L, int ED, int N) {
    extern __shared__ float smem[];
    float *hist = smem;                                  // [kSeg][kNP][kCh]: h_{t-1} per step
    float *red = smem + kSeg * kNP * kCh;                // [2 warps][32 lanes][2 * kNP + 1]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t b = blockIdx.y;
    const int e = blockIdx.x * kCh + threadIdx.x;
    const bool e_ok = e < ED;
    const int ec = e_ok ? e : ED - 1;                    // lanes past ED mirror a channel, add zero
    const int64_t c = b * ED + ec;
    const int64_t nch = int64_t(Bs) * ED;
    float A2[kNP], An[kNP], g[kNP], lA[kNP];
#pragma unroll
    for (int n = 0; n < kNP; ++n) {
        An[n] = n < N ? A[int64_t(ec) * N + n] : 0.0f;
        A2[n] = An[n] * SSM_LOG2E;
        g[n] = 0.0f;
        lA[n] = 0.0f;
    }
    const float Dv = D ? D[ec] : 0.0f;
    float lD = 0.0f;
    float *myred = red + (warp * 32 + lane) * (2 * kNP + 1);
    const int nseg = (L + kSeg - 1) / kSeg;
    for (int k = nseg - 1; k >= 0; --k) {
        const int t0 = k * kSeg;
        const int tl = min(kSeg, L - t0);
        float h[kNP];
        {
            const float4 *src = reinterpret_cast<const float4 *>(ckpt + (int64_t(k) * nch + c) * kNP);
#pragma unroll
            for (int q = 0; q < kNP / 4; ++q) {
                const float4 v = src[q];
                h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
            }
        }
        // forward over the segment: keep the entering state of every step
        for (int j = 0; j < tl; ++j) {
            const int64_t i = (b * L + t0 + j) * ED + ec;
            const float dl = to_f32(dlt[i]), dlx = dl * to_f32(x[i]);
            const Tin *br = Bm + (b * L + t0 + j) * N;
#pragma unroll
            for (int n = 0; n < kNP; ++n) {
                hist[(j * kNP + n) * kCh + threadIdx.x] = h[n];
                const float bv = n < N ? to_f32(br[n]) : 0.0f;
                h[n] = fmaf(ex2(dl * A2[n]), h[n], dlx * bv);
            }
        }
        // backward over the segment
        for (int j = tl - 1; j >= 0; --j) {
            const int t = t0 + j;
            const int64_t i = (b * L + t) * ED + ec;
            const float dl = to_f32(dlt[i]), xv = to_f32(x[i]);
            const float gy = e_ok ? dy[i] : 0.0f;
            const Tin *br = Bm + (b * L + t) * N;
            const Tin *cr = Cm + (b * L + t) * N;
            float sdx = 0.0f, sdd = 0.0f;
#pragma unroll
            for (int n = 0; n < kNP; ++n) {
                const float bv = n < N ? to_f32(br[n]) : 0.0f;
                const float cv = n < N ? to_f32(cr[n]) : 0.0f;
                const float a = ex2(dl * A2[n]);
                const float hp = hist[(j * kNP + n) * kCh + threadIdx.x];
                g[n] = fmaf(gy, cv, g[n]);                      // g_t
                sdx = fmaf(g[n] * dl, bv, sdx);
                sdd = fmaf(g[n], fmaf(An[n] * a, hp, bv * xv), sdd);
                lA[n] = fmaf(g[n] * dl * a, hp, lA[n]);
                myred[n] = e_ok ? g[n] * dl * xv : 0.0f;        // this channel's share of dB_t[n]
                myred[kNP + n] = gy * fmaf(a, hp, dl * bv * xv);  // share of dC_t[n] (dy_t h_t[n])
                g[n] *= a;                                      // a_t g_t, for step t - 1
            }
            if (e_ok) {
                dx[i] = fmaf(Dv, gy, sdx);
                ddelta[i] = sdd;
                lD = fmaf(gy, xv, lD);
            }
            __syncwarp();
            // lane l sums column l (l < 16: dB_t[l]; l >= 16: dC_t[l - 16]) over the warp
            float s = 0.0f;
            for (int r = 0; r < 32; ++r) s += red[(warp * 32 + r) * (2 * kNP + 1) + lane];
            const int n = lane & (kNP - 1);
            if (n < N) atomicAdd((lane < kNP ? dB : dC) + (b * L + t) * N + n, s);
            __syncwarp();
        }
    }
    if (e_ok) {
#pragma unroll
        for (int n = 0; n < kNP; ++n)
            if (n < N) atomicAdd(dA + int64_t(e) * N + n, lA[n]);
        if (dD) atomicAdd(dD + e, lD);
    }
}

template <typename Tin>
cudaError_t launch_bwd(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                       const float *D, const float *dy, float *dx, float *ddelta, float *dA,
                       float *dB, float *dC, float *dD, int64_t Bs, int64_t L, int64_t ED,
                       int64_t N, cudaStream_t st) {
    if (N > kNP) return cudaErrorNotSupported;
    if (Bs > 65535) return cudaErrorInvalidConfiguration;
    // parameter gradients are sums: start from zero
    cudaError_t err = cudaMemsetAsync(dA, 0, size_t(ED * N) * sizeof(float), st);
    if (err == cudaSuccess) err = cudaMemsetAsync(dB, 0, size_t(Bs * L * N) * sizeof(float), st);
    if (err == cudaSuccess) err = cudaMemsetAsync(dC, 0, size_t(Bs * L * N) * sizeof(float), st);
    if (err == cudaSuccess && dD) err = cudaMemsetAsync(dD, 0, size_t(ED) * sizeof(float), st);
    if (err != cudaSuccess) return err;
    const int64_t nseg = (L + kSeg - 1) / kSeg;
    void *scratch = nullptr;
    err = cudaMallocAsync(&scratch, size_t(nseg * Bs * ED) * kNP * sizeof(float), st);
    if (err != cudaSuccess) return err;
    float *ckpt = static_cast<float *>(scratch);
    const dim3 grid(unsigned((ED + kCh - 1) / kCh), unsigned(Bs));
    diag_ckpt_kernel<Tin><<<grid, kCh, 0, st>>>(x, dlt, A, Bm, ckpt, int(Bs), int(L), int(ED), int(N));
    err = cudaGetLastError();
    if (err == cudaSuccess) {
        const int smem = int((kSeg * kNP * kCh + 2 * 32 * (2 * kNP + 1)) * sizeof(float));
        err = cudaFuncSetAttribute(diag_bwd_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   smem);
        if (err == cudaSuccess) {
            diag_bwd_kernel<Tin><<<grid, kCh, smem, st>>>(x, dlt, A, Bm, Cm, D, dy, ckpt, dx, ddelta,
                                                          dA, dB, dC, dD, int(Bs), int(L), int(ED),
                                                          int(N));
            err = cudaGetLastError();
        }
    }
    cudaError_t e2 = cudaFreeAsync(scratch, st);
    return err != cudaSuccess ? err : e2;
}

template cudaError_t launch_bwd<float>(const float *, const float *, const float *, const float *,
                                       const float *, const float *, const float *, float *,
                                       float *, float *, float *, float *, float *, int64_t,
                                       int64_t, int64_t, int64_t, cudaStream_t);
template cudaError_t launch_bwd<__nv_bfloat16>(const __nv_bfloat16 *, const __nv_bfloat16 *,
                                               const float *, const __nv_bfloat16 *,
                                               const __nv_bfloat16 *, const float *, const float *,
                                               float *, float *, float *, float *, float *,
                                               float *, int64_t, int64_t, int64_t, int64_t,
                                               cudaStream_t);

}  // namespace diag_bwd
}  // namespace ssm
