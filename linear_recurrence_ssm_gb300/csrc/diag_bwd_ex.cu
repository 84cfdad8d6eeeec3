// diag_bwd_ex.cu -- gradients of the diagonal selective scan with its
// options (the delta bias, softplus and clamp, the silu gate z, the initial
// state h0): dz, ddt_bias and dh0 besides dx, ddelta, dA, dB, dC, dD, as the
// chunked backward of "Some questions of Bi-Mamba2 and Hydra" (Bi-Mamba2
// issue 1) returns them, for the diagonal form.
//
// The same composition as the chunked scan's (ssd_bwd_ex.cu): the options'
// elementwise steps (grad_options.cuh), the forward scan without z for the
// ungated output u, the plain gradients from a zero state for
// g = dy silu(z) (diag_scan_bwd.cu), and the terms of h0.  With
// csum_t[e] = sum_{r <= t} delta_r[e] and E_t[e, n] = exp(A[e, n] csum_t[e]),
// the part of the output h0 gives is y0_t[e] = sum_n C_t[n] E_t[e, n] h0[e, n],
// so
//   dh0[e, n]   = sum_t g_t[e] C_t[n] E_t[e, n]
//   dC_t[n]    += sum_e g_t[e] E_t[e, n] h0[e, n]
//   dA[e, n]   += sum_t g_t[e] C_t[n] csum_t[e] E_t[e, n] h0[e, n]
//   ddelta_r[e] += sum_{t >= r} q_t[e],  q_t[e] = g_t[e] sum_n C_t[n] A[e, n] E_t[e, n] h0[e, n].
#include "ssm_common.cuh"
#include "grad_options.cuh"

namespace ssm {
namespace diag {
template <typename Tin>
cudaError_t launch_ext(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                       const float *D, float *y, int64_t Bs, int64_t L, int64_t ED, int64_t N,
                       int num_sms, const ScanOpts &ex, cudaStream_t st);
}
namespace diag_bwd {
template <typename Tin>
cudaError_t launch_bwd(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                       const float *D, const float *dy, float *dx, float *ddelta, float *dA,
                       float *dB, float *dC, float *dD, int64_t Bs, int64_t L, int64_t ED,
                       int64_t N, int num_sms, cudaStream_t st);
}
namespace diag_bwd_ex {

using namespace grad_opts;
constexpr int kCh = 128;   // channels per CTA (one thread each)
constexpr int kMaxN = 16;  // states held in registers per walk

// The terms of h0: one thread per channel e of batch row blockIdx.y, walking
// t once per group of kMaxN states (their exponentials in registers); the
// dC_t[n] terms are summed over the warp's channels with shuffles and added
// with one atomic per warp; q_t, summed over the groups, goes to scratch and
// a backward walk forms its suffix sums.
__global__ void __launch_bounds__(kCh)
h0_terms_kernel(const float *__restrict__ Cm, const float *__restrict__ g,
                const float *__restrict__ dlt, const float *__restrict__ A,
                const float *__restrict__ h0, float *__restrict__ dC, float *__restrict__ dh0,
                float *__restrict__ ddelta, float *__restrict__ dA, float *__restrict__ q,
                int L, int ED, int N) {
    const int b = blockIdx.y, e = blockIdx.x * kCh + threadIdx.x, lane = threadIdx.x & 31;
    const bool ok = e < ED;
    for (int n0 = 0; n0 < N; n0 += kMaxN) {
        const int nc = N - n0 < kMaxN ? N - n0 : kMaxN;
        float hv[kMaxN], a2[kMaxN], acc[kMaxN], dA_acc[kMaxN];
#pragma unroll
        for (int n = 0; n < kMaxN; ++n) {
            const bool on = ok && n < nc;
            hv[n] = on ? h0[(size_t(b) * ED + e) * N + n0 + n] : 0.0f;
            a2[n] = on ? A[size_t(e) * N + n0 + n] * SSM_LOG2E : 0.0f;
            acc[n] = 0.0f;
            dA_acc[n] = 0.0f;
        }
        double csum = 0.0;
        for (int t = 0; t < L; ++t) {
            const size_t i = (size_t(b) * L + t) * ED + e;
            float gv = 0.0f;
            if (ok) {
                csum += double(dlt[i]);
                gv = g[i];
            }
            const float cs = float(csum);
            float qv = 0.0f;
#pragma unroll
            for (int n = 0; n < kMaxN; ++n) {
                if (n >= nc) break;
                const float c = Cm[(size_t(b) * L + t) * N + n0 + n];
                const float E = ok ? ex2(a2[n] * cs) : 0.0f;
                const float eh = E * hv[n];
                acc[n] = fmaf(gv * c, E, acc[n]);
                dA_acc[n] = fmaf(gv * c * cs, eh, dA_acc[n]);
                qv = fmaf(c * a2[n], eh, qv);
                // dC_t[n]: this warp's channels, then one atomic
                float dc = gv * eh;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dc += __shfl_xor_sync(0xffffffffu, dc, o);
                if (lane == 0 && dc != 0.0f) atomicAdd(&dC[(size_t(b) * L + t) * N + n0 + n], dc);
            }
            // (a2 carries log2 e)
            if (ok) q[i] = (n0 == 0 ? 0.0f : q[i]) + gv * qv * float(1.0 / SSM_LOG2E);
        }
        if (ok) {
#pragma unroll
            for (int n = 0; n < kMaxN; ++n) {
                if (n >= nc) break;
                if (dh0) dh0[(size_t(b) * ED + e) * N + n0 + n] = acc[n];
                atomicAdd(&dA[size_t(e) * N + n0 + n], dA_acc[n]);
            }
        }
    }
    if (!ok) return;
    float run = 0.0f;
    for (int t = L - 1; t >= 0; --t) {
        const size_t i = (size_t(b) * L + t) * ED + e;
        run += q[i];
        ddelta[i] += run;
    }
}

template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                   const float *D, const float *dy, float *dx, float *ddelta, float *dA, float *dB,
                   float *dC, float *dD, float *dz, float *ddt_bias, float *dh0, int64_t Bs,
                   int64_t L, int64_t ED, int64_t N, const ScanOpts &o, int num_sms,
                   cudaStream_t st) {
    const int64_t nx = Bs * L * ED, nbc = Bs * L * N;
    const bool wide = sizeof(Tin) == 2;
    const bool gate = o.z != nullptr, init = o.h0 != nullptr;
    auto up = [](size_t n) { return (n + 63) / 64 * 64; };
    size_t floats = 2 * up(nx);                                  // dseen, chain
    if (wide) floats += up(nx) + 2 * up(nbc);
    if (gate) floats += 2 * up(nx);
    if (init) floats += up(nx);
    void *scratch = nullptr;
    cudaError_t err = cudaMallocAsync(&scratch, floats * sizeof(float), st);
    if (err != cudaSuccess) return err;
    float *cur = static_cast<float *>(scratch);
    auto take = [&](size_t n) { float *p = cur; cur += up(n); return p; };
    float *dseen = take(nx), *chain = take(nx);
    const float *x32 = reinterpret_cast<const float *>(x);
    const float *B32 = reinterpret_cast<const float *>(Bm);
    const float *C32 = reinterpret_cast<const float *>(Cm);
    if (wide) {
        float *xw = take(nx), *bw = take(nbc), *cw = take(nbc);
        widen_kernel<<<grid_for(nx), kThreads, 0, st>>>(reinterpret_cast<const __nv_bfloat16 *>(x), xw, nx);
        widen_kernel<<<grid_for(nbc), kThreads, 0, st>>>(reinterpret_cast<const __nv_bfloat16 *>(Bm), bw, nbc);
        widen_kernel<<<grid_for(nbc), kThreads, 0, st>>>(reinterpret_cast<const __nv_bfloat16 *>(Cm), cw, nbc);
        x32 = xw;
        B32 = bw;
        C32 = cw;
    }
    prep_kernel<Tin><<<grid_for(nx), kThreads, 0, st>>>(dlt, o.dt_bias, o.dt_softplus, o.dt_limit,
                                                       o.dt_min, o.dt_max, dseen, chain, nx,
                                                       int(ED));
    err = cudaGetLastError();
    const float *g = dy;
    if (err == cudaSuccess && gate) {
        float *u = take(nx), *gw = take(nx);
        ScanOpts fo{};
        fo.h0 = o.h0;
        err = diag::launch_ext<float>(x32, dseen, A, B32, C32, D, u, Bs, L, ED, N, num_sms, fo, st);
        if (err == cudaSuccess) {
            gate_kernel<Tin><<<grid_for(nx), kThreads, 0, st>>>(dy, static_cast<const Tin *>(o.z), u,
                                                               gw, dz, nx);
            err = cudaGetLastError();
        }
        g = gw;
    }
    if (err == cudaSuccess)
        err = diag_bwd::launch_bwd<float>(x32, dseen, A, B32, C32, D, g, dx, ddelta, dA, dB, dC, dD,
                                          Bs, L, ED, N, num_sms, st);
    if (err == cudaSuccess && init) {
        float *q = take(nx);
        const dim3 grid(unsigned((ED + kCh - 1) / kCh), unsigned(Bs));
        h0_terms_kernel<<<grid, kCh, 0, st>>>(C32, g, dseen, A, o.h0, dC, dh0, ddelta, dA, q,
                                              int(L), int(ED), int(N));
        err = cudaGetLastError();
    }
    if (err == cudaSuccess && (o.dt_bias || o.dt_softplus || o.dt_limit)) {
        chain_bias_kernel<<<unsigned(ED), kThreads, 0, st>>>(ddelta, chain, ddt_bias, Bs * L,
                                                             int(ED));
        err = cudaGetLastError();
    }
    cudaError_t e2 = cudaFreeAsync(scratch, st);
    return err != cudaSuccess ? err : e2;
}

template cudaError_t launch<float>(const float *, const float *, const float *, const float *,
                                   const float *, const float *, const float *, float *, float *,
                                   float *, float *, float *, float *, float *, float *, float *,
                                   int64_t, int64_t, int64_t, int64_t, const ScanOpts &, int,
                                   cudaStream_t);
template cudaError_t launch<__nv_bfloat16>(const __nv_bfloat16 *, const __nv_bfloat16 *,
                                           const float *, const __nv_bfloat16 *,
                                           const __nv_bfloat16 *, const float *, const float *,
                                           float *, float *, float *, float *, float *, float *,
                                           float *, float *, float *, int64_t, int64_t, int64_t,
                                           int64_t, const ScanOpts &, int, cudaStream_t);
}  // namespace diag_bwd_ex
}  // namespace ssm
