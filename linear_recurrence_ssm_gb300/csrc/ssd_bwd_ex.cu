// ssd_bwd_ex.cu -- gradients of the chunked scalar-decay ("SSD") scan with
// its options: the dt bias, softplus and clamp, the silu gate z and the
// initial state h0 -- the outputs the chunked backward of "Some questions of
// Bi-Mamba2 and Hydra" (Bi-Mamba2 issue 1) returns besides dx, ddt, dA, dB,
// dC, dD: dz, ddt_bias and the initial states' gradient.
//
// With v = dt + dt_bias, s = softplus(v) (or v), dte = clamp(s, lo, hi) (or
// s), u = scan(dte) + D x (from h0) and y = u silu(z) (or u), the chain rule
// splits the gradient into steps that each have a kernel of their own:
//   dte and the chain factor f = [lo <= s <= hi] sig(v)   (elementwise)
//   g = dy silu(z), dz = dy u silu'(z)                    (u: the forward
//                                                          scan without z)
//   dx, d dte, dA, dB, dC, dD of the scan run from a zero state, for g
//                                                         (ssd_bwd.cu)
//   the terms of h0: its part of the output is
//     y0_t[p] = e^{cum_t} sum_n C_t[n] h0[p, n],  cum_t = A sum_{r <= t} dte_r,
//   so dh0 = sum_t e^{cum_t} g_t C_t^T, dC_t += e^{cum_t} h0^T g_t and, with
//   s_t = g_t . y0_t, d dte_r += A sum_{t >= r} s_t, dA += sum_t (cum_t / A) s_t
//   ddt = d dte f,  ddt_bias[h] = sum over (b, t) of ddt  (fixed order)
// bf16 inputs are widened to fp32 first (exactly), so every step runs on the
// fp32 kernels; h0 is single-direction only, as in the forward scan.
#include "ssm_common.cuh"
#include "grad_options.cuh"

#include <algorithm>

namespace ssm {
namespace ssd_general {
template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dt, const float *A_head, const Tin *Bm, const Tin *Cm,
                   const float *D, float *y, int64_t Bs, int64_t L, int64_t H, int64_t P,
                   int64_t N, bool bidir, int num_sms, const ScanOpts *opt, cudaStream_t st);
}
namespace ssd_bwd {
template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dt, const float *A_head, const Tin *Bm, const Tin *Cm,
                   const float *D, const float *dy, float *dx, float *ddt, float *dA, float *dB,
                   float *dC, float *dD, int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                   int64_t G, bool bidir, cudaStream_t st);
}
namespace ssd_bwd_ex {

constexpr int kThreads = 256;
using namespace grad_opts;

// The terms of the initial state h0 (single direction), one CTA of 256
// threads per (b, h), walking t in batches of kB steps.  Thread tid owns
// column n = tid % N and rows p = tid / N + k (256 / N) of h0 and of dh0;
// its partial sum over its rows c_t = sum_p h0[p, n] g_t[p] serves both
// dC_t[n] (the partials of the 256 / N threads of a column added in a fixed
// order) and s_t = e^{cum_t} sum_n C_t[n] c_t[n] (a CTA sum in a fixed
// order).  The s_t go to scratch; a second loop forms their suffix sums
// for ddt.  dC and dA are sums over heads / batch rows: atomics, as in the
// plain gradients.
constexpr int kB = 16;

__global__ void __launch_bounds__(kThreads)
h0_terms_kernel(const float *__restrict__ Cm, const float *__restrict__ g,
                const float *__restrict__ dte, const float *__restrict__ A,
                const float *__restrict__ h0, float *__restrict__ dC, float *__restrict__ dh0,
                float *__restrict__ ddt, float *__restrict__ dA, float *__restrict__ sarr, int L,
                int H, int P, int N, int G) {
    __shared__ float Cs[kB][256];
    __shared__ float gs[kB][128];
    __shared__ float es[kB];
    __shared__ double css[kB];
    __shared__ float red[kB * 256];      // [pg][j][n] partials of the column sums
    __shared__ float ws[kThreads / 32][kB];
    __shared__ float scan_buf[kThreads];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x, b = bh / H, h = bh % H, grp = h / (H / G);
    const float Ah = A[h];
    const float A2 = Ah * SSM_LOG2E;
    const int n = tid % N, pg0 = tid / N, pstep = kThreads / N;
    const int rows = P / pstep;          // rows of this thread (P * N / 256)
    float hv[32], acc[32];
    for (int k = 0; k < 32; ++k) {
        hv[k] = 0.0f;
        acc[k] = 0.0f;
    }
    for (int k = 0; k < rows; ++k) hv[k] = h0[(size_t(bh) * P + pg0 + k * pstep) * N + n];
    double csum = 0.0;                   // sum of dte up to the current step (thread 0)
    float dA_part = 0.0f;                // thread j < kB: sum of csum_t s_t over its steps
    for (int t0 = 0; t0 < L; t0 += kB) {
        const int nb = min(kB, L - t0);
        // stage the batch: C rows, g rows, decay factors
        for (int i = tid; i < kB * N; i += kThreads) {
            const int j = i / N, c = i % N;
            Cs[j][c] = j < nb ? Cm[((size_t(b) * L + t0 + j) * G + grp) * N + c] : 0.0f;
        }
        for (int i = tid; i < kB * P; i += kThreads) {
            const int j = i / P, c = i % P;
            gs[j][c] = j < nb ? g[((size_t(b) * L + t0 + j) * H + h) * P + c] : 0.0f;
        }
        if (tid == 0) {
            for (int j = 0; j < kB; ++j) {
                if (j < nb) csum += double(dte[(size_t(b) * L + t0 + j) * H + h]);
                css[j] = csum;
                es[j] = j < nb ? ex2(float(double(A2) * csum)) : 0.0f;
            }
        }
        __syncthreads();
        float sp[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const float e = es[j], cn = Cs[j][n];
            float c = 0.0f;
            for (int k = 0; k < rows; ++k) {
                const float gv = gs[j][pg0 + k * pstep];
                c = fmaf(hv[k], gv, c);
                acc[k] = fmaf(e * gv, cn, acc[k]);
            }
            red[(pg0 * kB + j) * N + n] = c;
            sp[j] = c * cn;
        }
        // s_t: the CTA sum of sp[j] for each j, in a fixed order
#pragma unroll
        for (int j = 0; j < kB; ++j) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sp[j] += __shfl_xor_sync(0xffffffffu, sp[j], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < kB; ++j) ws[warp][j] = sp[j];
        }
        __syncthreads();
        // dC_t[n] += e_t * (sum over the column's threads, in order)
        for (int i = tid; i < kB * N; i += kThreads) {
            const int j = i / N, c = i % N;
            if (j < nb) {
                float v = 0.0f;
                for (int q = 0; q < pstep; ++q) v += red[(q * kB + j) * N + c];
                atomicAdd(&dC[((size_t(b) * L + t0 + j) * G + grp) * N + c], es[j] * v);
            }
        }
        if (tid < kB && tid < nb) {
            float sv = 0.0f;
            for (int w = 0; w < kThreads / 32; ++w) sv += ws[w][tid];
            sv *= es[tid];
            sarr[size_t(bh) * L + t0 + tid] = sv;
            dA_part = fmaf(float(css[tid]), sv, dA_part);
        }
        __syncthreads();                 // the batch's buffers are free again
    }
    if (dh0)
        for (int k = 0; k < rows; ++k) dh0[(size_t(bh) * P + pg0 + k * pstep) * N + n] = acc[k];
    // dA: the kB partials in order
    if (tid < kB) ws[0][tid] = dA_part;
    __syncthreads();
    if (tid == 0) {
        float v = 0.0f;
        for (int j = 0; j < kB; ++j) v += ws[0][j];
        atomicAdd(&dA[h], v);
    }
    // ddt_r += A sum_{t >= r} s_t: thread i takes a block of steps, the block
    // sums are scanned from the right, then each block is walked backwards
    const int per = (L + kThreads - 1) / kThreads;
    const int t_lo = min(L, tid * per), t_hi = min(L, t_lo + per);
    float bsum = 0.0f;
    for (int t = t_lo; t < t_hi; ++t) bsum += sarr[size_t(bh) * L + t];
    scan_buf[tid] = bsum;
    __syncthreads();
    if (tid == 0) {                      // exclusive suffix sums of the blocks
        float run = 0.0f;
        for (int i = kThreads - 1; i >= 0; --i) {
            const float v = scan_buf[i];
            scan_buf[i] = run;
            run += v;
        }
    }
    __syncthreads();
    float run = scan_buf[tid];
    for (int t = t_hi - 1; t >= t_lo; --t) {
        run += sarr[size_t(bh) * L + t];
        ddt[(size_t(b) * L + t) * H + h] += Ah * run;
    }
}

// The whole call; every step stream-ordered on st, the scratch taken and
// released with cudaMallocAsync / cudaFreeAsync on st.
template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dt, const float *A_head, const Tin *Bm, const Tin *Cm,
                   const float *D, const float *dy, float *dx, float *ddt, float *dA, float *dB,
                   float *dC, float *dD, float *dz, float *ddt_bias, float *dh0, int64_t Bs,
                   int64_t L, int64_t H, int64_t P, int64_t N, int64_t G, bool bidir,
                   const ScanOpts &o, int num_sms, cudaStream_t st) {
    const int64_t nt = Bs * L * H, nx = nt * P, nbc = Bs * L * G * N;
    const bool wide = sizeof(Tin) == 2;
    const bool gate = o.z != nullptr, init = o.h0 != nullptr;
    // scratch: dte, chain [nt]; fp32 copies of x, B, C (bf16 inputs);
    // u, g [nx] (gate); s [Bs H L] (initial state)
    // (each part starts on a 256-byte boundary: the forward scan stages rows
    // of x, B, C with 16-byte copies)
    auto up = [](size_t n) { return (n + 63) / 64 * 64; };
    size_t floats = 2 * up(nt);
    if (wide) floats += up(nx) + 2 * up(nbc);
    if (gate) floats += 2 * up(nx);
    if (init) floats += up(size_t(Bs) * H * L);
    void *scratch = nullptr;
    cudaError_t err = cudaMallocAsync(&scratch, floats * sizeof(float), st);
    if (err != cudaSuccess) return err;
    float *cur = static_cast<float *>(scratch);
    auto take = [&](size_t n) { float *p = cur; cur += up(n); return p; };
    float *dte = take(nt), *chain = take(nt);
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
    prep_kernel<Tin><<<grid_for(nt), kThreads, 0, st>>>(dt, o.dt_bias, o.dt_softplus, o.dt_limit,
                                                       o.dt_min, o.dt_max, dte, chain, nt, int(H));
    err = cudaGetLastError();
    const float *g = dy;
    if (err == cudaSuccess && gate) {
        // the ungated output u: the scan of dte from h0, D x included
        float *u = take(nx), *gw = take(nx);
        ScanOpts fo{};
        fo.h0 = o.h0;
        fo.ngroups = int(G);
        err = ssd_general::launch<float>(x32, dte, A_head, B32, C32, D, u, Bs, L, H, P, N, bidir,
                                         num_sms, &fo, st);
        if (err == cudaSuccess) {
            gate_kernel<Tin><<<grid_for(nx), kThreads, 0, st>>>(dy, static_cast<const Tin *>(o.z), u,
                                                               gw, dz, nx);
            err = cudaGetLastError();
        }
        g = gw;
    }
    if (err == cudaSuccess)
        err = ssd_bwd::launch<float>(x32, dte, A_head, B32, C32, D, g, dx, ddt, dA, dB, dC, dD, Bs,
                                     L, H, P, N, G, bidir, st);
    if (err == cudaSuccess && init) {
        float *sarr = take(size_t(Bs) * H * L);
        h0_terms_kernel<<<unsigned(Bs * H), kThreads, 0, st>>>(C32, g, dte, A_head, o.h0, dC, dh0,
                                                              ddt, dA, sarr, int(L), int(H), int(P),
                                                              int(N), int(G));
        err = cudaGetLastError();
    }
    if (err == cudaSuccess && (o.dt_bias || o.dt_softplus || o.dt_limit)) {
        chain_bias_kernel<<<unsigned(H), kThreads, 0, st>>>(ddt, chain, ddt_bias, Bs * L, int(H));
        err = cudaGetLastError();
    }
    cudaError_t e2 = cudaFreeAsync(scratch, st);
    return err != cudaSuccess ? err : e2;
}

template cudaError_t launch<float>(const float *, const float *, const float *, const float *,
                                   const float *, const float *, const float *, float *, float *,
                                   float *, float *, float *, float *, float *, float *, float *,
                                   int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, bool,
                                   const ScanOpts &, int, cudaStream_t);
template cudaError_t launch<__nv_bfloat16>(const __nv_bfloat16 *, const __nv_bfloat16 *,
                                           const float *, const __nv_bfloat16 *,
                                           const __nv_bfloat16 *, const float *, const float *,
                                           float *, float *, float *, float *, float *, float *,
                                           float *, float *, float *, int64_t, int64_t, int64_t,
                                           int64_t, int64_t, int64_t, bool, const ScanOpts &, int,
                                           cudaStream_t);
}  // namespace ssd_bwd_ex
}  // namespace ssm
