// ssd_bwd.cu -- gradients of the chunked scalar-decay ("SSD") scan on CUDA
// cores: dx, ddt, dA, dB, dC, dD for an upstream gradient dy, both
// directions of the bidirectional scan and groups of B, C -- the quantities
// of the chunked backward pass named in "Some questions of Bi-Mamba2 and
// Hydra" (Bi-Mamba2 issue 1), computed from the recurrence step by step.
//
// Per (b, h) and direction, walking k = 0 .. L-1 over t = k (forward) or
// t = L-1-k (reversed), with H_k the P x N state after walk step k and
// a_k = exp(dt_t A_h):
//   H_k = a_k H_{k-1} + dt_t x_t B_t^T,   y_t += H_k C_t   (+ D_h x_t once).
// The adjoint of H_k is Gb_k = dy_t C_t^T + a_{k+1} Gb_{k+1} (Gb_L = 0), and
//   dx_t   += dt_t Gb_k B_t          (+ D_h dy_t once)
//   dB_t   += dt_t Gb_k^T x_t        dC_t += H_k^T dy_t     (summed over a group's heads)
//   ddt_t  += <Gb_k, x_t B_t^T> + A_h a_k <Gb_k, H_{k-1}>
//   dA_h   += sum_k dt_t a_k <Gb_k, H_{k-1}>,   dD_h += sum_t dy_t . x_t (once).
//
// Two kernels per direction, one CTA of 256 threads per (b, h): the first
// walks the recurrence and stores every state H_k (fp32) in a scratch
// buffer; the second walks backwards with the adjoint in registers (warp w
// holds rows p = w, w + 8, ...; lane l columns n = l, l + 32, ...), reduces
// over n with warp shuffles and over p through shared memory (one barrier
// per step), and adds dB, dC, dA, dD with atomics (so their last bits may
// differ between runs).  A correctness path: its scratch is Bs*H*L*P*N*4
// bytes and it reads two states per step.
#include "ssm_common.cuh"

namespace ssm {
namespace ssd_bwd {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename Tin>
struct Args {
    const Tin *x, *dt, *B, *C;
    const float *A, *D, *dy;
    float *dx, *ddt, *dA, *dB, *dC, *dD;
    float *hist;            // [Bs * H][L][P * N]
    int L, H, P, N, G;
};

// Time index of walk step k of direction dir (1: reversed).
__device__ __forceinline__ int walk(int k, int L, int dir) { return dir ? L - 1 - k : k; }

template <typename Tin, int PW, int NL>
__global__ void __launch_bounds__(kThreads)
ssd_bwd_history_kernel(const Args<Tin> a, int dir) {
    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H, g = h / (a.H / a.G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int P = a.P, N = a.N, L = a.L;
    const float Ah = a.A[h];
    float st[PW][NL];
#pragma unroll
    for (int i = 0; i < PW; ++i)
#pragma unroll
        for (int j = 0; j < NL; ++j) st[i][j] = 0.0f;
    float *hrow = a.hist + size_t(bh) * L * P * N;
    for (int k = 0; k < L; ++k) {
        const int t = walk(k, L, dir);
        const float dtv = to_f32(a.dt[(size_t(b) * L + t) * a.H + h]);
        const float dec = __expf(dtv * Ah);
        const Tin *xr = a.x + ((size_t(b) * L + t) * a.H + h) * P;
        const Tin *br = a.B + ((size_t(b) * L + t) * a.G + g) * N;
        float bv[NL];
#pragma unroll
        for (int j = 0; j < NL; ++j) bv[j] = to_f32(br[lane + 32 * j]);
        float *hk = hrow + size_t(k) * P * N;
#pragma unroll
        for (int i = 0; i < PW; ++i) {
            const int p = warp + kWarps * i;
            const float u = dtv * to_f32(xr[p]);
#pragma unroll
            for (int j = 0; j < NL; ++j) {
                st[i][j] = fmaf(dec, st[i][j], u * bv[j]);
                hk[p * N + lane + 32 * j] = st[i][j];
            }
        }
    }
}

// Reverse walk of one direction.  first: this launch writes dx and ddt (and
// adds the D terms); otherwise it adds to them (the second direction).
template <typename Tin, int PW, int NL>
__global__ void __launch_bounds__(kThreads)
ssd_bwd_reverse_kernel(const Args<Tin> a, int dir, int first) {
    // per-warp partial sums of one step (double buffered by step parity):
    // [0, N) dB column sums, [N, 2N) dC column sums, 2N the input part of
    // ddt, 2N + 1 <Gb_k, H_{k-1}>
    __shared__ float red[2][kWarps][2 * 256 + 2];
    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H, g = h / (a.H / a.G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int P = a.P, N = a.N, L = a.L;
    const float Ah = a.A[h];
    const float Dh = (first && a.D) ? a.D[h] : 0.0f;
    float gb[PW][NL];
#pragma unroll
    for (int i = 0; i < PW; ++i)
#pragma unroll
        for (int j = 0; j < NL; ++j) gb[i][j] = 0.0f;
    const float *hrow = a.hist + size_t(bh) * L * P * N;
    float dA_acc = 0.0f, dD_acc = 0.0f;
    for (int k = L - 1; k >= 0; --k) {
        const int t = walk(k, L, dir);
        const int par = k & 1;
        const size_t xo = ((size_t(b) * L + t) * a.H + h) * P;
        const size_t bo = ((size_t(b) * L + t) * a.G + g) * N;
        const float dtv = to_f32(a.dt[(size_t(b) * L + t) * a.H + h]);
        const float dec = __expf(dtv * Ah);
        float bv[NL], cv[NL], uB[NL], uC[NL];
#pragma unroll
        for (int j = 0; j < NL; ++j) {
            bv[j] = to_f32(a.B[bo + lane + 32 * j]);
            cv[j] = to_f32(a.C[bo + lane + 32 * j]);
            uB[j] = 0.0f;
            uC[j] = 0.0f;
        }
        const float *hk = hrow + size_t(k) * P * N;
        const float *hp = k > 0 ? hrow + size_t(k - 1) * P * N : nullptr;
        float din = 0.0f, sda = 0.0f;
#pragma unroll
        for (int i = 0; i < PW; ++i) {
            const int p = warp + kWarps * i;
            const float xv = to_f32(a.x[xo + p]);
            const float gy = a.dy[xo + p];
            float v = 0.0f;
#pragma unroll
            for (int j = 0; j < NL; ++j) {
                const int n = lane + 32 * j;
                gb[i][j] = fmaf(gy, cv[j], gb[i][j]);          // Gb_k
                v = fmaf(gb[i][j], bv[j], v);
                uB[j] = fmaf(gb[i][j], xv, uB[j]);
                uC[j] = fmaf(gy, hk[p * N + n], uC[j]);
                if (hp) sda = fmaf(gb[i][j], hp[p * N + n], sda);
                gb[i][j] *= dec;                                // a_k Gb_k, for step k - 1
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) {
                const float d = dtv * v + Dh * gy;
                if (first) a.dx[xo + p] = d;
                else a.dx[xo + p] += d;
                din = fmaf(xv, v, din);
                dD_acc = fmaf(gy, xv, dD_acc);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sda += __shfl_xor_sync(0xffffffffu, sda, o);
        float *rw = red[par][warp];
#pragma unroll
        for (int j = 0; j < NL; ++j) {
            rw[lane + 32 * j] = uB[j];
            rw[N + lane + 32 * j] = uC[j];
        }
        if (lane == 0) {
            rw[2 * N] = din;
            rw[2 * N + 1] = sda;
        }
        __syncthreads();
        if (tid < N) {
            float sb = 0.0f, sc = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                sb += red[par][w][tid];
                sc += red[par][w][N + tid];
            }
            atomicAdd(&a.dB[bo + tid], dtv * sb);
            atomicAdd(&a.dC[bo + tid], sc);
        }
        if (tid == kThreads - 1) {
            float s_in = 0.0f, s_da = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                s_in += red[par][w][2 * N];
                s_da += red[par][w][2 * N + 1];
            }
            const float d = s_in + Ah * dec * s_da;
            float *dd = a.ddt + (size_t(b) * L + t) * a.H + h;
            if (first) *dd = d;
            else *dd += d;
            dA_acc = fmaf(dtv * dec, s_da, dA_acc);
        }
    }
    if (tid == kThreads - 1) atomicAdd(&a.dA[h], dA_acc);
    if (first && a.dD && lane == 0) atomicAdd(&a.dD[h], dD_acc);
}

template <typename Tin, int PW, int NL>
static cudaError_t run(const Args<Tin> &a, int64_t grid, bool bidir, cudaStream_t st) {
    for (int dir = 0; dir < (bidir ? 2 : 1); ++dir) {
        ssd_bwd_history_kernel<Tin, PW, NL><<<unsigned(grid), kThreads, 0, st>>>(a, dir);
        ssd_bwd_reverse_kernel<Tin, PW, NL><<<unsigned(grid), kThreads, 0, st>>>(a, dir, dir == 0);
    }
    return cudaGetLastError();
}

template <typename Tin, int PW>
static cudaError_t run_pw(const Args<Tin> &a, int64_t grid, bool bidir, cudaStream_t st) {
    switch (a.N) {
        case 32: return run<Tin, PW, 1>(a, grid, bidir, st);
        case 64: return run<Tin, PW, 2>(a, grid, bidir, st);
        case 128: if constexpr (PW <= 8) return run<Tin, PW, 4>(a, grid, bidir, st); break;
        case 256: if constexpr (PW <= 4) return run<Tin, PW, 8>(a, grid, bidir, st); break;
    }
    return cudaErrorNotSupported;
}

// Head size P in {16, 32, 64, 128}, state size N in {32, 64, 128, 256},
// P * N <= 8192 (the adjoint's registers).
bool supported(int64_t P, int64_t N) {
    const bool p_ok = P == 16 || P == 32 || P == 64 || P == 128;
    const bool n_ok = N == 32 || N == 64 || N == 128 || N == 256;
    return p_ok && n_ok && P * N <= 8192;
}

template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dt, const float *A_head, const Tin *Bm, const Tin *Cm,
                   const float *D, const float *dy, float *dx, float *ddt, float *dA, float *dB,
                   float *dC, float *dD, int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                   int64_t G, bool bidir, cudaStream_t st) {
    if (!supported(P, N) || G < 1 || H % G != 0) return cudaErrorNotSupported;
    const int64_t grid = Bs * H;
    if (grid > 0x7fffffff || L > 0x7fffffff) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaMemsetAsync(dA, 0, size_t(H) * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, size_t(Bs * L * G * N) * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dC, 0, size_t(Bs * L * G * N) * sizeof(float), st);
    if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, size_t(H) * sizeof(float), st);
    if (e != cudaSuccess) return e;
    void *hist = nullptr;
    e = cudaMallocAsync(&hist, size_t(grid) * size_t(L) * size_t(P * N) * sizeof(float), st);
    if (e != cudaSuccess) return e;
    Args<Tin> a{x, dt, Bm, Cm, A_head, D, dy, dx, ddt, dA, dB, dC, dD,
                static_cast<float *>(hist), int(L), int(H), int(P), int(N), int(G)};
    switch (P) {
        case 16: e = run_pw<Tin, 2>(a, grid, bidir, st); break;
        case 32: e = run_pw<Tin, 4>(a, grid, bidir, st); break;
        case 64: e = run_pw<Tin, 8>(a, grid, bidir, st); break;
        case 128: e = run_pw<Tin, 16>(a, grid, bidir, st); break;
        default: e = cudaErrorNotSupported;
    }
    const cudaError_t e2 = cudaFreeAsync(hist, st);
    return e != cudaSuccess ? e : e2;
}

template cudaError_t launch<float>(const float *, const float *, const float *, const float *,
                                   const float *, const float *, const float *, float *, float *,
                                   float *, float *, float *, float *, int64_t, int64_t, int64_t,
                                   int64_t, int64_t, int64_t, bool, cudaStream_t);
template cudaError_t launch<__nv_bfloat16>(const __nv_bfloat16 *, const __nv_bfloat16 *,
                                           const float *, const __nv_bfloat16 *,
                                           const __nv_bfloat16 *, const float *, const float *,
                                           float *, float *, float *, float *, float *, float *,
                                           int64_t, int64_t, int64_t, int64_t, int64_t, int64_t,
                                           bool, cudaStream_t);

}  // namespace ssd_bwd
}  // namespace ssm
