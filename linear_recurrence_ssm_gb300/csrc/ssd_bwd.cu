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
// walks the recurrence (warp w holds rows p = w, w + 8, ...; lane l columns
// n = l, l + 32, ...), its inputs loaded a batch of steps at a time, and
// streams every state H_k (fp32) to a scratch buffer; the second walks
// backwards with the adjoint in registers.  Its inputs for step k (the state
// H_{k-1}, the rows x_t, dy_t, B_t, C_t, dt_t and, for the second direction,
// the dx and ddt written by the first) are fetched two steps ahead into a
// three-slot shared-memory ring -- the state with cp.async, the rest through
// registers -- and H_k is carried in registers from the step before.  Sums
// over n use warp shuffles, sums over p one shared-memory reduction per step
// (one barrier), and dB, dC, dA, dD are added with atomics (so their last
// bits may differ between runs).  The scratch is Bs*H*L*P*N*4 bytes.
#include "ssm_common.cuh"

namespace ssm {
namespace ssd_bwd_chunk {   // the chunked form (ssd_bwd_chunk.cu)
bool supported(int64_t P, int64_t N);
template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dt, const float *A_head, const Tin *Bm, const Tin *Cm,
                   const float *D, const float *dy, float *dx, float *ddt, float *dA, float *dB,
                   float *dC, float *dD, int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                   int64_t G, bool bidir, cudaStream_t st);
}  // namespace ssd_bwd_chunk
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

// Steps whose inputs the state pass loads at once (about 96 registers).
template <int PW, int NL>
__host__ __device__ constexpr int hist_batch() {
    return 96 / (1 + PW + NL) < 2 ? 2 : (96 / (1 + PW + NL) > 8 ? 8 : 96 / (1 + PW + NL));
}

template <typename Tin, int PW, int NL>
__global__ void __launch_bounds__(kThreads)
ssd_bwd_history_kernel(const Args<Tin> a, int dir) {
    constexpr int U = hist_batch<PW, NL>();
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
    for (int k0 = 0; k0 < L; k0 += U) {
        // the batch's inputs first, so that their loads overlap
        float dtv[U], xv[U][PW], bv[U][NL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = walk(k0 + u < L ? k0 + u : L - 1, L, dir);
            dtv[u] = to_f32(a.dt[(size_t(b) * L + t) * a.H + h]);
            const Tin *xr = a.x + ((size_t(b) * L + t) * a.H + h) * P;
            const Tin *br = a.B + ((size_t(b) * L + t) * a.G + g) * N;
#pragma unroll
            for (int i = 0; i < PW; ++i) xv[u][i] = to_f32(xr[warp + kWarps * i]);
#pragma unroll
            for (int j = 0; j < NL; ++j) bv[u][j] = to_f32(br[lane + 32 * j]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (k0 + u >= L) break;
            const float dec = __expf(dtv[u] * Ah);
            float *hk = hrow + size_t(k0 + u) * P * N;
#pragma unroll
            for (int i = 0; i < PW; ++i) {
                const int p = warp + kWarps * i;
                const float w = dtv[u] * xv[u][i];
#pragma unroll
                for (int j = 0; j < NL; ++j) {
                    st[i][j] = fmaf(dec, st[i][j], w * bv[u][j]);
                    __stcs(hk + p * N + lane + 32 * j, st[i][j]);   // read back much later
                }
            }
        }
    }
}

// Inputs of one reverse step, staged in a ring slot after the state H_{k-1}
// (P * N floats): x_t, dy_t, the first direction's dx_t (P each), B_t, C_t
// (N each), dt_t, the first direction's ddt_t, two pad floats.  Offsets in
// floats from the slot's start.
struct SlotLayout {
    int ox, ody, odx, oB, oC, odt, oddt, n_in, floats;
    __host__ __device__ SlotLayout(int P, int N)
        : ox(P * N), ody(ox + P), odx(ody + P), oB(odx + P), oC(oB + N), odt(oC + N),
          oddt(odt + 1), n_in(3 * P + 2 * N + 2), floats(odt + 4) {}
};
constexpr int kRing = 3;          // slots: step k in use, k - 1 and k - 2 in flight
constexpr int kInRegs = 3;        // inputs a thread stages per step: 3P + 2N + 2 <= 3 * 256

__host__ __device__ inline size_t reverse_smem_bytes(int P, int N) {
    return (size_t(kRing) * SlotLayout(P, N).floats + size_t(2) * kWarps * (2 * N + 2)) *
           sizeof(float);
}

// Loads walk step s's inputs (time t) into registers; element e of the slot's
// input block goes to thread e mod 256, register e / 256.
template <typename Tin>
__device__ __forceinline__ void fetch_inputs(const Args<Tin> &a, int b, int h, int g, int t,
                                             bool with_prev, float (&v)[kInRegs]) {
    const int P = a.P, N = a.N;
    const size_t xo = ((size_t(b) * a.L + t) * a.H + h) * P;
    const size_t bo = ((size_t(b) * a.L + t) * a.G + g) * N;
    const size_t to = (size_t(b) * a.L + t) * a.H + h;
#pragma unroll
    for (int r = 0; r < kInRegs; ++r) {
        int e = threadIdx.x + kThreads * r;
        float val = 0.0f;
        if (e < P) val = to_f32(a.x[xo + e]);
        else if ((e -= P) < P) val = a.dy[xo + e];
        else if ((e -= P) < P) { if (with_prev) val = a.dx[xo + e]; }
        else if ((e -= P) < N) val = to_f32(a.B[bo + e]);
        else if ((e -= N) < N) val = to_f32(a.C[bo + e]);
        else if ((e -= N) == 0) val = to_f32(a.dt[to]);
        else if (e == 1) { if (with_prev) val = a.ddt[to]; }
        v[r] = val;
    }
}

__device__ __forceinline__ void stage_inputs(float *slot, const SlotLayout &lay,
                                             const float (&v)[kInRegs]) {
#pragma unroll
    for (int r = 0; r < kInRegs; ++r) {
        const int e = threadIdx.x + kThreads * r;
        if (e < lay.n_in) slot[lay.ox + e] = v[r];
    }
}

// Reverse walk of one direction.  first: this launch writes dx and ddt (and
// adds the D terms); otherwise it adds to the values the first one wrote.
template <typename Tin, int PW, int NL>
__global__ void __launch_bounds__(kThreads)
ssd_bwd_reverse_kernel(const Args<Tin> a, int dir, int first) {
    extern __shared__ __align__(16) float sm[];
    const int P = a.P, N = a.N, L = a.L, PN = P * N;
    const SlotLayout lay(P, N);
    // per-warp partial sums of one step (double buffered by step parity):
    // [0, N) dB column sums, [N, 2N) dC column sums, 2N the input part of
    // ddt, 2N + 1 <Gb_k, H_{k-1}>
    const int red_f = 2 * N + 2;
    float *const red = sm + kRing * lay.floats;
    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H, g = h / (a.H / a.G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const float Ah = a.A[h];
    const float Dh = (first && a.D) ? a.D[h] : 0.0f;
    const bool with_prev = !first;
    const float *hrow = a.hist + size_t(bh) * L * PN;
    auto slot = [&](int s) { return sm + (s % kRing) * lay.floats; };
    // H_{s-1} into slot s (s >= 1), as one cp.async group (empty otherwise)
    auto issue_state = [&](int s) {
        if (s >= 1) {
            float *dst = slot(s);
            const float *src = hrow + size_t(s - 1) * PN;
            for (int c = tid; c < PN / 4; c += kThreads) cp_async16(dst + 4 * c, src + 4 * c, 16);
        }
        cp_async_commit();
    };

    float gb[PW][NL], hk[PW][NL];          // adjoint Gb, state H_k
#pragma unroll
    for (int i = 0; i < PW; ++i)
#pragma unroll
        for (int j = 0; j < NL; ++j) {
            gb[i][j] = 0.0f;
            hk[i][j] = hrow[size_t(L - 1) * PN + (warp + kWarps * i) * N + lane + 32 * j];
        }
    float vA[kInRegs], vB[kInRegs];
#pragma unroll
    for (int r = 0; r < kInRegs; ++r) vB[r] = 0.0f;
    issue_state(L - 1);
    fetch_inputs(a, b, h, g, walk(L - 1, L, dir), with_prev, vA);
    stage_inputs(slot(L - 1), lay, vA);
    issue_state(L - 2);
    if (L >= 2) fetch_inputs(a, b, h, g, walk(L - 2, L, dir), with_prev, vB);
    cp_async_wait<1>();
    __syncthreads();

    float dA_acc = 0.0f, dD_acc = 0.0f;
    // One reverse step k: prefetch step k - 2, compute step k, stage step k - 1.
    auto body = [&](int k, float (&vload)[kInRegs], const float (&vstore)[kInRegs]) {
        issue_state(k - 2);
        if (k >= 2) fetch_inputs(a, b, h, g, walk(k - 2, L, dir), with_prev, vload);
        const int t = walk(k, L, dir);
        const size_t xo = ((size_t(b) * L + t) * a.H + h) * P;
        const size_t bo = ((size_t(b) * L + t) * a.G + g) * N;
        const float *sl = slot(k);
        const float dtv = sl[lay.odt];
        const float dec = __expf(dtv * Ah);
        float bv[NL], cv[NL], uB[NL], uC[NL];
#pragma unroll
        for (int j = 0; j < NL; ++j) {
            bv[j] = sl[lay.oB + lane + 32 * j];
            cv[j] = sl[lay.oC + lane + 32 * j];
            uB[j] = 0.0f;
            uC[j] = 0.0f;
        }
        const bool has_prev = k > 0;
        float din = 0.0f, sda = 0.0f;
#pragma unroll
        for (int i = 0; i < PW; ++i) {
            const int p = warp + kWarps * i;
            const float xv = sl[lay.ox + p];
            const float gy = sl[lay.ody + p];
            float v = 0.0f;
#pragma unroll
            for (int j = 0; j < NL; ++j) {
                gb[i][j] = fmaf(gy, cv[j], gb[i][j]);          // Gb_k
                v = fmaf(gb[i][j], bv[j], v);
                uB[j] = fmaf(gb[i][j], xv, uB[j]);
                uC[j] = fmaf(gy, hk[i][j], uC[j]);
                if (has_prev) {
                    const float hp = sl[p * N + lane + 32 * j];     // H_{k-1}
                    sda = fmaf(gb[i][j], hp, sda);
                    hk[i][j] = hp;                              // H_k of step k - 1
                }
                gb[i][j] *= dec;                                // a_k Gb_k, for step k - 1
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) {
                const float d = dtv * v + Dh * gy;
                a.dx[xo + p] = with_prev ? sl[lay.odx + p] + d : d;
                din = fmaf(xv, v, din);
                dD_acc = fmaf(gy, xv, dD_acc);
            }
        }
        if (k >= 1) stage_inputs(slot(k - 1), lay, vstore);
        cp_async_wait<1>();                                     // H_{k-2}, for step k - 1
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sda += __shfl_xor_sync(0xffffffffu, sda, o);
        float *rw = red + ((k & 1) * kWarps + warp) * red_f;
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
        const float *rp = red + (k & 1) * kWarps * red_f;
        if (tid < N) {
            float sb = 0.0f, sc = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                sb += rp[w * red_f + tid];
                sc += rp[w * red_f + N + tid];
            }
            atomicAdd(&a.dB[bo + tid], dtv * sb);
            atomicAdd(&a.dC[bo + tid], sc);
        }
        if (tid == kThreads - 1) {
            float s_in = 0.0f, s_da = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                s_in += rp[w * red_f + 2 * N];
                s_da += rp[w * red_f + 2 * N + 1];
            }
            const float d = s_in + Ah * dec * s_da;
            float *dd = a.ddt + (size_t(b) * L + t) * a.H + h;
            *dd = with_prev ? sl[lay.oddt] + d : d;
            dA_acc = fmaf(dtv * dec, s_da, dA_acc);
        }
    };
    for (int k = L - 1; k >= 0; k -= 2) {
        body(k, vA, vB);
        if (k >= 1) body(k - 1, vB, vA);
    }
    if (tid == kThreads - 1) atomicAdd(&a.dA[h], dA_acc);
    if (first && a.dD && lane == 0) atomicAdd(&a.dD[h], dD_acc);
}

template <typename Tin, int PW, int NL>
static cudaError_t run(const Args<Tin> &a, int64_t grid, bool bidir, cudaStream_t st) {
    const size_t smem = reverse_smem_bytes(a.P, a.N);
    cudaError_t e = cudaFuncSetAttribute(ssd_bwd_reverse_kernel<Tin, PW, NL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    for (int dir = 0; dir < (bidir ? 2 : 1); ++dir) {
        ssd_bwd_history_kernel<Tin, PW, NL><<<unsigned(grid), kThreads, 0, st>>>(a, dir);
        ssd_bwd_reverse_kernel<Tin, PW, NL><<<unsigned(grid), kThreads, smem, st>>>(a, dir, dir == 0);
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
    // P = 64, N = 64 or 128: the chunked form (its reads of x, dy, B, C are
    // 16 bytes wide)
    auto a16 = [](const void *q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    if (ssd_bwd_chunk::supported(P, N) && Bs * H <= 65535 && a16(dx) && a16(x) && a16(dy) &&
        a16(Bm) && a16(Cm))
        return ssd_bwd_chunk::launch<Tin>(x, dt, A_head, Bm, Cm, D, dy, dx, ddt, dA, dB, dC, dD, Bs,
                                          L, H, P, N, G, bidir, st);
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
