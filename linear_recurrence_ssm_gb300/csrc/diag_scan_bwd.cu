// diag_scan_bwd.cu -- gradients of the diagonal selective scan (N <= 256;
// more than 16 states in groups of 16, see launch_bwd).
//
// Forward: h_t = a_t h_{t-1} + delta_t B_t x_t with a_t[n] = exp(delta_t A[e,n]),
// y_t = C_t . h_t + D[e] x_t.  Given dy, the adjoint of the state runs
// backwards in time,
//     g_t[n] = dy_t C_t[n] + a_{t+1}[n] g_{t+1}[n],    g_L = 0,
// and every input gradient is a sum over (t, n) of g_t with quantities of
// the forward pass (h_{t-1}, a_t): see the formulas at diag_bwd_kernel.
//
// Two passes.  The first is the forward scan itself (its kernel run as one
// time segment, y not written), keeping the state entering every kSeg-step
// segment (checkpoints).  The second walks the
// segments from the last to the first: it re-runs a segment forward from its
// checkpoint into shared memory (the entering state of each step), then
// walks the segment backwards carrying g.  Four lanes share a channel, each
// with four of the 16 (padded) states, so a CTA of 256 threads covers 64
// channels of one batch row.  The segment's inputs are staged into shared
// memory one segment ahead.  Gradients of the per-channel parameters (A, D)
// are summed in registers and added once per thread; gradients of B and C
// are sums over channels: each warp reduces its 8 channels with shuffles,
// the CTA sums its 8 warps once per segment and adds one value per (t, n)
// with an atomic add.
#include "ssm_common.cuh"

namespace ssm {
namespace diag {
template <typename Tin>
cudaError_t launch_ext(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                       const float *D, float *y, int64_t Bs, int64_t L, int64_t ED, int64_t N,
                       int num_sms, const ScanOpts &ex, cudaStream_t st);
}  // namespace diag

namespace diag_bwd {

constexpr int kNP = 16;               // states (padded)
constexpr int kLanes = 4;             // lanes per channel
constexpr int kSpl = kNP / kLanes;    // states per lane
constexpr int kSeg = 16;              // steps per checkpointed segment (the forward kernel's)
constexpr int kThreads = 128;      // 32 channels per CTA: small CTAs spread over the SMs evenly (measured: 1.17x faster than 64)
constexpr int kCh = kThreads / kLanes;    // channels per CTA
constexpr int kWarps = kThreads / 32;
static_assert(kSpl == 4, "a lane's states are moved as one float4");

// Inputs of one segment, staged in shared memory.
template <typename Tin>
struct Stage {
    Tin x[kSeg][kCh];
    Tin d[kSeg][kCh];
    float dy[kSeg][kCh];
    Tin B[kSeg][kNP];
    Tin C[kSeg][kNP];
};

template <typename Tin>
struct Shared {
    // state entering each step of the segment, [step][channel][state]: a
    // lane's four states are one 16-byte access, and the eight lanes of a
    // quarter-warp (two channels) cover 128 contiguous bytes
    float hist[kSeg][kCh][kNP];
    float red[kWarps][kSeg][2 * kNP];     // per-warp sums of dB_t, dC_t over the warp's channels
    float fB[kSeg][kNP], fC[kSeg][kNP];   // the segment's B, C rows in fp32 (converted once)
    Stage<Tin> st[2];
};

// Stage rows [t0, t0 + kSeg) of the segment (rows past L and channels past
// ED zero filled).  VEC: 16-byte cp.async copies (the caller checked that
// every row start is 16-byte aligned).
template <typename Tin, bool VEC>
__device__ __forceinline__ void stage_segment(Stage<Tin> &s, const Tin *__restrict__ x,
                                              const Tin *__restrict__ dlt,
                                              const float *__restrict__ dy,
                                              const Tin *__restrict__ Bm, const Tin *__restrict__ Cm,
                                              int64_t b, int t0, int L, int e0, int ED, int N) {
    const int tid = threadIdx.x;
    const int rows = min(kSeg, L - t0);
    if constexpr (VEC) {
        constexpr int EPC = 16 / sizeof(Tin);
        constexpr int CPR = kCh / EPC;                 // chunks per x row
        for (int i = tid; i < kSeg * CPR; i += kThreads) {
            const int t = i / CPR, cc = i % CPR;
            const int e = e0 + cc * EPC;
            const bool ok = t < rows && e < ED;
            const int64_t g = ok ? (b * L + t0 + t) * ED + e : 0;
            cp_async16(&s.x[t][cc * EPC], x + g, ok ? 16 : 0);
            cp_async16(&s.d[t][cc * EPC], dlt + g, ok ? 16 : 0);
        }
        constexpr int CPRY = kCh / 4;
        for (int i = tid; i < kSeg * CPRY; i += kThreads) {
            const int t = i / CPRY, cc = i % CPRY;
            const int e = e0 + cc * 4;
            const bool ok = t < rows && e < ED;
            cp_async16(&s.dy[t][cc * 4], dy + (ok ? (b * L + t0 + t) * ED + e : 0), ok ? 16 : 0);
        }
        // B, C rows: N == 16 here, one contiguous block of rows * 16 values
        const int nchunk = kSeg * kNP / EPC;
        const int64_t base = (b * L + t0) * kNP;
        for (int i = tid; i < nchunk; i += kThreads) {
            const bool ok = i * EPC < rows * kNP;
            const int64_t g = ok ? base + int64_t(i) * EPC : 0;
            cp_async16(&s.B[0][0] + i * EPC, Bm + g, ok ? 16 : 0);
            cp_async16(&s.C[0][0] + i * EPC, Cm + g, ok ? 16 : 0);
        }
    } else {
        for (int i = tid; i < kSeg * kCh; i += kThreads) {
            const int t = i / kCh, cc = i % kCh;
            const int e = e0 + cc;
            const bool ok = t < rows && e < ED;
            const int64_t g = (b * L + t0 + t) * ED + e;
            s.x[t][cc] = ok ? x[g] : Tin(0.0f);
            s.d[t][cc] = ok ? dlt[g] : Tin(0.0f);
            s.dy[t][cc] = ok ? dy[g] : 0.0f;
        }
        for (int i = tid; i < kSeg * kNP; i += kThreads) {
            const int t = i / kNP, n = i % kNP;
            const bool ok = t < rows && n < N;
            const int64_t g = (b * L + t0 + t) * N + n;
            s.B[t][n] = ok ? Bm[g] : Tin(0.0f);
            s.C[t][n] = ok ? Cm[g] : Tin(0.0f);
        }
    }
}

// Reverse pass.  Per step t (channel e of batch row b), with hp = h_{t-1}
// and g = g_t:
//   dx_t     = sum_n g[n] delta_t B_t[n] + D[e] dy_t
//   ddelta_t = sum_n g[n] (A[e,n] a_t[n] hp[n] + B_t[n] x_t)
//   dA[e,n] += g[n] delta_t a_t[n] hp[n]
//   dB_t[n] += g[n] delta_t x_t        (summed over the channels e)
//   dC_t[n] += dy_t h_t[n]             (summed over the channels e)
//   dD[e]   += dy_t x_t
template <typename Tin, bool VEC>
__global__ void __launch_bounds__(kThreads)
diag_bwd_kernel(const Tin *__restrict__ x, const Tin *__restrict__ dlt, const float *__restrict__ A,
                const Tin *__restrict__ Bm, const Tin *__restrict__ Cm, const float *__restrict__ D,
                const float *__restrict__ dy, const float *__restrict__ ckpt,
                float *__restrict__ dx, float *__restrict__ ddelta, float *__restrict__ dA,
                float *__restrict__ dB, float *__restrict__ dC, float *__restrict__ dD, int Bs,
                int L, int ED, int N) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Shared<Tin> &sm = *reinterpret_cast<Shared<Tin> *>(smem_raw);
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int q = tid % kLanes;                      // states q*4 .. q*4+3
    const int cl = tid / kLanes;                     // channel within the CTA
    const int64_t b = blockIdx.y;
    const int e0 = blockIdx.x * kCh;
    const int e = e0 + cl;
    const bool e_ok = e < ED;
    const int ec = e_ok ? e : ED - 1;                // lanes past ED mirror a channel, add zero
    const int64_t c = b * ED + ec;
    const int64_t nch = int64_t(Bs) * ED;
    float A2[kSpl], An[kSpl], g[kSpl], lA[kSpl];
#pragma unroll
    for (int i = 0; i < kSpl; ++i) {
        const int n = q * kSpl + i;
        An[i] = n < N ? A[int64_t(ec) * N + n] : 0.0f;
        A2[i] = An[i] * SSM_LOG2E;
        g[i] = 0.0f;
        lA[i] = 0.0f;
    }
    const float Dv = D ? D[ec] : 0.0f;
    float lD = 0.0f;
    const int nseg = (L + kSeg - 1) / kSeg;

    stage_segment<Tin, VEC>(sm.st[(nseg - 1) & 1], x, dlt, dy, Bm, Cm, b, (nseg - 1) * kSeg, L, e0,
                            ED, N);
    cp_async_commit();
    for (int k = nseg - 1; k >= 0; --k) {
        Stage<Tin> &s = sm.st[k & 1];
        if (k > 0)
            stage_segment<Tin, VEC>(sm.st[(k - 1) & 1], x, dlt, dy, Bm, Cm, b, (k - 1) * kSeg, L,
                                    e0, ED, N);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();                              // segment k staged everywhere
        // B, C rows of the segment in fp32, once, instead of at every use
        for (int i = tid; i < kSeg * kNP; i += kThreads) {
            sm.fB[i / kNP][i % kNP] = to_f32(s.B[i / kNP][i % kNP]);
            sm.fC[i / kNP][i % kNP] = to_f32(s.C[i / kNP][i % kNP]);
        }
        __syncthreads();
        const int t0 = k * kSeg;
        const int tl = min(kSeg, L - t0);
        float h[kSpl];
        {
            const float4 v = *reinterpret_cast<const float4 *>(ckpt + (int64_t(k) * nch + c) * kNP +
                                                               q * kSpl);
            h[0] = v.x; h[1] = v.y; h[2] = v.z; h[3] = v.w;
        }
        // forward over the segment: keep the entering state of every step
        // (unrolled by 4: the next steps' exponentials overlap this step's chain)
#pragma unroll 4
        for (int j = 0; j < tl; ++j) {
            const float dl = to_f32(s.d[j][cl]), dlx = dl * to_f32(s.x[j][cl]);
            *reinterpret_cast<float4 *>(&sm.hist[j][cl][q * kSpl]) = make_float4(h[0], h[1], h[2], h[3]);
            const float4 b4 = *reinterpret_cast<const float4 *>(&sm.fB[j][q * kSpl]);
            const float bb[kSpl] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i = 0; i < kSpl; ++i) h[i] = fmaf(ex2(dl * A2[i]), h[i], dlx * bb[i]);
        }
        // backward over the segment
#pragma unroll 4
        for (int j = tl - 1; j >= 0; --j) {
            const float dl = to_f32(s.d[j][cl]), xv = to_f32(s.x[j][cl]);
            const float gy = s.dy[j][cl];                 // zero past ED
            float sdx = 0.0f, sdd = 0.0f, vb[kSpl], vc[kSpl];
            const float4 b4 = *reinterpret_cast<const float4 *>(&sm.fB[j][q * kSpl]);
            const float4 c4 = *reinterpret_cast<const float4 *>(&sm.fC[j][q * kSpl]);
            const float4 h4 = *reinterpret_cast<const float4 *>(&sm.hist[j][cl][q * kSpl]);
            const float bb[kSpl] = {b4.x, b4.y, b4.z, b4.w}, cc[kSpl] = {c4.x, c4.y, c4.z, c4.w},
                        hh[kSpl] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
            for (int i = 0; i < kSpl; ++i) {
                const float bv = bb[i], cv = cc[i];
                const float a = ex2(dl * A2[i]);
                const float hp = hh[i];
                g[i] = fmaf(gy, cv, g[i]);                      // g_t
                sdx = fmaf(g[i] * dl, bv, sdx);
                sdd = fmaf(g[i], fmaf(An[i] * a, hp, bv * xv), sdd);
                lA[i] = fmaf(g[i] * dl * a, hp, lA[i]);
                vb[i] = e_ok ? g[i] * dl * xv : 0.0f;           // share of dB_t[n]
                vc[i] = gy * fmaf(a, hp, dl * bv * xv);         // share of dC_t[n] (dy_t h_t[n])
                g[i] *= a;                                      // a_t g_t, for step t - 1
            }
            // the channel's four lanes hold disjoint states: sum their parts
            sdx += __shfl_xor_sync(0xffffffffu, sdx, 1);
            sdd += __shfl_xor_sync(0xffffffffu, sdd, 1);
            sdx += __shfl_xor_sync(0xffffffffu, sdx, 2);
            sdd += __shfl_xor_sync(0xffffffffu, sdd, 2);
            if (q == 0 && e_ok) {
                const int64_t i = (b * L + t0 + j) * ED + e;
                dx[i] = fmaf(Dv, gy, sdx);
                ddelta[i] = sdd;
                lD = fmaf(gy, xv, lD);
            }
            // Sum the 8 values (dB, dC shares of this lane's states) over the
            // warp's 8 channels (lane = 4 * channel + q) by halving exchanges:
            // at each level a lane keeps half of its values, adds the partner's
            // copy of that half and hands over the other half; after three
            // levels lane (channel c, q) holds the warp sum of value c.
            float v[8] = {vb[0], vb[1], vb[2], vb[3], vc[0], vc[1], vc[2], vc[3]};
#pragma unroll
            for (int lvl = 0, half = 4; lvl < 3; ++lvl, half >>= 1) {
                const bool hi = (lane >> (4 - lvl)) & 1;     // channel bit 2 - lvl
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float keep = hi ? v[i + half] : v[i];
                    const float give = hi ? v[i] : v[i + half];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, give, 16 >> lvl);
                }
            }
            {
                const int o = lane >> 2;                       // value index 0..7
                sm.red[warp][j][(o < 4 ? 0 : kNP) + q * kSpl + (o & 3)] = v[0];
            }
        }
        __syncthreads();                              // per-warp sums of the segment are in place
        // one atomic add per (t, n) for B and C
        for (int o = tid; o < tl * 2 * kNP; o += kThreads) {
            const int j = o / (2 * kNP), r = o % (2 * kNP);
            const int n = r % kNP;
            if (n >= N) continue;
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) sum += sm.red[w][j][r];
            atomicAdd((r < kNP ? dB : dC) + (b * L + t0 + j) * N + n, sum);
        }
        // the next iteration's staging (issued above) and this one's reads of
        // s, hist and red are ordered by the barrier at its top
    }
    cp_async_wait<0>();
    if (e_ok) {
#pragma unroll
        for (int i = 0; i < kSpl; ++i) {
            const int n = q * kSpl + i;
            if (n < N) atomicAdd(dA + int64_t(e) * N + n, lA[i]);
        }
        if (dD && q == 0) atomicAdd(dD + e, lD);
    }
}

// The gradients for at most kNP states.
template <typename Tin>
cudaError_t launch_bwd16(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm,
                         const Tin *Cm, const float *D, const float *dy, float *dx,
                         float *ddelta, float *dA, float *dB, float *dC, float *dD, int64_t Bs,
                         int64_t L, int64_t ED, int64_t N, int num_sms, cudaStream_t st) {
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
    // forward pass for the checkpoints (dx stands in for y, which is not written)
    ScanOpts fw{};
    fw.ckpt = ckpt;
    fw.no_y = 1;
    err = diag::launch_ext<Tin>(x, dlt, A, Bm, Cm, D, dx, Bs, L, ED, N, num_sms, fw, st);
    if (err == cudaSuccess) {
        const size_t esz = sizeof(Tin);
        const bool vec = N == kNP && (ED * esz) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(dlt) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(dy) % 16 == 0 && ED % 4 == 0 &&
                         reinterpret_cast<uintptr_t>(Bm) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(Cm) % 16 == 0;
        const int smem = int(sizeof(Shared<Tin>));
        auto kern = vec ? diag_bwd_kernel<Tin, true> : diag_bwd_kernel<Tin, false>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err == cudaSuccess) {
            kern<<<grid, kThreads, smem, st>>>(x, dlt, A, Bm, Cm, D, dy, ckpt, dx, ddelta, dA, dB,
                                               dC, dD, int(Bs), int(L), int(ED), int(N));
            err = cudaGetLastError();
        }
    }
    cudaError_t e2 = cudaFreeAsync(scratch, st);
    return err != cudaSuccess ? err : e2;
}

// More than kNP states.  The recurrence is separate per state n: y is a sum
// over n, so dx and ddelta are sums over groups of states, while dA, dB, dC
// hold one column per state and D enters once.  So the states are taken in
// groups of kNP: each group's columns of A, B and C are gathered into
// contiguous scratch, its gradients formed by launch_bwd16 (D and dD with the
// first group only), its columns of dA, dB, dC scattered back, and its dx,
// ddelta added to the first group's in group order (deterministic).
namespace {
constexpr int kElemThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kElemThreads)
gather_cols(const T *__restrict__ src, T *__restrict__ dst, int64_t rows, int N, int n0, int ng) {
    const int64_t n = rows * ng;
    for (int64_t i = blockIdx.x * int64_t(kElemThreads) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * kElemThreads) {
        const int64_t r = i / ng;
        dst[i] = src[r * N + n0 + (i - r * ng)];
    }
}

__global__ void __launch_bounds__(kElemThreads)
scatter_cols(const float *__restrict__ src, float *__restrict__ dst, int64_t rows, int N, int n0,
             int ng) {
    const int64_t n = rows * ng;
    for (int64_t i = blockIdx.x * int64_t(kElemThreads) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * kElemThreads) {
        const int64_t r = i / ng;
        dst[r * N + n0 + (i - r * ng)] = src[i];
    }
}

__global__ void __launch_bounds__(kElemThreads)
add_into(float *__restrict__ dst, const float *__restrict__ src, int64_t n) {
    for (int64_t i = blockIdx.x * int64_t(kElemThreads) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * kElemThreads)
        dst[i] += src[i];
}

unsigned elem_grid(int64_t n, int num_sms) {
    const int64_t want = (n + kElemThreads - 1) / kElemThreads;
    const int64_t cap = int64_t(num_sms) * 8;
    return unsigned(want < 1 ? 1 : (want < cap ? want : cap));
}
}  // namespace

template <typename Tin>
cudaError_t launch_bwd(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                       const float *D, const float *dy, float *dx, float *ddelta, float *dA,
                       float *dB, float *dC, float *dD, int64_t Bs, int64_t L, int64_t ED,
                       int64_t N, int num_sms, cudaStream_t st) {
    if (N <= kNP)
        return launch_bwd16<Tin>(x, dlt, A, Bm, Cm, D, dy, dx, ddelta, dA, dB, dC, dD, Bs, L, ED, N,
                                 num_sms, st);
    if (Bs > 65535) return cudaErrorInvalidConfiguration;
    const int64_t rows = Bs * L, nx = rows * ED;
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t bytes = up(size_t(ED) * kNP * 4) * 2 + up(size_t(rows) * kNP * sizeof(Tin)) * 2 +
                         up(size_t(rows) * kNP * 4) * 2 + up(size_t(nx) * 4) * 2;
    void *scratch = nullptr;
    cudaError_t err = cudaMallocAsync(&scratch, bytes, st);
    if (err != cudaSuccess) return err;
    char *cur = static_cast<char *>(scratch);
    auto take = [&](size_t b) { char *p = cur; cur += up(b); return p; };
    float *Ag = reinterpret_cast<float *>(take(size_t(ED) * kNP * 4));
    float *dAg = reinterpret_cast<float *>(take(size_t(ED) * kNP * 4));
    Tin *Bg = reinterpret_cast<Tin *>(take(size_t(rows) * kNP * sizeof(Tin)));
    Tin *Cg = reinterpret_cast<Tin *>(take(size_t(rows) * kNP * sizeof(Tin)));
    float *dBg = reinterpret_cast<float *>(take(size_t(rows) * kNP * 4));
    float *dCg = reinterpret_cast<float *>(take(size_t(rows) * kNP * 4));
    float *dxg = reinterpret_cast<float *>(take(size_t(nx) * 4));
    float *ddg = reinterpret_cast<float *>(take(size_t(nx) * 4));
    for (int64_t n0 = 0; n0 < N && err == cudaSuccess; n0 += kNP) {
        const int ng = int(N - n0 < kNP ? N - n0 : kNP);
        const bool first = n0 == 0;
        gather_cols<float><<<elem_grid(ED * ng, num_sms), kElemThreads, 0, st>>>(A, Ag, ED, int(N),
                                                                               int(n0), ng);
        gather_cols<Tin><<<elem_grid(rows * ng, num_sms), kElemThreads, 0, st>>>(Bm, Bg, rows,
                                                                               int(N), int(n0), ng);
        gather_cols<Tin><<<elem_grid(rows * ng, num_sms), kElemThreads, 0, st>>>(Cm, Cg, rows,
                                                                               int(N), int(n0), ng);
        err = cudaGetLastError();
        if (err != cudaSuccess) break;
        err = launch_bwd16<Tin>(x, dlt, Ag, Bg, Cg, first ? D : nullptr, dy, first ? dx : dxg,
                                first ? ddelta : ddg, dAg, dBg, dCg, first ? dD : nullptr, Bs, L,
                                ED, ng, num_sms, st);
        if (err != cudaSuccess) break;
        scatter_cols<<<elem_grid(ED * ng, num_sms), kElemThreads, 0, st>>>(dAg, dA, ED, int(N),
                                                                           int(n0), ng);
        scatter_cols<<<elem_grid(rows * ng, num_sms), kElemThreads, 0, st>>>(dBg, dB, rows, int(N),
                                                                             int(n0), ng);
        scatter_cols<<<elem_grid(rows * ng, num_sms), kElemThreads, 0, st>>>(dCg, dC, rows, int(N),
                                                                             int(n0), ng);
        if (!first) {
            add_into<<<elem_grid(nx, num_sms), kElemThreads, 0, st>>>(dx, dxg, nx);
            add_into<<<elem_grid(nx, num_sms), kElemThreads, 0, st>>>(ddelta, ddg, nx);
        }
        err = cudaGetLastError();
    }
    cudaError_t e2 = cudaFreeAsync(scratch, st);
    return err != cudaSuccess ? err : e2;
}

template cudaError_t launch_bwd<float>(const float *, const float *, const float *, const float *,
                                       const float *, const float *, const float *, float *,
                                       float *, float *, float *, float *, float *, int64_t,
                                       int64_t, int64_t, int64_t, int, cudaStream_t);
template cudaError_t launch_bwd<__nv_bfloat16>(const __nv_bfloat16 *, const __nv_bfloat16 *,
                                               const float *, const __nv_bfloat16 *,
                                               const __nv_bfloat16 *, const float *, const float *,
                                               float *, float *, float *, float *, float *,
                                               float *, int64_t, int64_t, int64_t, int64_t, int,
                                               cudaStream_t);

}  // namespace diag_bwd
}  // namespace ssm
