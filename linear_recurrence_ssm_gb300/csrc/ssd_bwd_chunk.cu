// ssd_bwd_chunk.cu -- gradients of the chunked scalar-decay ("SSD") scan in
// chunked form on CUDA cores, for head size P = 64 and N = 64 or 128 states:
// dx, ddt, dA, dB, dC, dD for an upstream gradient dy, both directions of the
// bidirectional scan and groups of B, C -- the outputs of the chunked
// backward pass named in "Some questions of Bi-Mamba2 and Hydra" (Bi-Mamba2
// issue 1).
//
// One direction, per (b, h), walk order (t for the forward direction, L-1-t
// for the reversed one), chunks of Q steps with cum_t = sum_{r <= t} dt_r A
// inside the chunk (inclusive) and tot = cum at the chunk's last step:
//   state entering chunk k:   S(k+1) = e^{tot_k} S(k) + sum_s e^{tot_k - cum_s} dt_s x_s B_s^T
//   adjoint leaving chunk k:  Gin(k) = e^{tot_{k+1}} Gin(k+1) + sum_{u in k+1} e^{cum_u} dy_u C_u^T
// and inside the chunk, with L(u,s) = e^{cum_u - cum_s} [u >= s]:
//   v_s   = G_s B_s = sum_u L(u,s) (C_u . B_s) dy_u + e^{tot - cum_s} Gin B_s
//   dx_s  = dt_s v_s (+ D dy_s once),          ddt1_s = x_s . v_s
//   dB_s  = dt_s [sum_u L(u,s) (dy_u . x_s) C_u + e^{tot - cum_s} Gin^T x_s]
//   dC_t  = sum_s L(t,s) dt_s (dy_t . x_s) B_s + e^{cum_t} S^T dy_t
//   yt_t  = sum_s L(t,s) dt_s (C_t . B_s) x_s + e^{cum_t} S C_t     (the output without D)
// where G_s is the adjoint of the state after step s.  dt enters through the
// input term (ddt1) and through dA_r = dt_r A.  For the latter,
// dL/ddA_r = a_r <G_r, H_{r-1}> = <G_r, H_r> - dt_r ddt1_r, and the adjoint
// recursion turns <G_r, H_r> into a suffix sum, so that
//   dL/ddA_r = sum_{u >= r} q_u,   q_u = dy_u . yt_u - dt_u ddt1_u,
//   ddt_r = ddt1_r + A dL/ddA_r,   dA = sum_r dt_r dL/ddA_r
// -- per-step scalars only: no state of any step but the chunks' entering
// ones is formed.
//
// Four kernels per direction: chunk-local products (the two sums of the
// chunk recursions), a scan over the chunks per (b, h) and state element,
// the per-chunk gradients (ten products from shared memory, fp32 on CUDA
// cores), and the suffix sums of q.  Scratch: the chunks' states and
// adjoints, 2 Bs H ceil(L/Q) P N fp32, plus q and the chunk totals.  dB, dC,
// dA, dD are added with atomics (their last bits may differ between runs).
#include "ssm_common.cuh"

namespace ssm {
namespace ssd_bwd_chunk {

constexpr int kQ = 64;         // steps per chunk
constexpr int kP = 64;         // head dimension served here
constexpr int kThreads = 256;  // a 16 x 16 grid of threads over every product
constexpr int kPad = 4;        // fp32 padding of a shared-memory row

template <typename Tin>
struct Args {
    const Tin *x, *dt, *B, *C;
    const float *A, *D, *dy;
    float *dx, *ddt, *dA, *dB, *dC, *dD;
    float *Sx;      // [Bs H][nc][P N]: chunk-local states, then the entering states
    float *Ux;      // [Bs H][nc][P N]: chunk-local adjoint sums, then the incoming adjoints
    float *tot;     // [Bs H][nc]: sum of dt A over each chunk (log2 units)
    float *q;       // [Bs H][L] in walk order
    int L, H, G, nc;
};

__device__ __forceinline__ int walk_row(int lam, int L, int dir) { return dir ? L - 1 - lam : lam; }

// Output column c of a thread at column index tj (0..15) of the 16 x 16
// thread grid.  IL (interleaved): j = tj + 16 c, so that the 16 threads of a
// row group read 16 consecutive rows or columns (no bank conflicts when the
// operand's contiguous index is k); otherwise groups of four consecutive
// columns, the groups of the 16 threads side by side: j = 4 tj + 64 (c / 4)
// + c % 4 (float4 loads along j without bank conflicts).
template <bool IL>
__device__ __forceinline__ int colj(int tj, int c) {
    return IL ? tj + 16 * c : 4 * tj + 64 * (c >> 2) + (c & 3);
}

// acc[r][c] += sum_k A(i0 + r, k) B(k, colj(tj, c)), k = 0 .. K-1 (K a
// multiple of 4), from shared memory: A(i, k) = a[i sa + k] if AK (k
// contiguous) else a[k sa + i]; B(k, j) = b[j sb + k] if BK else b[k sb + j]
// (BK requires IL).  Loads are float4 along the contiguous index, four k at a
// time, except B with j contiguous and IL: four scalars per k.
template <int K, int TN, bool AK, bool BK, bool IL>
__device__ __forceinline__ void mm(float (&acc)[4][TN], const float *a, int sa, const float *b,
                                   int sb, int i0, int tj) {
    static_assert(!BK || IL, "k-contiguous B operands are read interleaved");
    static_assert(K % 4 == 0, "K is taken four at a time");
    // (K known at compile time: the loop is unrolled, so the loads of the
    // next four k overlap the multiply-adds of these)
#pragma unroll 4
    for (int k = 0; k < K; k += 4) {
        float av[4][4];   // av[r][kk] = A(i0 + r, k + kk)
        if (AK) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float4 v = *reinterpret_cast<const float4 *>(a + (i0 + r) * sa + k);
                av[r][0] = v.x; av[r][1] = v.y; av[r][2] = v.z; av[r][3] = v.w;
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 v = *reinterpret_cast<const float4 *>(a + (k + kk) * sa + i0);
                av[0][kk] = v.x; av[1][kk] = v.y; av[2][kk] = v.z; av[3][kk] = v.w;
            }
        }
        float bv[4][TN];  // bv[kk][c] = B(k + kk, colj(tj, c))
        if (BK) {
#pragma unroll
            for (int c = 0; c < TN; ++c) {
                const float4 v = *reinterpret_cast<const float4 *>(b + (tj + 16 * c) * sb + k);
                bv[0][c] = v.x; bv[1][c] = v.y; bv[2][c] = v.z; bv[3][c] = v.w;
            }
        } else if (IL) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int c = 0; c < TN; ++c) bv[kk][c] = b[(k + kk) * sb + tj + 16 * c];
        } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int c4 = 0; c4 < TN / 4; ++c4) {
                    const float4 v = *reinterpret_cast<const float4 *>(b + (k + kk) * sb + 4 * tj + 64 * c4);
                    bv[kk][4 * c4] = v.x; bv[kk][4 * c4 + 1] = v.y;
                    bv[kk][4 * c4 + 2] = v.z; bv[kk][4 * c4 + 3] = v.w;
                }
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < TN; ++c) acc[r][c] = fmaf(av[r][kk], bv[kk][c], acc[r][c]);
    }
}

template <int R, int C>
__device__ __forceinline__ void zero(float (&v)[R][C]) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) v[r][c] = 0.0f;
}

// Sum over the 16 threads of a row group (consecutive lanes).
__device__ __forceinline__ float row_sum16(float v) {
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 16 bytes of Tin as fp32 (8 bf16 or 4 floats) into shared memory.
__device__ __forceinline__ void put16(float *dst, uint4 v, const __nv_bfloat16 *) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        dst[2 * i] = __uint_as_float(w[i] << 16);
        dst[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void put16(float *dst, uint4 v, const float *) {
    *reinterpret_cast<uint4 *>(dst) = v;
}

// Rows of chunk k (walk order) into shared memory: x, dy [Q][P], B, C
// [Q][N] (fp32, padded rows), dt [Q]; rows past L are zero.  Global reads
// are 16 bytes wide (x, dy, B, C are 16-byte aligned: checked by the caller).
template <typename Tin, int N>
__device__ __forceinline__ void load_chunk(const Args<Tin> &a, int dir, int b, int h, int g,
                                           int k, float *X, float *DY, float *Bs, float *Cs,
                                           float *dtv, bool with_dy, bool with_b, bool with_c) {
    constexpr int ldP = kP + kPad, ldN = N + kPad;
    constexpr int EV = 16 / sizeof(Tin);   // input elements per 16 bytes
    const int L = a.L, H = a.H, G = a.G;
    for (int i = threadIdx.x; i < kQ * kP / EV; i += kThreads) {
        const int r = i / (kP / EV), p = (i % (kP / EV)) * EV;
        const int lam = k * kQ + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (lam < L) {
            const size_t o = (size_t(b) * L + walk_row(lam, L, dir)) * H + h;
            v = *reinterpret_cast<const uint4 *>(a.x + o * kP + p);
        }
        put16(X + r * ldP + p, v, a.x);
    }
    if (with_dy) {
        for (int i = threadIdx.x; i < kQ * kP / 4; i += kThreads) {
            const int r = i / (kP / 4), p = (i % (kP / 4)) * 4;
            const int lam = k * kQ + r;
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (lam < L) {
                const size_t o = (size_t(b) * L + walk_row(lam, L, dir)) * H + h;
                v = *reinterpret_cast<const float4 *>(a.dy + o * kP + p);
            }
            *reinterpret_cast<float4 *>(DY + r * ldP + p) = v;
        }
    }
    for (int i = threadIdx.x; i < kQ * N / EV; i += kThreads) {
        const int r = i / (N / EV), n = (i % (N / EV)) * EV;
        const int lam = k * kQ + r;
        uint4 bv = make_uint4(0u, 0u, 0u, 0u), cv = bv;
        if (lam < L) {
            const size_t o = ((size_t(b) * L + walk_row(lam, L, dir)) * G + g) * N + n;
            if (with_b) bv = *reinterpret_cast<const uint4 *>(a.B + o);
            if (with_c) cv = *reinterpret_cast<const uint4 *>(a.C + o);
        }
        if (with_b) put16(Bs + r * ldN + n, bv, a.B);
        if (with_c) put16(Cs + r * ldN + n, cv, a.C);
    }
    for (int r = threadIdx.x; r < kQ; r += kThreads) {
        const int lam = k * kQ + r;
        dtv[r] = lam < L ? to_f32(a.dt[(size_t(b) * L + walk_row(lam, L, dir)) * H + h]) : 0.0f;
    }
}

// Inclusive sums of dt A (log2 units) over the chunk's rows: threads 0..63,
// two warps, each a shuffle scan, the first warp's total added to the second.
__device__ __forceinline__ void chunk_cumsum(const float *dtv, float A2, float *cum, float *wtot) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < kQ) {
        float v = dtv[tid] * A2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        cum[tid] = v;
        if (tid == 31) *wtot = v;
    }
    __syncthreads();
    if (tid >= 32 && tid < kQ) cum[tid] += *wtot;
    __syncthreads();
}

// ---- kernel 1: chunk-local sums -----------------------------------------------------------
// Sloc[p][n] = sum_s dt_s e^{tot - cum_s} x_s[p] B_s[n],  Uloc[p][n] = sum_u e^{cum_u} dy_u[p] C_u[n].
template <typename Tin, int N>
__global__ void __launch_bounds__(kThreads)
chunk_local_kernel(const Args<Tin> a, int dir) {
    constexpr int ldP = kP + kPad, ldN = N + kPad, TN = N / 16;
    extern __shared__ __align__(16) float sm[];
    float *X = sm, *DY = X + kQ * ldP, *Bs = DY + kQ * ldP, *Cs = Bs + kQ * ldN;
    float *dtv = Cs + kQ * ldN, *cum = dtv + kQ, *wtot = cum + kQ;
    const int bh = blockIdx.x / a.nc, k = blockIdx.x % a.nc;
    const int b = bh / a.H, h = bh % a.H, g = h / (a.H / a.G);
    const int tid = threadIdx.x, i0 = 4 * (tid >> 4), tj = tid & 15;
    load_chunk<Tin, N>(a, dir, b, h, g, k, X, DY, Bs, Cs, dtv, true, true, true);
    __syncthreads();
    chunk_cumsum(dtv, a.A[h] * SSM_LOG2E, cum, wtot);
    const float tot = cum[kQ - 1];
    // weigh the rows: x_s by dt_s e^{tot - cum_s}, dy_u by e^{cum_u}
    for (int i = tid; i < kQ * kP; i += kThreads) {
        const int r = i / kP, p = i % kP;
        X[r * ldP + p] *= dtv[r] * ex2(tot - cum[r]);
        DY[r * ldP + p] *= ex2(cum[r]);
    }
    __syncthreads();
    const size_t base = (size_t(bh) * a.nc + k) * kP * N;
    float acc[4][TN];
    zero(acc);
    mm<kQ, TN, false, false, false>(acc, X, ldP, Bs, ldN, i0, tj);   // A(p, s) = X[s][p], B(s, n) = B[s][n]
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c4 = 0; c4 < TN / 4; ++c4)
            *reinterpret_cast<float4 *>(a.Sx + base + (i0 + r) * N + 4 * tj + 64 * c4) =
                make_float4(acc[r][4 * c4], acc[r][4 * c4 + 1], acc[r][4 * c4 + 2], acc[r][4 * c4 + 3]);
    zero(acc);
    mm<kQ, TN, false, false, false>(acc, DY, ldP, Cs, ldN, i0, tj);  // A(p, u) = DY[u][p], B(u, n) = C[u][n]
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c4 = 0; c4 < TN / 4; ++c4)
            *reinterpret_cast<float4 *>(a.Ux + base + (i0 + r) * N + 4 * tj + 64 * c4) =
                make_float4(acc[r][4 * c4], acc[r][4 * c4 + 1], acc[r][4 * c4 + 2], acc[r][4 * c4 + 3]);
    if (tid == 0) a.tot[size_t(bh) * a.nc + k] = tot;
}

// ---- kernel 2: the chunk recursions, per (b, h) and state element --------------------------
// Sx[k] <- S(k) (entering chunk k), Ux[k] <- Gin(k) (leaving chunk k).
__global__ void __launch_bounds__(kThreads)
chunk_scan_kernel(float *Sx, float *Ux, const float *tot, int nc, int PN) {
    const int bh = blockIdx.y;
    const int e = blockIdx.x * kThreads + threadIdx.x;
    if (e >= PN) return;
    const float *tb = tot + size_t(bh) * nc;
    float *sp = Sx + size_t(bh) * nc * PN + e;
    float *up = Ux + size_t(bh) * nc * PN + e;
    // (a batch of chunks is read before any of it is written: the loads of a
    // batch are in flight together)
    constexpr int kB = 16;
    float loc[kB];
    float s = 0.0f;
    for (int k0 = 0; k0 < nc; k0 += kB) {
#pragma unroll
        for (int j = 0; j < kB; ++j)
            if (k0 + j < nc) loc[j] = sp[size_t(k0 + j) * PN];
#pragma unroll
        for (int j = 0; j < kB; ++j)
            if (k0 + j < nc) {
                sp[size_t(k0 + j) * PN] = s;
                s = fmaf(ex2(tb[k0 + j]), s, loc[j]);
            }
    }
    float gv = 0.0f;
    for (int k1 = nc - 1; k1 >= 0; k1 -= kB) {
#pragma unroll
        for (int j = 0; j < kB; ++j)
            if (k1 - j >= 0) loc[j] = up[size_t(k1 - j) * PN];
#pragma unroll
        for (int j = 0; j < kB; ++j)
            if (k1 - j >= 0) {
                up[size_t(k1 - j) * PN] = gv;
                gv = fmaf(ex2(tb[k1 - j]), gv, loc[j]);
            }
    }
}

// ---- kernel 3: the gradients of one chunk -------------------------------------------------
template <typename Tin, int N>
struct GradSmem {
    static constexpr int ldP = kP + kPad, ldN = N + kPad, ldQ = kQ + kPad;
    static constexpr size_t floats = size_t(2) * kQ * ldP + size_t(2) * kQ * ldN +
                                     size_t(2) * kP * ldN + size_t(2) * kQ * ldQ + 6 * kQ + 8;
    static constexpr size_t bytes = floats * sizeof(float);
};

template <typename Tin, int N>
__global__ void __launch_bounds__(kThreads, 1)
chunk_grad_kernel(const Args<Tin> a, int dir) {
    using Sm = GradSmem<Tin, N>;
    constexpr int ldP = Sm::ldP, ldN = Sm::ldN, ldQ = Sm::ldQ, TN = N / 16;
    extern __shared__ __align__(16) float sm[];
    float *X = sm, *DY = X + kQ * ldP, *Bs = DY + kQ * ldP, *Cs = Bs + kQ * ldN;
    float *S = Cs + kQ * ldN, *Gi = S + kP * ldN, *GL = Gi + kP * ldN, *WL = GL + kQ * ldQ;
    float *dtv = WL + kQ * ldQ, *cum = dtv + kQ, *eo = cum + kQ, *ec = eo + kQ, *d1 = ec + kQ;
    float *wtot = d1 + kQ, *part = wtot + 1;
    const int L = a.L, H = a.H, G = a.G;
    const int bh = blockIdx.x / a.nc, k = blockIdx.x % a.nc;
    const int b = bh / H, h = bh % H, g = h / (H / G);
    const int tid = threadIdx.x, lane = tid & 31, ti = tid >> 4, tj = tid & 15, i0 = 4 * ti;
    const float Dh = (dir == 0 && a.D) ? a.D[h] : 0.0f;

    {   // the entering state and the incoming adjoint, [p][n]: asynchronous
        // copies, first needed after the masked products below
        const size_t base = (size_t(bh) * a.nc + k) * kP * N;
        for (int i = tid; i < kP * N / 4; i += kThreads) {
            const int p = (4 * i) / N, n = (4 * i) % N;
            cp_async16(S + p * ldN + n, a.Sx + base + 4 * i, 16);
            cp_async16(Gi + p * ldN + n, a.Ux + base + 4 * i, 16);
        }
        cp_async_commit();
    }
    load_chunk<Tin, N>(a, dir, b, h, g, k, X, DY, Bs, Cs, dtv, true, true, true);
    __syncthreads();
    chunk_cumsum(dtv, a.A[h] * SSM_LOG2E, cum, wtot);
    const float tot = cum[kQ - 1];
    if (tid < kQ) {
        eo[tid] = ex2(tot - cum[tid]);
        ec[tid] = ex2(cum[tid]);
    }
    // GL = (C B^T) o L, WL = (dY X^T) o L
    {
        float acc[4][4];
        zero(acc);
        mm<N, 4, true, true, true>(acc, Cs, ldN, Bs, ldN, i0, tj);   // A(u, n) = C[u][n], B(n, s) = B[s][n]
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int u = i0 + r, s = colj<true>(tj, c);
                GL[u * ldQ + s] = u >= s ? acc[r][c] * ex2(cum[u] - cum[s]) : 0.0f;
            }
        zero(acc);
        mm<kP, 4, true, true, true>(acc, DY, ldP, X, ldP, i0, tj);   // A(u, p) = dy[u][p], B(p, s) = x[s][p]
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int u = i0 + r, s = colj<true>(tj, c);
                WL[u * ldQ + s] = u >= s ? acc[r][c] * ex2(cum[u] - cum[s]) : 0.0f;
            }
    }
    cp_async_wait<0>();                  // this thread's copies of S and Gin have landed
    __syncthreads();
    // v = GL^T dY + eo o (B Gin^T): dx and ddt1 = x . v
    {
        float v[4][4], w[4][4];
        zero(v);
        zero(w);
        mm<kQ, 4, false, false, true>(v, GL, ldQ, DY, ldP, i0, tj);  // A(s, u) = GL[u][s], B(u, p) = dy[u][p]
        mm<N, 4, true, true, true>(w, Bs, ldN, Gi, ldN, i0, tj);     // A(s, n) = B[s][n], B(n, p) = Gin[p][n]
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int s = i0 + r, lam = k * kQ + s;
            float sum = 0.0f, o[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int p = colj<true>(tj, c);
                const float vv = fmaf(eo[s], w[r][c], v[r][c]);
                sum = fmaf(X[s * ldP + p], vv, sum);
                o[c] = fmaf(Dh, DY[s * ldP + p], dtv[s] * vv);
            }
            sum = row_sum16(sum);
            if (tj == 0) d1[s] = sum;
            if (lam < L) {
                float *dst = a.dx + ((size_t(b) * L + walk_row(lam, L, dir)) * H + h) * kP;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int p = colj<true>(tj, c);
                    dst[p] = dir ? dst[p] + o[c] : o[c];
                }
            }
        }
    }
    // dB = dt o (WL^T C + eo o (X Gin))
    {
        float u1[4][TN], u2[4][TN];
        zero(u1);
        zero(u2);
        mm<kQ, TN, false, false, false>(u1, WL, ldQ, Cs, ldN, i0, tj);  // A(s, u) = WL[u][s], B(u, n) = C[u][n]
        mm<kP, TN, true, false, false>(u2, X, ldP, Gi, ldN, i0, tj);    // A(s, p) = x[s][p], B(p, n) = Gin[p][n]
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int s = i0 + r, lam = k * kQ + s;
            if (lam >= L) continue;
            float *dst = a.dB + ((size_t(b) * L + walk_row(lam, L, dir)) * G + g) * N;
#pragma unroll
            for (int c = 0; c < TN; ++c)
                atomicAdd(dst + colj<false>(tj, c), dtv[s] * fmaf(eo[s], u2[r][c], u1[r][c]));
        }
    }
    __syncthreads();
    // columns of GL and WL times dt_s
    for (int i = tid; i < kQ * kQ; i += kThreads) {
        const int u = i / kQ, s = i % kQ;
        GL[u * ldQ + s] *= dtv[s];
        WL[u * ldQ + s] *= dtv[s];
    }
    __syncthreads();
    // dC = (WL dt) B + ec o (dY S)
    {
        float u1[4][TN], u2[4][TN];
        zero(u1);
        zero(u2);
        mm<kQ, TN, true, false, false>(u1, WL, ldQ, Bs, ldN, i0, tj);   // A(t, s) = WL[t][s] dt_s, B(s, n) = B[s][n]
        mm<kP, TN, true, false, false>(u2, DY, ldP, S, ldN, i0, tj);    // A(t, p) = dy[t][p], B(p, n) = S[p][n]
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = i0 + r, lam = k * kQ + t;
            if (lam >= L) continue;
            float *dst = a.dC + ((size_t(b) * L + walk_row(lam, L, dir)) * G + g) * N;
#pragma unroll
            for (int c = 0; c < TN; ++c) atomicAdd(dst + colj<false>(tj, c), fmaf(ec[t], u2[r][c], u1[r][c]));
        }
    }
    // the output without D, yt = (GL dt) X + ec o (C S^T); q = dy . yt - dt ddt1
    {
        float y1[4][4], y2[4][4];
        zero(y1);
        zero(y2);
        mm<kQ, 4, true, false, true>(y1, GL, ldQ, X, ldP, i0, tj);    // A(t, s) = GL[t][s] dt_s, B(s, p) = x[s][p]
        mm<N, 4, true, true, true>(y2, Cs, ldN, S, ldN, i0, tj);      // A(t, n) = C[t][n], B(n, p) = S[p][n]
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = i0 + r, lam = k * kQ + t;
            float sum = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                sum = fmaf(DY[t * ldP + colj<true>(tj, c)], fmaf(ec[t], y2[r][c], y1[r][c]), sum);
            sum = row_sum16(sum);
            if (tj == 0 && lam < L) {
                a.q[size_t(bh) * L + lam] = sum - dtv[t] * d1[t];
                float *dd = a.ddt + (size_t(b) * L + walk_row(lam, L, dir)) * H + h;
                *dd = dir ? *dd + d1[t] : d1[t];
            }
        }
    }
    // dD (once): sum of dy . x over the chunk
    if (dir == 0 && a.dD) {
        float sdd = 0.0f;
        for (int i = tid; i < kQ * kP; i += kThreads) sdd = fmaf(DY[(i / kP) * ldP + i % kP], X[(i / kP) * ldP + i % kP], sdd);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sdd += __shfl_xor_sync(0xffffffffu, sdd, o);
        if (lane == 0) part[tid >> 5] = sdd;
        __syncthreads();
        if (tid == 0) {
            float t8 = 0.0f;
            for (int w = 0; w < kThreads / 32; ++w) t8 += part[w];
            atomicAdd(a.dD + h, t8);
        }
    }
}

// ---- kernel 4: suffix sums of q: the dt A parts of ddt and dA ---------------------------
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
finish_kernel(const Args<Tin> a, int dir) {
    __shared__ float tsum[kThreads];
    __shared__ float wred[kThreads / 32];
    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int L = a.L, tid = threadIdx.x, lane = tid & 31;
    const int per = (L + kThreads - 1) / kThreads;
    const int l0 = min(L, tid * per), l1 = min(L, l0 + per);
    const float *qb = a.q + size_t(bh) * L;
    float loc = 0.0f;
    for (int l = l0; l < l1; ++l) loc += qb[l];
    tsum[tid] = loc;
    __syncthreads();
    // the sum of q over the blocks after this thread's (a serial pass over
    // 256 values by one warp's lanes would be shorter; 256 adds are cheap)
    float after = 0.0f;
    for (int j = tid + 1; j < kThreads; ++j) after += tsum[j];
    const float A = a.A[h];
    float run = after, da = 0.0f;
    for (int l = l1 - 1; l >= l0; --l) {
        run += qb[l];
        const size_t o = (size_t(b) * L + walk_row(l, L, dir)) * a.H + h;
        a.ddt[o] = fmaf(A, run, a.ddt[o]);
        da = fmaf(to_f32(a.dt[o]), run, da);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) da += __shfl_xor_sync(0xffffffffu, da, o);
    if (lane == 0) wred[tid >> 5] = da;
    __syncthreads();
    if (tid == 0) {
        float s = 0.0f;
        for (int w = 0; w < kThreads / 32; ++w) s += wred[w];
        atomicAdd(a.dA + h, s);
    }
}

template <typename Tin, int N>
static cudaError_t run(const Args<Tin> &a, int64_t nbh, bool bidir, cudaStream_t st) {
    const size_t smem1 = (size_t(2) * kQ * (kP + kPad) + size_t(2) * kQ * (N + kPad) + 2 * kQ + 8) * sizeof(float);
    const size_t smem3 = GradSmem<Tin, N>::bytes;
    cudaError_t e = cudaFuncSetAttribute(chunk_local_kernel<Tin, N>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem1));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(chunk_grad_kernel<Tin, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem3));
    if (e != cudaSuccess) return e;
    const unsigned units = unsigned(nbh * a.nc);
    const dim3 sgrid(unsigned((kP * N + kThreads - 1) / kThreads), unsigned(nbh));
    for (int dir = 0; dir < (bidir ? 2 : 1); ++dir) {
        chunk_local_kernel<Tin, N><<<units, kThreads, smem1, st>>>(a, dir);
        chunk_scan_kernel<<<sgrid, kThreads, 0, st>>>(a.Sx, a.Ux, a.tot, a.nc, kP * N);
        chunk_grad_kernel<Tin, N><<<units, kThreads, smem3, st>>>(a, dir);
        finish_kernel<Tin><<<unsigned(nbh), kThreads, 0, st>>>(a, dir);
    }
    return cudaGetLastError();
}

bool supported(int64_t P, int64_t N) { return P == kP && (N == 64 || N == 128); }

template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dt, const float *A_head, const Tin *Bm, const Tin *Cm,
                   const float *D, const float *dy, float *dx, float *ddt, float *dA, float *dB,
                   float *dC, float *dD, int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                   int64_t G, bool bidir, cudaStream_t st) {
    if (!supported(P, N) || G < 1 || H % G != 0) return cudaErrorNotSupported;
    const int64_t nbh = Bs * H, nc = (L + kQ - 1) / kQ;
    if (nbh > 65535 || nbh * nc > 0x7fffffff || L > 0x7fffffff) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaMemsetAsync(dA, 0, size_t(H) * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, size_t(Bs * L * G * N) * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dC, 0, size_t(Bs * L * G * N) * sizeof(float), st);
    if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, size_t(H) * sizeof(float), st);
    if (e != cudaSuccess) return e;
    const size_t states = size_t(nbh) * nc * P * N;
    const size_t bytes = (2 * states + size_t(nbh) * nc + size_t(nbh) * L) * sizeof(float);
    void *scratch = nullptr;
    e = cudaMallocAsync(&scratch, bytes, st);
    if (e != cudaSuccess) return e;
    float *f = static_cast<float *>(scratch);
    Args<Tin> a{x, dt, Bm, Cm, A_head, D, dy, dx, ddt, dA, dB, dC, dD,
                f, f + states, f + 2 * states, f + 2 * states + nbh * nc,
                int(L), int(H), int(G), int(nc)};
    e = N == 64 ? run<Tin, 64>(a, nbh, bidir, st) : run<Tin, 128>(a, nbh, bidir, st);
    const cudaError_t e2 = cudaFreeAsync(scratch, st);
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

}  // namespace ssd_bwd_chunk
}  // namespace ssm
