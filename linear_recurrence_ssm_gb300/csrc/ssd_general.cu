// ssd_general.cu -- the chunked scalar-decay ("SSD") scan on CUDA cores, for
// the shapes and input types the tensor-core kernel (ssd_chunk_scan.cu: bf16,
// P = 64, N in {64, 128}) does not take: fp32 inputs, P and N in
// {16, 32, 64, 128, 256}.
//
// Per (b, h), with H_t the P x N state,
//     H_t = exp(dt_t A_h) H_{t-1} + dt_t x_t (outer) B_t,   y_t = H_t C_t + D_h x_t,
// walked sequentially over t with the state in registers.  Rows p of the
// state are independent of one another (they share only dt, B and C), so the
// P rows are cut into slices of PS = min(P, 128) rows (64 when N = 256, to
// keep at most 64 state values per thread) and a CTA of 256 threads owns one
// slice of one (b, h); warp w holds rows p0 + w, p0 + w + 8, ... and lane l
// columns n = l, l + 32, ... of the state (lanes l >= N idle when N = 16).
// y_t[p] is a sum over n: the warp's lanes reduce it with shuffles each step.  The inputs of kT steps
// are staged in shared memory one tile ahead.  The bidirectional scan runs
// a second pass from the last step that adds its part to y.  The scan
// options (dt bias / softplus / clamp, silu gate, initial and final state,
// groups of B and C) are applied as in the tensor-core kernel.
#include "ssm_common.cuh"

#include <algorithm>

namespace ssm {
namespace ssd_general {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kT = 16;            // steps per staged tile

struct Args {
    const void *x, *dt, *B, *C, *z;
    const float *A, *D, *dt_bias, *h0;
    float *y, *h_final;
    int L, H, P, N, G;
    int slices;       // CTAs per (b, h): row slices of PS = kWarps * PW rows
    float dt_min, dt_max;
    int dt_softplus, dt_limit;
};

// The staged rows of kT steps: the slice's x columns, B and C rows padded
// to the 32 NL states the kernel instance holds.
template <typename Tin, int PW, int NL>
struct Tile {
    Tin x[kT][8 * PW];
    Tin B[kT][32 * NL];
    Tin C[kT][32 * NL];
    float dt[kT];
};

// Stage the x (columns [p0, p0 + ps) of the row), B, C rows of steps
// [t0, t0 + kT) (in walk order: `rev` walks backwards) of one (b, h) with
// 16-byte asynchronous copies (slices and rows are multiples of 16 bytes; the
// entry points require 16-byte aligned x, B, C).  Rows outside [0, L) are
// zero filled.
template <typename Tin, typename TileT>
__device__ __forceinline__ void stage_rows(TileT &s, const Args &a, int64_t b, int h, int g,
                                           int p0, int ps, int t0, bool rev) {
    constexpr int EPC = 16 / sizeof(Tin);
    const Tin *x = static_cast<const Tin *>(a.x);
    const Tin *Bm = static_cast<const Tin *>(a.B);
    const Tin *Cm = static_cast<const Tin *>(a.C);
    const int cpx = ps / EPC, cpn = a.N / EPC;
    for (int i = threadIdx.x; i < kT * cpx; i += kThreads) {
        const int k = i / cpx, c = i % cpx;
        const int t = rev ? a.L - 1 - (t0 + k) : t0 + k;
        const bool ok = t0 + k < a.L;
        cp_async16(&s.x[k][c * EPC],
                   x + (ok ? ((b * a.L + t) * a.H + h) * a.P + p0 + c * EPC : 0), ok ? 16 : 0);
    }
    for (int i = threadIdx.x; i < kT * cpn; i += kThreads) {
        const int k = i / cpn, c = i % cpn;
        const int t = rev ? a.L - 1 - (t0 + k) : t0 + k;
        const bool ok = t0 + k < a.L;
        const int64_t o = ok ? ((b * a.L + t) * a.G + g) * a.N + c * EPC : 0;
        cp_async16(&s.B[k][c * EPC], Bm + o, ok ? 16 : 0);
        cp_async16(&s.C[k][c * EPC], Cm + o, ok ? 16 : 0);
    }
}

// The preprocessed dt of step t0 + k (walk order) for k = threadIdx.x < kT;
// 0 outside [0, L).
template <typename Tin>
__device__ __forceinline__ float load_dt(const Args &a, int64_t b, int h, int t0, bool rev,
                                         float dbias) {
    const int k = threadIdx.x;
    if (k >= kT || t0 + k >= a.L) return 0.0f;
    const int t = rev ? a.L - 1 - (t0 + k) : t0 + k;
    float d = to_f32(static_cast<const Tin *>(a.dt)[(b * a.L + t) * a.H + h]) + dbias;
    if (a.dt_softplus) d = softplus_fast(d);
    if (a.dt_limit) d = fminf(fmaxf(d, a.dt_min), a.dt_max);
    return d;
}

// One direction.  pass 0: forward, writes y (= scan + D x, gated unless a
// reverse pass follows); pass 1: reverse, adds its scan to y and gates.
template <typename Tin, int PW, int NL>
__global__ void __launch_bounds__(kThreads)
ssd_general_kernel(Args a, int pass, int gate_now) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    using TileT = Tile<Tin, PW, NL>;
    TileT *tiles = reinterpret_cast<TileT *>(smem_raw);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    constexpr int PS = kWarps * PW;              // rows of this CTA's slice
    const int bh = blockIdx.x / a.slices;
    const int p0 = (blockIdx.x % a.slices) * PS;
    const int64_t b = bh / a.H;
    const int h = bh % a.H;
    const int g = h / (a.H / a.G);
    const bool rev = pass == 1;
    const float A2 = a.A[h] * SSM_LOG2E;
    const float Dh = (a.D && !rev) ? a.D[h] : 0.0f;
    const float dbias = a.dt_bias ? a.dt_bias[h] : 0.0f;
    const Tin *zg = static_cast<const Tin *>(a.z);

    float st[PW][NL];
#pragma unroll
    for (int i = 0; i < PW; ++i)
#pragma unroll
        for (int j = 0; j < NL; ++j) {
            const int p = p0 + w + kWarps * i, n = lane + 32 * j;
            st[i][j] = (a.h0 && !rev && n < a.N) ? a.h0[((int64_t(bh) * a.P) + p) * a.N + n] : 0.0f;
        }

    const int ntiles = (a.L + kT - 1) / kT;
    stage_rows<Tin>(tiles[0], a, b, h, g, p0, PS, 0, rev);
    cp_async_commit();
    if (threadIdx.x < kT) tiles[0].dt[threadIdx.x] = load_dt<Tin>(a, b, h, 0, rev, dbias);
    cp_async_wait<0>();
    __syncthreads();
    for (int k = 0; k < ntiles; ++k) {
        TileT &s = tiles[k & 1];
        // the next tile's copies run while this one is used
        float dnext = 0.0f;
        if (k + 1 < ntiles) {
            stage_rows<Tin>(tiles[(k + 1) & 1], a, b, h, g, p0, PS, (k + 1) * kT, rev);
            dnext = load_dt<Tin>(a, b, h, (k + 1) * kT, rev, dbias);
        }
        cp_async_commit();
        const int steps = min(kT, a.L - k * kT);
        // Batches of kBatch steps: each lane keeps its partial sums of the
        // batch's PW rows (32 values), then one reduce-scatter over the warp
        // (31 shuffles) leaves lane l with the whole sum of value l = (step,
        // row) -- so the shuffle latencies overlap and each lane writes one
        // output.  Rows past L have dt = 0 and zero inputs: the state passes
        // through them unchanged, and their outputs are not written.
        constexpr int kBatch = 32 / PW;
#pragma unroll 1
        for (int j0 = 0; j0 < kT; j0 += kBatch) {
            if (j0 >= steps) break;
            float v[32];
#pragma unroll
            for (int jj = 0; jj < kBatch; ++jj) {
                const int j = j0 + jj;
                const float d = s.dt[j];
                const float dec = ex2(d * A2);
                float bv[NL], cv[NL];
#pragma unroll
                for (int q = 0; q < NL; ++q) {
                    // (N = 16: lanes past N hold no state and add nothing)
                    const bool n_ok = NL > 1 || lane + 32 * q < a.N;
                    bv[q] = n_ok ? to_f32(s.B[j][lane + 32 * q]) : 0.0f;
                    cv[q] = n_ok ? to_f32(s.C[j][lane + 32 * q]) : 0.0f;
                }
#pragma unroll
                for (int i = 0; i < PW; ++i) {
                    const float dx = d * to_f32(s.x[j][w + kWarps * i]);
                    float acc = 0.0f;
#pragma unroll
                    for (int q = 0; q < NL; ++q) {
                        st[i][q] = fmaf(dec, st[i][q], dx * bv[q]);
                        acc = fmaf(st[i][q], cv[q], acc);
                    }
                    v[jj * PW + i] = acc;
                }
            }
            // reduce-scatter: at distance o the lanes with bit o set keep the
            // upper half of their values, the others the lower half
#pragma unroll
            for (int o = 16, half = 16; o > 0; o >>= 1, half >>= 1) {
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int e = 0; e < half; ++e) {
                    const float send = up ? v[e] : v[e + half];
                    const float keep = up ? v[e + half] : v[e];
                    v[e] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            // lane l: value l = (step j0 + l / PW, row w + 8 (l % PW))
            const int j = j0 + lane / PW, pl = w + kWarps * (lane % PW);
            if (j < steps) {
                const int t = rev ? a.L - 1 - (k * kT + j) : k * kT + j;
                const int64_t o = ((b * a.L + t) * a.H + h) * a.P + p0 + pl;
                float val = v[0];
                if (rev) val += a.y[o];                       // forward part, written by pass 0
                else val = fmaf(Dh, to_f32(s.x[j][pl]), val);
                if (gate_now && zg) val *= silu_fast(to_f32(zg[o]));
                a.y[o] = val;
            }
        }
        cp_async_wait<0>();
        if (k + 1 < ntiles && threadIdx.x < kT) tiles[(k + 1) & 1].dt[threadIdx.x] = dnext;
        __syncthreads();    // the next tile is staged; this one's reads are done
    }
    if (a.h_final && !rev) {
#pragma unroll
        for (int i = 0; i < PW; ++i)
#pragma unroll
            for (int j = 0; j < NL; ++j) {
                const int p = p0 + w + kWarps * i, n = lane + 32 * j;
                if (n < a.N) a.h_final[((int64_t(bh) * a.P) + p) * a.N + n] = st[i][j];
            }
    }
}

template <typename Tin, int PW, int NL>
static cudaError_t run(const Args &a, int64_t grid, bool bidir, cudaStream_t st) {
    const int smem = int(2 * sizeof(Tile<Tin, PW, NL>));
    auto kern = ssd_general_kernel<Tin, PW, NL>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    kern<<<unsigned(grid), kThreads, smem, st>>>(a, 0, bidir ? 0 : 1);
    err = cudaGetLastError();
    if (err != cudaSuccess || !bidir) return err;
    kern<<<unsigned(grid), kThreads, smem, st>>>(a, 1, 1);
    return cudaGetLastError();
}

template <typename Tin, int PW>
static cudaError_t run_pw(const Args &a, int64_t grid, bool bidir, cudaStream_t st) {
    switch (a.N) {
        case 16:
        case 32: return run<Tin, PW, 1>(a, grid, bidir, st);
        case 64: return run<Tin, PW, 2>(a, grid, bidir, st);
        case 128: return run<Tin, PW, 4>(a, grid, bidir, st);
        case 256:
            if constexpr (PW <= 8) return run<Tin, PW, 8>(a, grid, bidir, st);
            return cudaErrorNotSupported;
    }
    return cudaErrorNotSupported;
}

static bool pow2_16_256(int64_t v) {
    return v == 16 || v == 32 || v == 64 || v == 128 || v == 256;
}

// Shapes this path takes: P and N in {16, 32, 64, 128, 256}.
bool supported(int64_t P, int64_t N) { return pow2_16_256(P) && pow2_16_256(N); }

template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dt, const float *A_head, const Tin *Bm, const Tin *Cm,
                   const float *D, float *y, int64_t Bs, int64_t L, int64_t H, int64_t P,
                   int64_t N, bool bidir, int num_sms, const ScanOpts *opt, cudaStream_t st) {
    if (!supported(P, N)) return cudaErrorNotSupported;
    // slice height: at most 64 state values per thread (16 rows per warp of
    // up to 4 columns, or 8 rows of 8 columns when N = 256), and narrower
    // slices (down to 16 rows) while there are fewer than two CTAs per SM
    int64_t ps = std::min<int64_t>(P, N == 256 ? 64 : 128);
    while (ps > 16 && Bs * H * (P / ps) < 2 * int64_t(num_sms)) ps /= 2;
    const int64_t grid = Bs * H * (P / ps);
    if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const ScanOpts none{};
    const ScanOpts &o = opt ? *opt : none;
    Args a;
    a.x = x; a.dt = dt; a.B = Bm; a.C = Cm; a.z = o.z;
    a.A = A_head; a.D = D; a.dt_bias = o.dt_bias; a.h0 = o.h0;
    a.y = y; a.h_final = o.h_final;
    a.L = int(L); a.H = int(H); a.P = int(P); a.N = int(N);
    a.G = o.ngroups > 1 ? o.ngroups : 1;
    a.slices = int(P / ps);
    a.dt_min = o.dt_min; a.dt_max = o.dt_max;
    a.dt_softplus = o.dt_softplus; a.dt_limit = o.dt_limit;
    switch (ps) {
        case 16: return run_pw<Tin, 2>(a, grid, bidir, st);
        case 32: return run_pw<Tin, 4>(a, grid, bidir, st);
        case 64: return run_pw<Tin, 8>(a, grid, bidir, st);
        case 128: return run_pw<Tin, 16>(a, grid, bidir, st);
    }
    return cudaErrorNotSupported;
}

template cudaError_t launch<float>(const float *, const float *, const float *, const float *,
                                   const float *, const float *, float *, int64_t, int64_t, int64_t,
                                   int64_t, int64_t, bool, int, const ScanOpts *, cudaStream_t);
template cudaError_t launch<__nv_bfloat16>(const __nv_bfloat16 *, const __nv_bfloat16 *,
                                           const float *, const __nv_bfloat16 *,
                                           const __nv_bfloat16 *, const float *, float *, int64_t,
                                           int64_t, int64_t, int64_t, int64_t, bool, int,
                                           const ScanOpts *, cudaStream_t);

}  // namespace ssd_general
}  // namespace ssm
