// diag_scan.cuh -- diagonal-A selective scan (Mamba-1 style) for sm_103a:
// the kernels and their launch path, shared by diag_scan.cu (plain scan)
// and diag_scan_ext.cu (the variant with the scan options).
//
// Computes, per channel (b, e) and state n, with h_{-1} = 0,
//     h_t[n] = exp(delta_t * A[e,n]) * h_{t-1}[n] + delta_t * B_t[n] * x_t
//     y_t    = sum_n C_t[n] * h_t[n] + D[e] * x_t
// -- the sequential form selective_scan_seq of "scan output is different
// between sequential and parallel versions" (mamba.py issue 26), with the
// shape API given there (x, delta (Bs,L,ED); A (ED,N); B, C (Bs,L,N); D (ED)).
//
// Design (one pass over HBM, state never leaves registers):
//   * A CTA of 128 threads owns ET = 128 / G consecutive channels of one
//     batch row b for the whole sequence.  G lanes share a channel, each
//     holding S = NP / G of its (padded) states in registers, so the work
//     per thread is S independent fp32 recurrences (instruction-level
//     parallelism) and the y reduction over the G lanes is a shuffle.
//   * Time is walked in tiles of TT steps.  x and delta tiles (TT x ET) and
//     the B, C rows of the tile (TT x N, contiguous in memory) are staged
//     into shared memory by 16-byte cp.async copies, two tiles ahead of the
//     compute (double buffered), so HBM latency overlaps the recurrence.
//   * B and C are converted once per tile to fp32 (zero padded to NP) and
//     read back as broadcast float4 loads by every channel's lanes.
//   * exp(delta*A) is one MUFU ex2 per element-step: A is pre-scaled by
//     log2(e) once per (e, n) in registers.
//   * y is stored from registers: per step a warp writes 32/G consecutive
//     fp32 values of one row.
#pragma once

#include "ssm_common.cuh"

#include <algorithm>

namespace ssm {
namespace diag {

constexpr int kThreads = 128;
constexpr int kTileT = 32;   // time steps per shared-memory tile
constexpr int kStages = 2;   // tiles in flight (cp.async ring): one ahead hides HBM latency

template <typename Tin, int S, int G>
struct Shape {
    static constexpr int ET = kThreads / G;  // channels per CTA
    static constexpr int NP = S * G;         // padded state count
    static constexpr size_t raw_x = size_t(kTileT) * ET;     // elements per x tile
    static constexpr size_t raw_bc = size_t(kTileT) * NP;    // elements per B tile
    static constexpr size_t smem_bytes =
        (kStages * 2 * raw_x + kStages * 2 * raw_bc) * sizeof(Tin) + 2 * raw_bc * sizeof(float);
    // with the optional gate z: one more x-shaped ring after the fp32 B, C rows
    static constexpr size_t smem_bytes_z = smem_bytes + kStages * raw_x * sizeof(Tin);
    // option kernels: the gate ring, then the tile's silu(z) in fp32 (x-shaped)
    static constexpr size_t smem_bytes_ext = smem_bytes_z + raw_x * sizeof(float);
};

// Stage one time tile of x, delta, B, C into a shared-memory ring slot.
// Rows past the end of the sequence are zero filled: delta = 0 there makes
// exp(delta*A) = 1 and delta*B*x = 0, so the state passes through unchanged.
template <typename Tin, int S, int G, bool VEC>
__device__ __forceinline__ void load_tile(Tin *sx, Tin *sd, Tin *sB, Tin *sC,
                                          const Tin *__restrict__ x, const Tin *__restrict__ dlt,
                                          const Tin *__restrict__ Bm, const Tin *__restrict__ Cm,
                                          int64_t b, int t0, int te, int L, int e0, int ED,
                                          int N, Tin *sz = nullptr,
                                          const Tin *__restrict__ zg = nullptr) {
    using Sh = Shape<Tin, S, G>;
    constexpr int ET = Sh::ET;
    const int tid = threadIdx.x;
    const int rows = max(0, min(kTileT, te - t0));   // rows of this segment (te <= L)
    if constexpr (VEC) {
        constexpr int EPC = 16 / sizeof(Tin);       // elements per 16-byte chunk
        constexpr int CPR = ET / EPC;               // chunks per x row
        for (int i = tid; i < kTileT * CPR; i += kThreads) {
            const int t = i / CPR, c = i % CPR;
            const int e = e0 + c * EPC;
            const bool ok = (t < rows) && (e < ED);
            const int64_t g = ok ? ((b * L + t0 + t) * ED + e) : 0;
            cp_async16(sx + t * ET + c * EPC, x + g, ok ? 16 : 0);
            cp_async16(sd + t * ET + c * EPC, dlt + g, ok ? 16 : 0);
            if (zg) cp_async16(sz + t * ET + c * EPC, zg + g, ok ? 16 : 0);
        }
        // B, C rows t0..t0+rows-1 are one contiguous block of rows*N elements.
        const int nchunk = kTileT * N / EPC;
        const int valid = rows * N / EPC;
        const int64_t base = (b * L + t0) * N;
        for (int i = tid; i < nchunk; i += kThreads) {
            const bool ok = i < valid;
            const int64_t g = ok ? base + int64_t(i) * EPC : 0;
            cp_async16(sB + i * EPC, Bm + g, ok ? 16 : 0);
            cp_async16(sC + i * EPC, Cm + g, ok ? 16 : 0);
        }
    } else {
        // Any alignment: element-wise synchronous copies.
        for (int i = tid; i < kTileT * ET; i += kThreads) {
            const int t = i / ET, c = i % ET;
            const int e = e0 + c;
            const bool ok = (t < rows) && (e < ED);
            const int64_t g = ok ? (b * L + t0 + t) * ED + e : 0;
            sx[i] = ok ? x[g] : Tin(0.0f);
            sd[i] = ok ? dlt[g] : Tin(0.0f);
            if (zg) sz[i] = ok ? zg[g] : Tin(0.0f);
        }
        const int64_t base = (b * L + t0) * N;
        for (int i = tid; i < kTileT * N; i += kThreads) {
            const bool ok = i < rows * N;
            sB[i] = ok ? Bm[base + i] : Tin(0.0f);
            sC[i] = ok ? Cm[base + i] : Tin(0.0f);
        }
    }
}

// Summary of one time segment of one channel, written when the sequence is
// split into K > 1 segments: the segment's end state started from zero, the
// sum of its deltas, and its smallest delta.
struct SegSummary {
    float *h_end;   // [K][Bs][ED][16]
    float *dsum;    // [K][Bs][ED]
    float *dmin;    // [K][Bs][ED]
};

// Optional parts of the scan (the options of the chunked scan's argument
// list in "Some questions of Bi-Mamba2 and Hydra", Bi-Mamba2 issue 1), see
// ScanOpts: shapes (ED) for dt_bias, (Bs, L, ED) for z, (Bs, ED, N) for the
// states.
using Ext = ScanOpts;

// The delta the recurrence sees, from the stored one and the channel's bias.
__device__ __forceinline__ float prep_delta(float d, float bias, const Ext &ex) {
    d += bias;
    if (ex.dt_softplus) d = softplus_fast(d);
    if (ex.dt_limit) d = fminf(fmaxf(d, ex.dt_min), ex.dt_max);
    return d;
}

// silu(z) = z * sigmoid(z)
__device__ __forceinline__ float silu(float z) { return silu_fast(z); }

template <typename Tin, int S, int G, bool VEC, bool SPLIT, bool EXT>
__global__ void __launch_bounds__(kThreads)
diag_scan_kernel(const Tin *__restrict__ x, const Tin *__restrict__ dlt,
                 const float *__restrict__ A, const Tin *__restrict__ Bm,
                 const Tin *__restrict__ Cm, const float *__restrict__ D,
                 float *__restrict__ y, int L, int ED, int N, int n_etiles, int seg_len,
                 SegSummary summ, Ext ex) {
    using Sh = Shape<Tin, S, G>;
    constexpr int ET = Sh::ET;
    constexpr int NP = Sh::NP;
    static_assert(S % 4 == 0, "states per thread must be a multiple of 4");

    // With a time split the carry pass follows as a programmatic dependent
    // launch: it may start once every CTA of this pass has started, stage its
    // first inputs, and wait (griddepcontrol.wait) for this grid's results.
    if constexpr (SPLIT) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    extern __shared__ __align__(16) unsigned char smem_raw[];
    Tin *sx = reinterpret_cast<Tin *>(smem_raw);     // [kStages][TT][ET]
    Tin *sd = sx + kStages * Sh::raw_x;              // [kStages][TT][ET]
    Tin *sB = sd + kStages * Sh::raw_x;              // [kStages][TT*N] (dense rows)
    Tin *sC = sB + kStages * Sh::raw_bc;             // [kStages][TT*N]
    float *fB = reinterpret_cast<float *>(sC + kStages * Sh::raw_bc);  // [TT][NP]
    float *fC = fB + Sh::raw_bc;                                        // [TT][NP]
    Tin *sz = reinterpret_cast<Tin *>(fC + Sh::raw_bc);                 // [kStages][TT][ET] (gate)
    float *fZ = reinterpret_cast<float *>(sz + kStages * Sh::raw_x);    // [TT][ET] silu(z)
    const Tin *zg = EXT ? static_cast<const Tin *>(ex.z) : nullptr;

    const int64_t b = blockIdx.x / n_etiles;
    const int e0 = (blockIdx.x % n_etiles) * ET;
    const int seg = blockIdx.y;
    const int tb = seg * seg_len;                    // this CTA's time range [tb, te)
    const int te = min(L, tb + seg_len);
    const int tid = threadIdx.x;
    const int ch = tid / G;
    const int g = tid % G;
    const int e = e0 + ch;
    const bool e_ok = e < ED;

    // States and A * log2(e) in registers.  The per-step arithmetic is scalar
    // fp32: on this part a packed fp32x2 multiply-add occupies the FMA pipe
    // longer than two scalar ones.
    float A2[S], h[S];
#pragma unroll
    for (int j = 0; j < S; ++j) {
        const int n = g * S + j;
        A2[j] = (e_ok && n < N) ? A[int64_t(e) * N + n] * SSM_LOG2E : 0.0f;
        h[j] = 0.0f;
        // the first segment starts from the given initial state
        if (EXT && ex.h0 && seg == 0 && e_ok && n < N) h[j] = ex.h0[(b * ED + e) * N + n];
    }
    const float dbias = (EXT && ex.dt_bias && e_ok) ? ex.dt_bias[e] : 0.0f;
    // delta preparation in use (a uniform flag: the option kernels also serve
    // calls with only state I/O or checkpoints)
    const bool prep = EXT && (ex.dt_bias != nullptr || ex.dt_softplus || ex.dt_limit);
    const float Dv = (D != nullptr && e_ok) ? D[e] : 0.0f;
    float dsum = 0.0f, dmin = 3.0e38f;

    const int n_tiles = (te - tb + kTileT - 1) / kTileT;
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
        if (k < n_tiles)
            load_tile<Tin, S, G, VEC>(sx + k * Sh::raw_x, sd + k * Sh::raw_x, sB + k * Sh::raw_bc,
                                      sC + k * Sh::raw_bc, x, dlt, Bm, Cm, b, tb + k * kTileT, te,
                                      L, e0, ED, N, sz + k * Sh::raw_x, zg);
        cp_async_commit();
    }

    for (int k = 0; k < n_tiles; ++k) {
        const int st = k % kStages;
        cp_async_wait<kStages - 2>();
        __syncthreads();   // tile k landed everywhere; tile k-1 fully consumed
        {
            const int kn = k + kStages - 1;
            const int sn = kn % kStages;
            if (kn < n_tiles)
                load_tile<Tin, S, G, VEC>(sx + sn * Sh::raw_x, sd + sn * Sh::raw_x,
                                          sB + sn * Sh::raw_bc, sC + sn * Sh::raw_bc, x, dlt, Bm,
                                          Cm, b, tb + kn * kTileT, te, L, e0, ED, N,
                                          sz + sn * Sh::raw_x, zg);
            cp_async_commit();
        }
        const int t0 = tb + k * kTileT;
        const int tl = min(kTileT, te - t0);
        // B, C of this tile -> fp32, zero padded to NP states.
        {
            const Tin *rb = sB + st * Sh::raw_bc;
            const Tin *rc = sC + st * Sh::raw_bc;
            for (int i = tid; i < kTileT * NP; i += kThreads) {
                const int t = i / NP, n = i % NP;
                fB[i] = n < N ? to_f32(rb[t * N + n]) : 0.0f;
                fC[i] = n < N ? to_f32(rc[t * N + n]) : 0.0f;
            }
        }
        if (EXT && zg) {
            // The gate's silu(z) for the whole tile in one pass (independent
            // elements, so the special-function latencies overlap) instead of
            // at each store.  The G lanes of a channel share its rows.  (The
            // delta preparation measured faster inline, in the step's fetch.)
            const Tin *rz = sz + st * Sh::raw_x;
            for (int t = g; t < kTileT; t += G) fZ[t * ET + ch] = silu(to_f32(rz[t * ET + ch]));
        }
        __syncthreads();

        const Tin *xs = sx + st * Sh::raw_x + ch;
        const Tin *ds = sd + st * Sh::raw_x + ch;
        const float *bq = fB + g * S;
        const float *cq = fC + g * S;
        float *yp = y + (b * L + t0) * ED + e;
        const bool store_ok = (g == 0) && e_ok && !(EXT && ex.no_y);
        // Operands of the next step are read from shared memory before this
        // step's result is stored: y is a generic pointer, and the compiler
        // may not move shared loads across a store that could alias them.
        // Two register sets hold the operands of consecutive steps: the next
        // step's operands are fetched before the current step's arithmetic.
        // Eight steps per loop iteration: unrolling the whole tile overflows
        // the instruction cache once several warps share a scheduler.
        constexpr int kUnroll = 8;
        float o_dl[2], o_xv[2], o_z[2];
        float4 o_b[2][S / 4], o_c[2][S / 4];
        auto fetch = [&](int t, int r) {
            const int tt = min(t, kTileT - 1);   // past the tile's end: a harmless re-read
            o_dl[r] = to_f32(ds[tt * ET]);
            // rows past the segment keep delta = 0 (the state passes through)
            if (EXT && prep) o_dl[r] = tt < tl ? prep_delta(o_dl[r], dbias, ex) : 0.0f;
            o_xv[r] = to_f32(xs[tt * ET]);
            if (EXT && zg) o_z[r] = fZ[tt * ET + ch];
#pragma unroll
            for (int q = 0; q < S / 4; ++q) {
                o_b[r][q] = reinterpret_cast<const float4 *>(bq + tt * NP)[q];
                o_c[r][q] = reinterpret_cast<const float4 *>(cq + tt * NP)[q];
            }
        };
        auto step = [&](int t, int r) {
            const float dl = o_dl[r], xv = o_xv[r];
            float bv[S], cv[S];
#pragma unroll
            for (int q = 0; q < S / 4; ++q) {
                bv[4 * q] = o_b[r][q].x; bv[4 * q + 1] = o_b[r][q].y; bv[4 * q + 2] = o_b[r][q].z; bv[4 * q + 3] = o_b[r][q].w;
                cv[4 * q] = o_c[r][q].x; cv[4 * q + 1] = o_c[r][q].y; cv[4 * q + 2] = o_c[r][q].z; cv[4 * q + 3] = o_c[r][q].w;
            }
            const float dlx = dl * xv;
            if constexpr (SPLIT) {
                // (rows past the segment hold delta = 0: they leave the sum
                // unchanged and cannot make the minimum negative)
                dsum += dl;
                dmin = fminf(dmin, dl);
            }
            // Products with the step's delta and delta*x are formed two states
            // at a time (packed fp32x2 multiply: one issue slot for two), the
            // state update and the readout as scalar fused multiply-adds
            // (packed fused multiply-adds measured slower here: they hold the
            // FMA pipe longer than two scalar ones).
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const float2 dl2 = make_float2(dl, dl), dlx2 = make_float2(dlx, dlx);
#pragma unroll
            for (int n = 0; n < S; n += 2) {
                const float2 z = __fmul2_rn(dl2, make_float2(A2[n], A2[n + 1]));
                const float2 u = __fmul2_rn(dlx2, make_float2(bv[n], bv[n + 1]));
                h[n] = fmaf(ex2(z.x), h[n], u.x);
                h[n + 1] = fmaf(ex2(z.y), h[n + 1], u.y);
                acc[n & 3] = fmaf(cv[n], h[n], acc[n & 3]);
                acc[(n + 1) & 3] = fmaf(cv[n + 1], h[n + 1], acc[(n + 1) & 3]);
            }
            float yv = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
            for (int o = 1; o < G; o <<= 1) yv += __shfl_xor_sync(0xffffffffu, yv, o);
            float out = fmaf(Dv, xv, yv);
            if (EXT && zg) out *= o_z[r];
            if (store_ok && t < tl) yp[int64_t(t) * ED] = out;
        };
        fetch(0, 0);
#pragma unroll 1
        for (int t = 0; t < kTileT; t += kUnroll) {
            if (EXT && ex.ckpt && (t & 15) == 0 && e_ok && t0 + t < te) {
                // state entering steps t0 + t .. t0 + t + 15 (one segment, K = 1)
                float4 *dst = reinterpret_cast<float4 *>(
                    ex.ckpt + ((int64_t((t0 + t) >> 4) * (gridDim.x / n_etiles) + b) * ED + e) * 16 +
                    g * S);
#pragma unroll
                for (int q = 0; q < S / 4; ++q)
                    dst[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; u += 2) {
                fetch(t + u + 1, 1);
                step(t + u, 0);
                fetch(t + u + 2, 0);
                step(t + u + 1, 1);
            }
        }
    }
    cp_async_wait<0>();

    if constexpr (EXT && !SPLIT) {
        // one segment: this thread's states are the final ones
        if (ex.h_final && e_ok) {
#pragma unroll
            for (int j = 0; j < S; ++j) {
                const int n = g * S + j;
                if (n < N) ex.h_final[(b * ED + e) * N + n] = h[j];
            }
        }
    }
    if constexpr (SPLIT) {
        // Rows past the segment's end were zero filled (delta = 0), so h and
        // dsum are exactly the segment's end state and delta sum.
        if (e_ok) {
            const int64_t c = (int64_t(seg) * (gridDim.x / n_etiles) + b) * ED + e;
#pragma unroll
            for (int j = 0; j < S; ++j) summ.h_end[c * 16 + g * S + j] = h[j];
            if (g == 0) {
                summ.dsum[c] = dsum;
                summ.dmin[c] = dmin;
            }
        }
    }
}

// Copy rows [t0, t0 + kTileT) x channels [e0, e0 + CW) of a (Bs, L, ED)
// tensor into shared memory [kTileT][CW]; rows >= te and channels >= ED are
// zero filled.  VEC: 16-byte cp.async chunks (caller checked alignment).
template <typename T, bool VEC, int CW>
__device__ __forceinline__ void stage_rows(T *dst, const T *__restrict__ src, int64_t b, int t0,
                                           int te, int L, int e0, int ED) {
    constexpr int EPC = 16 / sizeof(T);
    const int rows = max(0, min(kTileT, te - t0));
    if constexpr (VEC) {
        constexpr int CPR = CW / EPC;
        for (int i = threadIdx.x; i < kTileT * CPR; i += kThreads) {
            const int t = i / CPR, c = i % CPR;
            const int e = e0 + c * EPC;
            const bool ok = (t < rows) && (e < ED);
            const int64_t g = ok ? ((b * L + t0 + t) * ED + e) : 0;
            cp_async16(dst + t * CW + c * EPC, src + g, ok ? 16 : 0);
        }
    } else {
        for (int i = threadIdx.x; i < kTileT * CW; i += kThreads) {
            const int t = i / CW, c = i % CW;
            const int e = e0 + c;
            const bool ok = (t < rows) && (e < ED);
            dst[i] = ok ? src[(b * L + t0 + t) * ED + e] : T(0.0f);
        }
    }
}

// Second pass of a time-split scan (16 padded states): for every segment
// k >= 1, fold the summaries of segments 0..k-1 into the state entering
// segment k, h_in, and add its contribution
//     y_t += sum_n C_t[n] * exp(A[e,n] * (delta_{tb} + ... + delta_t)) * h_in[n]
// to the segment's outputs, which the first pass computed from a zero state.
// Every (t, n) term is independent once the running delta sums are known, so
// the work is spread over time: a CTA covers 32 channels (lane = channel) and
// its warp w takes rows 8w..8w+7 of each 32-step tile.  A term is evaluated
// as sign(h_in) * exp2(A log2(e) cumsum + log2|h_in|).  exp2 flushes results
// below 2^-126 to zero, so once that exponent is below -126 for state n in
// every channel of the CTA, the state adds exactly zero from then on, as long
// as delta >= 0 and A <= 0 (checked per segment and channel); the same holds,
// up to a relative 2^-40 (kDecayCut), once the decay alone is below 2^-40.
// Such states are skipped (the test is uniform over the CTA, so the skip is a
// uniform branch), and the CTA stops when all are.  delta and C are staged through a
// ring of kFixRing tiles in shared memory, so several tiles' copies are in
// flight at once; each output receives its correction with one atomic add
// (one add per element, so the result does not depend on ordering).
constexpr int kFixCh = 32;
constexpr int kFixRing = 4;
// A state whose carried part has decayed by more than 2^-40 (relative to the
// entering state, i.e. exp2(A log2(e) cumsum) < 2^-40) is also dropped: every
// correction it would still add is below 2^-40 of the one it added at the
// segment's first step, far inside fp32 rounding of the outputs; the carry
// pass then stops after ~90 instead of ~280 steps on the benchmark data.
constexpr float kDecayCut = 40.0f;
constexpr int kMaxSeg = 8;     // time segments a split may use
template <typename Tin, bool VEC, bool EXT>
__global__ void __launch_bounds__(kThreads)
diag_fixup_kernel(const Tin *__restrict__ dlt, const float *__restrict__ A,
                  const Tin *__restrict__ Cm, float *__restrict__ y, int Bs, int L, int ED, int N,
                  int seg_len, SegSummary summ, Ext ex) {
    constexpr int NP = 16;
    constexpr int CW = kFixCh;
    constexpr int RW = kTileT / 4;           // rows of a tile per warp
    constexpr int R = kFixRing;
    __shared__ __align__(16) Tin s_d[R][kTileT * CW];
    __shared__ __align__(16) Tin s_z[EXT ? R : 1][EXT ? kTileT * CW : 8];
    __shared__ __align__(16) Tin s_c[R][kTileT * NP];
    __shared__ __align__(16) float s_cf[kTileT * NP];
    __shared__ float s_lh[NP][CW];
    __shared__ unsigned s_sg[NP][CW];
    __shared__ float s_psum[4][CW];
    __shared__ unsigned s_live[4];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int w = tid >> 5;
    const int e0 = blockIdx.x * CW;
    const int e = e0 + lane;
    const int64_t b = blockIdx.y;
    const int seg = blockIdx.z + 1;
    const bool e_ok = e < ED;
    const int ec = e_ok ? e : ED - 1;    // lanes past ED mirror a valid channel, store nothing
    const Tin *zg = EXT ? static_cast<const Tin *>(ex.z) : nullptr;
    const float dbias = (EXT && ex.dt_bias) ? ex.dt_bias[ec] : 0.0f;

    const int tb = seg * seg_len;
    const int te = min(L, tb + seg_len);
    const int n_tiles = (te - tb + kTileT - 1) / kTileT;
    auto stage = [&](int k) {
        const int t0 = tb + k * kTileT;
        const int slot = k % R;
        stage_rows<Tin, VEC, CW>(s_d[slot], dlt, b, t0, te, L, e0, ED);
        if (EXT && zg) stage_rows<Tin, VEC, CW>(s_z[slot], zg, b, t0, te, L, e0, ED);
        // C rows t0..t0+rows-1: one contiguous block, zero padded to 16 states
        const int rows = max(0, min(kTileT, te - t0));
        const int64_t base = (b * L + t0) * N;
        if (VEC && N == NP) {
            constexpr int EPC = 16 / sizeof(Tin);
            for (int i = tid; i < kTileT * NP / EPC; i += kThreads) {
                const bool ok = i * EPC < rows * NP;
                cp_async16(&s_c[slot][i * EPC], Cm + (ok ? base + int64_t(i) * EPC : 0), ok ? 16 : 0);
            }
        } else {
            for (int i = tid; i < kTileT * NP; i += kThreads) {
                const int t = i / NP, n = i % NP;
                s_c[slot][i] = (t < rows && n < N) ? Cm[base + t * N + n] : Tin(0.0f);
            }
        }
    };
    // The first tiles' copies go out before the summaries are read.
#pragma unroll
    for (int k = 0; k < R - 1; ++k) {
        if (k < n_tiles) stage(k);
        cp_async_commit();
    }

    // h_in for states 4w..4w+3 of channel `lane`, shared as log2|h_in| and
    // sign.  All summary loads are issued before the fold uses them.
    // The main pass's results (summaries, y, checkpoints) are read only
    // after it has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    bool mono = summ.dmin[(int64_t(seg) * Bs + b) * ED + ec] >= 0.0f;
    {
        float a2[4], hin[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = 4 * w + j;
            a2[j] = n < N ? A[int64_t(ec) * N + n] * SSM_LOG2E : 0.0f;
        }
        float ds[kMaxSeg];
        float4 he[kMaxSeg];
#pragma unroll
        for (int k = 0; k < kMaxSeg; ++k) {
            if (k < seg) {
                const int64_t c = (int64_t(k) * Bs + b) * ED + ec;
                ds[k] = summ.dsum[c];
                he[k] = reinterpret_cast<const float4 *>(summ.h_end + c * 16)[w];
            }
        }
#pragma unroll
        for (int k = 0; k < kMaxSeg; ++k) {
            if (k < seg) {
                hin[0] = fmaf(ex2(a2[0] * ds[k]), hin[0], he[k].x);
                hin[1] = fmaf(ex2(a2[1] * ds[k]), hin[1], he[k].y);
                hin[2] = fmaf(ex2(a2[2] * ds[k]), hin[2], he[k].z);
                hin[3] = fmaf(ex2(a2[3] * ds[k]), hin[3], he[k].w);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            s_lh[4 * w + j][lane] = __log2f(fabsf(hin[j]));   // -inf for a zero state
            s_sg[4 * w + j][lane] = __float_as_uint(hin[j]) & 0x80000000u;
        }
        // The last segment's CTAs also produce the final state:
        // h_final = exp(A sum(delta of the segment)) h_in + (its end state from zero).
        if (EXT && ex.h_final && seg == gridDim.z && e_ok) {
            const int64_t c = (int64_t(seg) * Bs + b) * ED + ec;
            const float dseg = summ.dsum[c];
            const float4 hs = reinterpret_cast<const float4 *>(summ.h_end + c * 16)[w];
            const float hv[4] = {hs.x, hs.y, hs.z, hs.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = 4 * w + j;
                if (n < N) ex.h_final[(b * ED + e) * N + n] = fmaf(ex2(a2[j] * dseg), hin[j], hv[j]);
            }
        }
    }
    float A2[NP], lh[NP];
    unsigned sg[NP];
    __syncthreads();
#pragma unroll
    for (int n = 0; n < NP; ++n) {
        A2[n] = n < N ? A[int64_t(ec) * N + n] * SSM_LOG2E : 0.0f;
        mono = mono && (A2[n] <= 0.0f);
        lh[n] = s_lh[n][lane];
        sg[n] = s_sg[n][lane];
    }
    const bool all_mono = __syncthreads_and(mono) != 0;

    float cum_run = 0.0f;      // delta summed over the tiles already done (same in every warp)
    for (int k = 0; k < n_tiles; ++k) {
        const int slot = k % R;
        // The slot refilled here was last read in iteration k - 1, before
        // its closing barrier.
        if (k + R - 1 < n_tiles) stage(k + R - 1);
        cp_async_commit();
        // States that can still contribute from this tile on.
        unsigned m = 0xffffu;
        if (all_mono) {
            m = 0;
#pragma unroll
            for (int n = 0; n < NP; ++n)
                if (A2[n] * cum_run >= -kDecayCut && fmaf(A2[n], cum_run, lh[n]) >= -126.0f)
                    m |= 1u << n;
            m = __reduce_or_sync(0xffffffffu, m);
        }
        cp_async_wait<R - 1>();
        float d[RW], psum = 0.0f;
        const int t0 = tb + k * kTileT;
        const int tl = min(kTileT, te - t0);
        __syncthreads();     // tile k landed everywhere
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            d[r] = to_f32(s_d[slot][(RW * w + r) * CW + lane]);
            if (EXT) d[r] = (RW * w + r) < tl ? prep_delta(d[r], dbias, ex) : 0.0f;
            psum += d[r];
        }
        s_psum[w][lane] = psum;
        if (lane == 0) s_live[w] = m;
        for (int i = 4 * tid; i < kTileT * NP; i += 4 * kThreads)
            reinterpret_cast<float4 *>(s_cf + i)[0] = to_f32x4(&s_c[slot][i]);
        __syncthreads();
        const unsigned live = s_live[0] | s_live[1] | s_live[2] | s_live[3];
        if (live == 0) break;    // every state's carried part has decayed to zero
        float cum[RW], acc[RW], tile_sum = 0.0f, run = cum_run;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const float p = s_psum[v][lane];
            tile_sum += p;
            run += (v < w) ? p : 0.0f;
        }
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            run += d[r];
            cum[r] = run;
            acc[r] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (!((live >> (4 * j)) & 0xfu)) continue;
            float4 c4[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) c4[r] = reinterpret_cast<const float4 *>(s_cf + (RW * w + r) * NP)[j];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = 4 * j + q;
                if (!((live >> n) & 1u)) continue;
#pragma unroll
                for (int r = 0; r < RW; ++r) {
                    const float cv = q == 0 ? c4[r].x : q == 1 ? c4[r].y : q == 2 ? c4[r].z : c4[r].w;
                    const float z = fmaf(A2[n], cum[r], lh[n]);
                    acc[r] = fmaf(cv, __uint_as_float(__float_as_uint(ex2(z)) ^ sg[n]), acc[r]);
                }
            }
        }
        if (e_ok && !(EXT && ex.no_y)) {
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int t = RW * w + r;
                float v = acc[r];
                if (EXT && zg) v *= silu(to_f32(s_z[slot][t * CW + lane]));   // the output gate
                if (t < tl && v != 0.0f) atomicAdd(y + (b * L + t0 + t) * ED + e, v);
            }
        }
        if (EXT && ex.ckpt && e_ok) {
            // checkpoints (the state entering every 16th step) of this
            // segment were written from a zero entering state: add the
            // carried part, exp(A (delta summed before the step)) h_in
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int t = RW * w + r;
                if (((t0 + t) & 15) != 0 || t >= tl) continue;
                const float exc = cum[r] - d[r];
                float4 *dst = reinterpret_cast<float4 *>(
                    ex.ckpt + ((int64_t((t0 + t) >> 4) * Bs + b) * ED + e) * 16);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float cv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int n = 4 * j + q;
                        cv[q] = ((live >> n) & 1u)
                                    ? __uint_as_float(__float_as_uint(ex2(fmaf(A2[n], exc, lh[n]))) ^ sg[n])
                                    : 0.0f;
                    }
                    float4 v4 = dst[j];
                    v4.x += cv[0]; v4.y += cv[1]; v4.z += cv[2]; v4.w += cv[3];
                    dst[j] = v4;
                }
            }
        }
        cum_run += tile_sum;
        __syncthreads();     // every read of this tile's slot and of s_cf is done
    }
    cp_async_wait<0>();
}

template <typename Tin, int S, int G, bool VEC, bool SPLIT, bool EXT>
static cudaError_t launch_one(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm,
                              const Tin *Cm, const float *D, float *y, int64_t Bs, int L, int ED,
                              int N, int K, int seg_len, SegSummary summ, const Ext &ex,
                              cudaStream_t stream) {
    using Sh = Shape<Tin, S, G>;
    const int n_etiles = (ED + Sh::ET - 1) / Sh::ET;
    const int64_t grid = Bs * n_etiles;
    if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
    auto kern = diag_scan_kernel<Tin, S, G, VEC, SPLIT, EXT>;
    const int smem = int(EXT ? Sh::smem_bytes_ext : Sh::smem_bytes);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
    }
    kern<<<dim3(unsigned(grid), unsigned(K)), dim3(kThreads), smem, stream>>>(
        x, dlt, A, Bm, Cm, D, y, L, ED, N, n_etiles, seg_len, summ, ex);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || !SPLIT) return err;
    const dim3 fgrid(unsigned((ED + kFixCh - 1) / kFixCh), unsigned(Bs), unsigned(K - 1));
    const bool yvec = (reinterpret_cast<uintptr_t>(y) % 16 == 0) && (ED % 4 == 0);
    // a programmatic dependent launch: its prologue overlaps the main pass's tail
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = fgrid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int Bsi = int(Bs);
    if (VEC && yvec)
        return cudaLaunchKernelEx(&cfg, diag_fixup_kernel<Tin, true, EXT>, dlt, A, Cm, y, Bsi, L, ED, N,
                                  seg_len, summ, ex);
    return cudaLaunchKernelEx(&cfg, diag_fixup_kernel<Tin, false, EXT>, dlt, A, Cm, y, Bsi, L, ED, N,
                              seg_len, summ, ex);
}

template <typename Tin, bool VEC, bool SPLIT, bool EXT>
static cudaError_t dispatch_sg(int S, int G, const Tin *x, const Tin *dlt, const float *A,
                               const Tin *Bm, const Tin *Cm, const float *D, float *y, int64_t Bs,
                               int L, int ED, int N, int K, int seg_len, SegSummary summ,
                               const Ext &ex, cudaStream_t st) {
#define SSM_DIAG_CASE(s_, g_)                                                                    \
    if (S == s_ && G == g_)                                                                      \
        return launch_one<Tin, s_, g_, VEC, SPLIT, EXT>(x, dlt, A, Bm, Cm, D, y, Bs, L, ED, N,    \
                                                        K, seg_len, summ, ex, st);
    SSM_DIAG_CASE(16, 1)
    SSM_DIAG_CASE(8, 2)
    SSM_DIAG_CASE(4, 4)
    if constexpr (!SPLIT) {
        SSM_DIAG_CASE(16, 2)
        SSM_DIAG_CASE(8, 4)
        SSM_DIAG_CASE(16, 4)
        SSM_DIAG_CASE(16, 8)
        SSM_DIAG_CASE(16, 16)
    }
#undef SSM_DIAG_CASE
    return cudaErrorInvalidValue;
}

struct Plan {
    int S, G, K, seg_len;
};
// The decomposition used for a shape (diag_scan.cu).
Plan plan_for(int64_t Bs, int64_t L, int64_t ED, int64_t N, int esz, int num_sms);

// The whole call: plan, per-segment summaries (stream-ordered scratch,
// released once the second pass is enqueued), one or two launches.
template <typename Tin, bool EXT>
cudaError_t launch_impl(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm,
                        const Tin *Cm, const float *D, float *y, int64_t Bs, int64_t L,
                        int64_t ED, int64_t N, int num_sms, const Ext &ex, cudaStream_t st) {
    const int esz = int(sizeof(Tin));
    // checkpointing for the gradients (N <= 16): the time split too, the carry
    // pass adding the carried state to a later segment's checkpoints
    Plan p = (EXT && ex.ckpt && N > 16) ? Plan{16, 1, 1, int(L)} : plan_for(Bs, L, ED, N, esz, num_sms);
    const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(dlt) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(Bm) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(Cm) % 16 == 0) && ((ED * esz) % 16 == 0) &&
                     ((N * esz) % 16 == 0) &&
                     (!EXT || !ex.z || reinterpret_cast<uintptr_t>(ex.z) % 16 == 0);
    SegSummary summ{nullptr, nullptr, nullptr};
    if (p.K == 1) {
        if (vec)
            return dispatch_sg<Tin, true, false, EXT>(p.S, p.G, x, dlt, A, Bm, Cm, D, y, Bs, int(L),
                                                      int(ED), int(N), 1, int(L), summ, ex, st);
        return dispatch_sg<Tin, false, false, EXT>(p.S, p.G, x, dlt, A, Bm, Cm, D, y, Bs, int(L),
                                                   int(ED), int(N), 1, int(L), summ, ex, st);
    }
    const size_t nsum = size_t(p.K) * size_t(Bs) * size_t(ED);
    void *scratch = nullptr;
    cudaError_t err = cudaMallocAsync(&scratch, nsum * (16 + 2) * sizeof(float), st);
    if (err != cudaSuccess) return err;
    summ.h_end = static_cast<float *>(scratch);
    summ.dsum = summ.h_end + nsum * 16;
    summ.dmin = summ.dsum + nsum;
    if (vec)
        err = dispatch_sg<Tin, true, true, EXT>(p.S, p.G, x, dlt, A, Bm, Cm, D, y, Bs, int(L),
                                                int(ED), int(N), p.K, p.seg_len, summ, ex, st);
    else
        err = dispatch_sg<Tin, false, true, EXT>(p.S, p.G, x, dlt, A, Bm, Cm, D, y, Bs, int(L),
                                                 int(ED), int(N), p.K, p.seg_len, summ, ex, st);
    cudaError_t e2 = cudaFreeAsync(scratch, st);
    return err != cudaSuccess ? err : e2;
}

}  // namespace diag
}  // namespace ssm
