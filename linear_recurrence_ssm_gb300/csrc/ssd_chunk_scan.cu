// ssd_chunk_scan.cu -- chunked scalar-decay ("SSD") scan on 5th-generation
// tensor cores (tcgen05, TMEM accumulators, TMA-fed bf16 tiles) for sm_103a.
//
// Computes, per batch row b and head h (state H_t in R^{P x N}, H_{-1} = 0),
//     H_t = exp(dt_t A_h) H_{t-1} + dt_t x_t (outer) B_t,   y_t = H_t C_t + D_h x_t
// and, when bidirectional, adds the same recurrence run from the end of the
// sequence (shared x, dt, A, B, C), counting D_h x_t once -- the sum of a
// forward and a backward SSM with shared weights plus the skip term, as the
// author describes Bi-Mamba2 in "Some questions of Bi-Mamba2 and Hydra"
// (Bi-Mamba2 issue 1), whose chunked forward pass names the stages used here
// (dA cumulative sums per direction, chunk states, state passing, chunk-scan
// output).
//
// Chunked form, for a tile of Q = 128 rows with dA_r = dt_r A_h,
// cum = inclusive prefix sum of dA in the tile, excl = cum - dA, tot = cum
// at the tile's end (every exponent below is a difference of cumulative sums
// and is <= 0 when dt A_h <= 0: the segment sums are formed by subtracting
// cumulative sums, the numerically stable way that page discusses):
//   G     = C B^T                                   (tensor core, Q x Q)
//   M[t,s]= G[t,s] dt_s (exp(cum_t - cum_s) [s <= t] + exp(excl_s - excl_t) [s >= t, reverse])
//   Y     = M X                                     (tensor core, Q x P)
//   Zf    = C S_in^T,  Zr = C R_in^T                (tensor core, Q x P)
//   y[t]  = Y[t] + exp(cum_t) Zf[t] + exp(tot - excl_t) Zr[t] + D_h x[t]
//   S_c   = B^T (w x), w_s = dt_s exp(tot - cum_s)   (tensor core, N x P)
//   S_in <- exp(tot) S_in + S_c                      (fp32, in registers)
// The reverse direction's entering states R_in come from a first sweep over
// the tiles from the last to the first: R_in <- exp(tot) R_in + B^T (w' x),
// w'_s = dt_s exp(excl_s).  Both directions read each tile of x, dt, B, C in
// place -- no reversed copy of any input is materialised.
//
// Three kernels compute it.  The unidirectional scan runs on a warp-
// specialised kernel (ws::ssd_ws_kernel below): eight math warps, an
// MMA-issuing thread each for the G / Zf and the Y / S_c streams, a copying
// thread and a warp for the per-tile vectors.  Short bidirectional sequences
// (at most four tiles, N = 64) run as two passes over independent tiles
// (ssd_bidir.cu).  Every other bidirectional call runs on
// ssd_chunk_scan_kernel: one CTA of 128 threads owns one (b, h) and walks its
// tiles in order; thread t owns tile row t (and TMEM lane t), and thread 0
// issues the TMA copies and the tensor-core MMAs.  Every wait is bounded in
// time and reports through an error word instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "ssm_common.cuh"
#include "tc_ptx.cuh"

namespace ssm {
namespace bidir {
bool supported(int64_t L, int64_t P, int64_t N);
cudaError_t launch(const __nv_bfloat16 *x, const __nv_bfloat16 *dt, const float *A_head,
                   const __nv_bfloat16 *Bm, const __nv_bfloat16 *Cm, const float *D, float *y,
                   int64_t Bs, int64_t L, int64_t H, int num_sms, const ScanOpts *opt,
                   cudaStream_t stream);
}  // namespace bidir
namespace ssd {

using namespace ssm::tc;

constexpr int kQ = 128;          // tile rows (MMA M)
constexpr int kP = 64;           // head dimension
constexpr int kThreads = 256;         // two warpgroups; both cover the 128 tile rows
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColG = 0;    // G: 128 columns
constexpr uint32_t kColY = 128;  // Y: 64 columns
constexpr uint32_t kColZf = 192; // Zf: 64
constexpr uint32_t kColZr = 256; // Zr: 64
constexpr uint32_t kColS = 320;  // chunk state S_c^T: 64
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kTile = kQ * 128;      // bytes of a 128-row x 128-byte tile region
constexpr uint32_t kStateRegion = kP * 128;

__device__ unsigned int g_device_error;   // non-zero once a bounded wait ran out
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB, see launch_noalloc
static_assert(kNoAllocScratchBytes == SSM_NOALLOC_SCRATCH_BYTES, "header and library disagree");

template <int NB>  // NB = N / 64
struct __align__(1024) Smem {
    uint8_t C[NB][kTile];       // C tile, K-major: row t, 64 n per region (128B swizzle)
    uint8_t B[2][2][kTile];     // B tiles (double buffered), rows s; region 1 stays zero when N = 64
    uint8_t X[2][kTile];        // x tiles (double buffered), rows s, 64 p (MN-major B operand)
    uint8_t Xw[kTile];          // weighted x rows
    uint8_t M[2][kTile];        // masked G, K-major: row t, s in two 64-wide regions; then y rows
    uint8_t S[NB][kStateRegion];  // forward entering state (bf16), MN-major: row n, 64 p
    uint8_t R[NB][kStateRegion];  // reverse entering state (bf16), same layout
    // per-tile vectors, double buffered by tile parity
    float cum[2][kQ];
    float excl[2][kQ];
    float dtv[2][kQ];
    float csf[2][kQ];           // column factors of the forward decay mask
    float csr[2][kQ];           // column factors of the reverse decay mask
    float wsum[kThreads / 32];
    uint64_t bar_x[2];          // x tile landed (one per buffer)
    uint64_t bar_c;             // C tile (and the reverse entering state) landed
    uint64_t bar_b[2];          // B tile landed (one per buffer)
    uint64_t bar_g;             // G, Zf, Zr of a tile finished
    uint64_t bar_m2;            // Y and S_c of a tile finished
    uint64_t bar_fin;           // every MMA issued so far finished (error path)
    uint32_t tmem_base;
};

struct Params {
    const __nv_bfloat16 *dt;
    const float *A;
    const float *D;
    float *y;
    uint8_t *rstate;   // reverse entering states, [Bs*H][nc][NB * kStateRegion] (bidirectional)
    int L, H, nc;
    // options (kernels built with them only): dt <- clamp(softplus(dt + bias)),
    // y <- y * silu(z), initial / final state (Bs, H, P, N) fp32
    const float *dt_bias;
    const __nv_bfloat16 *z;
    const float *h0;
    float *h_final;
    float dt_min, dt_max;
    int dt_softplus, dt_limit;
    int G;             // groups of B, C; head h reads group h / (H / G)
};

// Scan options: see ScanOpts (z is bf16 here; states are (Bs, H, P, N)).
using Options = ScanOpts;

// Byte offset of element (row, col) of a 128-byte-swizzled tile whose rows
// are 128 bytes (64 bf16): the 16-byte chunk index is XORed with row % 8.
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return uint32_t(row) * 128u + ((uint32_t((col >> 3) ^ (row & 7))) << 4) + uint32_t(col & 7) * 2u;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t w) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&w);
    return __bfloat1622float2(v);
}

// Inclusive prefix sum of one value per tile row.  Both warpgroups hold the
// same 128 values (thread and thread + 128 share row tid % 128) and compute
// the same sums; returns the total too.
__device__ __forceinline__ float tile_inclusive_scan(float v, float *wsum, float *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    const int w0 = warp & ~3, wr = warp & 3;
    float off = 0.0f, tot = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float s = wsum[w0 + w];
        off += (w < wr) ? s : 0.0f;
        tot += s;
    }
    *total = tot;
    return v + off;
}

// Scale half `half` (four of the eight 16-byte chunks) of row s of the x tile
// by w into the Xw tile.  Both tiles share the same swizzle and the scale is
// uniform along the row, so chunks are processed in place; the XOR with
// s % 8 makes the 32 rows a warp touches at once fall in different banks.
__device__ __forceinline__ void scale_row(const uint8_t *X, uint8_t *Xw, int s, float w, int half) {
    const uint4 *src = reinterpret_cast<const uint4 *>(X + s * 128);
    uint4 *dst = reinterpret_cast<uint4 *>(Xw + s * 128);
#pragma unroll
    for (int jj = 4 * half; jj < 4 * half + 4; ++jj) {
        const int j = jj ^ (s & 7);
        uint4 v = src[j];
        float2 a = unpack_bf16(v.x), b = unpack_bf16(v.y), c = unpack_bf16(v.z), d = unpack_bf16(v.w);
        v.x = pack_bf16(a.x * w, a.y * w);
        v.y = pack_bf16(b.x * w, b.y * w);
        v.z = pack_bf16(c.x * w, c.y * w);
        v.w = pack_bf16(d.x * w, d.y * w);
        dst[j] = v;
    }
}

// Store entries [p0, p0 + 32) of state row n (thread n holds them, fp32)
// as bf16 into an MN-major state image: 128-byte rows n of 64 p, 128-byte
// swizzle (the 16-byte chunk index XORed with n % 8) -- the layout of a TMA
// x tile, so the image is the B operand of Zf = C S_in^T directly.
template <int NB>
__device__ __forceinline__ void store_state_bf16(uint8_t (*img)[kStateRegion], int n, int p0,
                                                 const float (&s)[32]) {
    uint8_t *rowp = &img[0][0] + n * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int chunk = (p0 >> 3) + j;
        *reinterpret_cast<uint4 *>(rowp + ((chunk ^ (n & 7)) << 4)) =
            make_uint4(pack_bf16(s[8 * j], s[8 * j + 1]), pack_bf16(s[8 * j + 2], s[8 * j + 3]),
                       pack_bf16(s[8 * j + 4], s[8 * j + 5]), pack_bf16(s[8 * j + 6], s[8 * j + 7]));
    }
}

// Waits of the CTA: every thread polls the mbarrier (bounded in time), and
// the CTA agrees on the outcome so that all threads leave together.
#define SSM_CTA_WAIT(bar, ph)                                                             \
    do {                                                                                  \
        ok = mbar_wait_bounded(&(bar), (ph), &abort_flag, kWaitLimitNs);                  \
        (ph) ^= 1u;                                                                       \
        if (__syncthreads_or(!ok)) {                                                      \
            ok = false;                                                                   \
            goto done;                                                                    \
        }                                                                                 \
    } while (0)

// The bidirectional scan for sequences the two-pass kernels do not take:
// first the reverse sweep from the last tile (entering states R_in of every
// tile, stored bf16 in scratch), then the forward sweep with the outputs.
// (The options that go with state input / output are not accepted with the
// bidirectional scan, so neither appears here.)
template <int NB, bool EXT>
__global__ void __launch_bounds__(kThreads, 1)
ssd_chunk_scan_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                      const Params prm) {
    constexpr int N = NB * 64;
    extern __shared__ uint8_t smem_raw[];
    Smem<NB> &sm = *reinterpret_cast<Smem<NB> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int row = tid & (kQ - 1);      // tile row == TMEM lane of this thread
    const int wg = tid >> 7;             // warpgroup: which half of the columns it handles
    const int bh = blockIdx.x;
    const int b = bh / prm.H;
    const int h = bh % prm.H;
    const int L = prm.L;
    const int nc = prm.nc;
    const int grp = h / (prm.H / prm.G);          // this head's group of B, C
    const float Ah = prm.A[h] * SSM_LOG2E;        // decays are exp2 of log2e-scaled sums
    const float Dh = prm.D ? prm.D[h] : 0.0f;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const size_t rstride = size_t(NB) * kStateRegion;

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&sm.bar_x[0], 1);
        mbar_init(&sm.bar_x[1], 1);
        mbar_init(&sm.bar_c, 1);
        mbar_init(&sm.bar_b[0], 1);
        mbar_init(&sm.bar_b[1], 1);
        mbar_init(&sm.bar_g, 1);
        mbar_init(&sm.bar_m2, 1);
        mbar_init(&sm.bar_fin, 1);
        mbar_fence_init();
        prefetch_tmap(&tmC);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmY);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    // The second B region (n = 64..127) of both buffers is read as zero rows
    // when N = 64.
    if (NB == 1) {
        for (int i = tid; i < int(kTile / 16); i += kThreads) {
            reinterpret_cast<uint4 *>(sm.B[0][1])[i] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4 *>(sm.B[1][1])[i] = make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    uint32_t ph_x[2] = {0, 0}, ph_c = 0, ph_b[2] = {0, 0}, ph_g = 0, ph_m2 = 0;
    bool ok = true;

    const uint32_t sC = smem_addr(sm.C);
    const uint32_t sXw = smem_addr(sm.Xw), sM = smem_addr(sm.M), sS = smem_addr(sm.S);
    const uint32_t sR = smem_addr(sm.R);
    constexpr uint32_t idG = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idZ = idesc_bf16_f32(128, 64, false, true);
    constexpr uint32_t idY = idesc_bf16_f32(128, 64, false, true);
    constexpr uint32_t idS = idesc_bf16_f32(128, 64, true, true);

    // ---- copies issued by thread 0 -------------------------------------------------
    auto load_x = [&](int c, int buf) {
        mbar_arrive_expect_tx(&sm.bar_x[buf], kTile);
        tma_load_4d(sm.X[buf], &tmX, &sm.bar_x[buf], 0, h, c * kQ, b);
    };
    auto load_b = [&](int c, int buf) {
        mbar_arrive_expect_tx(&sm.bar_b[buf], NB * kTile);
#pragma unroll
        for (int r = 0; r < NB; ++r)
            tma_load_4d(sm.B[buf][r], &tmB, &sm.bar_b[buf], r * 64, grp, c * kQ, b);
    };
    auto load_c = [&](int c, bool with_r) {
        mbar_arrive_expect_tx(&sm.bar_c, NB * kTile + (with_r ? uint32_t(rstride) : 0u));
#pragma unroll
        for (int r = 0; r < NB; ++r) tma_load_4d(sm.C[r], &tmC, &sm.bar_c, r * 64, grp, c * kQ, b);
        if (with_r)
            bulk_load(sm.R, prm.rstate + (size_t(bh) * nc + c) * rstride, uint32_t(rstride),
                      &sm.bar_c);
    };
    const float dbias = (EXT && prm.dt_bias) ? prm.dt_bias[h] : 0.0f;
    auto load_dt = [&](int c) {
        const int r = c * kQ + row;
        if (r >= L) return 0.0f;   // rows past L: no decay, no input
        float d = __bfloat162float(prm.dt[(int64_t(b) * L + r) * prm.H + h]);
        if (EXT) {
            d += dbias;
            if (prm.dt_softplus) d = softplus_fast(d);
            if (prm.dt_limit) d = fminf(fmaxf(d, prm.dt_min), prm.dt_max);
        }
        return d;
    };
    // Per-tile cumulative sums of dt * A (log2 units) into the vectors of
    // parity p, and the column factors of the decay mask.  Rows past L have
    // dt = 0 (no decay, no input).  Contains a CTA barrier.
    auto tile_prep = [&](float dv, int p, float *tot_out) {
        const float dA = dv * Ah;
        float tot;
        const float cum = tile_inclusive_scan(dA, sm.wsum, &tot);
        if (wg == 0) {
            sm.cum[p][row] = cum;
            sm.excl[p][row] = cum - dA;
            sm.dtv[p][row] = dv;
            __syncwarp();
            // Column factors for the blocks of the mask below (above) the
            // diagonal: for s in a 32-column block that ends at row r (starts
            // at row r') and t past that block,
            //   exp2(cum_t - cum_s)   = exp2(cum_t - cum_r)   * exp2(cum_r - cum_s),
            //   exp2(excl_s - excl_t) = exp2(excl_s - excl_r') * exp2(excl_r' - excl_t),
            // and both factors are <= 1.  Diagonal blocks use the direct form.
            // (Rows r, r' are in the same warp as s.)
            const int s = row;
            sm.csf[p][s] = ex2(sm.cum[p][s | 31] - cum) * dv;
            sm.csr[p][s] = ex2(cum - dA - sm.excl[p][s & ~31]) * dv;
        }
        *tot_out = tot;
    };
    // S_c^T = B^T Xw (tensor core, N x P) from B buffer `bb`.
    auto issue_state_mma = [&](int bb) {
        const uint32_t sB = smem_addr(sm.B[bb]);
#pragma unroll
        for (int kk = 0; kk < kQ / 16; ++kk) {
            const uint64_t a = smem_desc(sB + kk * 2048, kTile, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(sXw + kk * 2048, kTile, 1024, kSwizzle128B);
            mma_bf16_ss(tmem + kColS, a, bd, idS, kk > 0);
        }
    };
    // G = C B^T from B buffer `bb`.
    auto issue_g = [&](int bb) {
        const uint32_t sB = smem_addr(sm.B[bb]);
#pragma unroll
        for (int kk = 0; kk < N / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kTile + (kk & 3) * 32;
            mma_bf16_ss(tmem + kColG, smem_desc(sC + koff, 16, 1024, kSwizzle128B),
                        smem_desc(sB + koff, 16, 1024, kSwizzle128B), idG, kk > 0);
        }
    };
    // Zf = C S_in^T, Zr = C R_in^T.
    auto issue_z = [&](bool has_s, bool has_r) {
#pragma unroll
        for (int kk = 0; kk < N / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kTile + (kk & 3) * 32;
            const uint64_t a = smem_desc(sC + koff, 16, 1024, kSwizzle128B);
            // state images: 16 rows of n per K step
            if (has_s)
                mma_bf16_ss(tmem + kColZf, a, smem_desc(sS + kk * 2048, kTile, 1024, kSwizzle128B), idZ, kk > 0);
            if (has_r)
                mma_bf16_ss(tmem + kColZr, a, smem_desc(sR + kk * 2048, kTile, 1024, kSwizzle128B), idZ, kk > 0);
        }
    };
    // State update for column n = row, rows p in [32 wg, 32 wg + 32):
    // st = e * st + S_c^T[n, p] (TMEM lane n, columns kColS + p).
    auto state_update = [&](float *st, float e) {
        uint32_t v[32];
        tmem_ld32_async(tmem + lane_base + kColS + wg * 32, v);
        tmem_wait_tie(v);
#pragma unroll
        for (int j = 0; j < 32; ++j) st[j] = fmaf(e, st[j], __uint_as_float(v[j]));
    };

    float st[32];   // rows [32 wg, 32 wg + 32) of this thread's state column (n = row), fp32

    // ---------------- reverse sweep: entering states of the reverse scan -------------
    {
#pragma unroll
        for (int p = 0; p < 32; ++p) st[p] = 0.0f;
        if (tid == 0) {
            load_x(nc - 1, (nc - 1) & 1);
            load_b(nc - 1, 0);
        }
        float dv = load_dt(nc - 1);
        for (int c = nc - 1; c >= 0; --c) {
            const int xb = c & 1;
            if (tid == 0 && c >= 1) load_x(c - 1, xb ^ 1);
            float tot;
            tile_prep(dv, 0, &tot);
            if (c >= 1) dv = load_dt(c - 1);
            // R_in of this tile (state entering from the right) -> scratch.
            if (c < nc - 1) {
                if (row < N) store_state_bf16<NB>(sm.R, row, wg * 32, *reinterpret_cast<float(*)[32]>(st));
                __syncthreads();
                uint4 *dst = reinterpret_cast<uint4 *>(prm.rstate + (size_t(bh) * nc + c) * rstride);
                const uint4 *src = reinterpret_cast<const uint4 *>(sm.R);
                for (int i = tid; i < int(rstride / 16); i += kThreads) dst[i] = src[i];
                fence_proxy_async_all();
            }
            SSM_CTA_WAIT(sm.bar_x[xb], ph_x[xb]);
            scale_row(sm.X[xb], sm.Xw, row, ex2(sm.excl[0][row]) * sm.dtv[0][row], wg);
            fence_proxy_async_smem();
            SSM_CTA_WAIT(sm.bar_b[0], ph_b[0]);
            if (tid == 0) {
                tc_fence_after_sync();
                issue_state_mma(0);
                mma_commit(&sm.bar_m2);
            }
            SSM_CTA_WAIT(sm.bar_m2, ph_m2);
            tc_fence_after_sync();
            if (tid == 0 && c >= 1) load_b(c - 1, 0);
            if (row < N) state_update(st, ex2(tot));
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncthreads();
        }
    }

    // ---------------- forward sweep with the outputs ----------------------------------
    // Software pipeline over the tiles: while the mask of tile c is built, the
    // copies of tile c + 1 land; G of tile c + 1 runs on the tensor core behind
    // Y and S_c of tile c, and Zf, Zr of tile c + 1 right after the state
    // update, so that the mask pass of tile c + 1 can start at once.
#pragma unroll
    for (int p = 0; p < 32; ++p) st[p] = 0.0f;
    fence_proxy_async_smem();
    if (tid == 0) {
        load_x(0, 0);
        load_c(0, nc > 1);
        load_b(0, 0);
        if (nc > 1) {
            load_b(1, 1);
            load_x(1, 1);
        }
    }
    {
    float dv = load_dt(0);
    float tot_cur, tot_nxt = 0.0f;
    tile_prep(dv, 0, &tot_cur);
    if (nc > 1) dv = load_dt(1);
    SSM_CTA_WAIT(sm.bar_x[0], ph_x[0]);
    scale_row(sm.X[0], sm.Xw, row, ex2(tot_cur - sm.cum[0][row]) * sm.dtv[0][row], wg);
    fence_proxy_async_smem();
    SSM_CTA_WAIT(sm.bar_c, ph_c);
    SSM_CTA_WAIT(sm.bar_b[0], ph_b[0]);
    if (tid == 0) {
        tc_fence_after_sync();
        issue_g(0);
        issue_z(false, nc > 1);
        mma_commit(&sm.bar_g);
    }
    for (int c = 0; c < nc; ++c) {
        const int c0 = c * kQ;
        const int par = c & 1;      // buffers and per-tile vectors of tile c
        const bool more = c + 1 < nc;
        const bool has_s = c > 0;
        const bool has_r = c < nc - 1;
        // The previous tile's output rows staged in the mask buffer must have
        // been read by their store before the mask pass overwrites it.
        if (tid == 0) bulk_wait_read0();
        SSM_CTA_WAIT(sm.bar_g, ph_g);          // G, Zf, Zr of tile c; C and R buffers free
        tc_fence_after_sync();
        if (tid == 0 && more) load_c(c + 1, c + 1 < nc - 1);

        // Decay mask on row t of G -> bf16 M (K-major, swizzled).
        {
            const int t = row;
            const int tb = t >> 5;                 // warp-uniform: the warp owns rows 32 tb..
            const float *cum = sm.cum[par];
            const float *excl = sm.excl[par];
            const float *dtv = sm.dtv[par];
            const float cum_t = cum[t], excl_t = excl[t];
            // Blocks {0, 3} to warpgroup 0 and {1, 2} to warpgroup 1 (every
            // block of the two-sided mask is needed).
            const int sbs[2] = {wg == 0 ? 0 : 1, wg == 0 ? 3 : 2};
            uint32_t gr[2][32];
            tmem_ld32_async(tmem + lane_base + kColG + sbs[0] * 32, gr[0]);
            tmem_ld32_async(tmem + lane_base + kColG + sbs[1] * 32, gr[1]);
            tmem_wait_tie(gr[0]);
            reg_tie(gr[1]);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int sb = sbs[i];
                uint32_t packed[16];
                {
                    float m[32];
                    if (sb == tb) {
                        // diagonal block: direct differences of cumulative sums
                        const float4 *c4 = reinterpret_cast<const float4 *>(cum + sb * 32);
                        const float4 *e4 = reinterpret_cast<const float4 *>(excl + sb * 32);
                        const float4 *d4 = reinterpret_cast<const float4 *>(dtv + sb * 32);
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            const float4 cs = c4[j4], ds = d4[j4];
                            const float4 es = e4[j4];
                            const float csv[4] = {cs.x, cs.y, cs.z, cs.w};
                            const float esv[4] = {es.x, es.y, es.z, es.w};
                            const float dsv[4] = {ds.x, ds.y, ds.z, ds.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int s = sb * 32 + 4 * j4 + q;
                                float w = (s <= t) ? ex2(cum_t - csv[q]) : 0.0f;
                                if (s >= t) w += ex2(esv[q] - excl_t);
                                m[4 * j4 + q] = __uint_as_float(gr[i][4 * j4 + q]) * (w * dsv[q]);
                            }
                        }
                    } else {
                        const bool fwd = sb < tb;
                        const float e = fwd ? ex2(cum_t - cum[sb * 32 + 31])
                                            : ex2(excl[sb * 32] - excl_t);
                        const float4 *f4 = reinterpret_cast<const float4 *>((fwd ? sm.csf[par] : sm.csr[par]) + sb * 32);
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            const float4 f = f4[j4];
                            m[4 * j4 + 0] = __uint_as_float(gr[i][4 * j4 + 0]) * (e * f.x);
                            m[4 * j4 + 1] = __uint_as_float(gr[i][4 * j4 + 1]) * (e * f.y);
                            m[4 * j4 + 2] = __uint_as_float(gr[i][4 * j4 + 2]) * (e * f.z);
                            m[4 * j4 + 3] = __uint_as_float(gr[i][4 * j4 + 3]) * (e * f.w);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) packed[j] = pack_bf16(m[2 * j], m[2 * j + 1]);
                }
                uint8_t *reg = sm.M[sb >> 1];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int col = (sb & 1) * 32 + q * 8;   // column inside the 64-wide region
                    *reinterpret_cast<uint4 *>(reg + swz(t, col)) =
                        make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // Y = M X and S_c^T = B^T Xw of tile c.
        if (tid == 0) {
            tc_fence_after_sync();
            const uint32_t sX = smem_addr(sm.X[par]);
#pragma unroll
            for (int kk = 0; kk < kQ / 16; ++kk) {
                const uint64_t a = smem_desc(sM + (kk >> 2) * kTile + (kk & 3) * 32, 16, 1024, kSwizzle128B);
                const uint64_t bd = smem_desc(sX + kk * 2048, kTile, 1024, kSwizzle128B);
                mma_bf16_ss(tmem + kColY, a, bd, idY, kk > 0);
            }
            issue_state_mma(par);
            mma_commit(&sm.bar_m2);
        }
        // The gate's row for the epilogue (optional), loaded while the MMAs run.
        uint4 zq[4];
        const bool gate = EXT && prm.z != nullptr;
        if (gate) {
            const int r = c0 + row;
            const uint4 *zp = reinterpret_cast<const uint4 *>(
                prm.z + ((int64_t(b) * L + (r < L ? r : L - 1)) * prm.H + h) * kP + wg * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) zq[j] = zp[j];
        }
        // Meanwhile: vectors of tile c + 1, then its G behind them.
        if (more) {
            tile_prep(dv, par ^ 1, &tot_nxt);
            if (c + 2 < nc) dv = load_dt(c + 2);
            SSM_CTA_WAIT(sm.bar_c, ph_c);
            SSM_CTA_WAIT(sm.bar_b[par ^ 1], ph_b[par ^ 1]);
            if (tid == 0) {
                tc_fence_after_sync();
                issue_g(par ^ 1);
            }
        }
        SSM_CTA_WAIT(sm.bar_m2, ph_m2);
        tc_fence_after_sync();
        if (tid == 0 && c + 2 < nc) load_b(c + 2, par);

        // Epilogue: row t of y, columns p in [32 wg, 32 wg + 32).
        {
            const int t = row;
            const int q = wg;
            uint32_t yv[32], zf[32], zr[32];
            tmem_ld32_async(tmem + lane_base + kColY + q * 32, yv);
            if (has_s) tmem_ld32_async(tmem + lane_base + kColZf + q * 32, zf);
            if (has_r) tmem_ld32_async(tmem + lane_base + kColZr + q * 32, zr);
            const float ef = ex2(sm.cum[par][t]);
            const float er = ex2(tot_cur - sm.excl[par][t]);
            float xr[32];
            const uint4 *xs = reinterpret_cast<const uint4 *>(sm.X[par] + t * 128);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 v = xs[(q * 4 + j) ^ (t & 7)];
                const float2 a = unpack_bf16(v.x), bb = unpack_bf16(v.y),
                             cc = unpack_bf16(v.z), dd = unpack_bf16(v.w);
                xr[8 * j + 0] = a.x; xr[8 * j + 1] = a.y; xr[8 * j + 2] = bb.x; xr[8 * j + 3] = bb.y;
                xr[8 * j + 4] = cc.x; xr[8 * j + 5] = cc.y; xr[8 * j + 6] = dd.x; xr[8 * j + 7] = dd.y;
            }
            tmem_wait_tie(yv);
            reg_tie(zf);
            reg_tie(zr);
            float out[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                float v = fmaf(Dh, xr[j], __uint_as_float(yv[j]));
                if (has_s) v = fmaf(ef, __uint_as_float(zf[j]), v);
                if (has_r) v = fmaf(er, __uint_as_float(zr[j]), v);
                out[j] = v;
            }
            if (gate) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w4[4] = {zq[j].x, zq[j].y, zq[j].z, zq[j].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 zz = unpack_bf16(w4[k]);
                        out[8 * j + 2 * k] *= silu_fast(zz.x);
                        out[8 * j + 2 * k + 1] *= silu_fast(zz.y);
                    }
                }
            }
            // Stage the row in the (now free) mask buffer as a 128-byte-swizzled
            // [128 rows][32 fp32] tile per warpgroup; one TMA store per tile
            // writes it out coalesced (rows past L are clipped by the store).
            uint8_t *ys = sm.M[wg] + t * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4 *>(ys + ((j ^ (t & 7)) << 4)) =
                    make_float4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
        }
        // State passing: column n = row of S_in, rows [32 wg, 32 wg + 32).
        if (row < N) {
            state_update(st, ex2(tot_cur));
            store_state_bf16<NB>(sm.S, row, wg * 32, *reinterpret_cast<float(*)[32]>(st));
        }
        // Weighted x rows of tile c + 1 (its S_c reads them).
        if (more) {
            SSM_CTA_WAIT(sm.bar_x[par ^ 1], ph_x[par ^ 1]);
            scale_row(sm.X[par ^ 1], sm.Xw, row,
                      ex2(tot_nxt - sm.cum[par ^ 1][row]) * sm.dtv[par ^ 1][row], wg);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tma_store_4d(&tmY, sm.M[0], 0, h, c0, b);
            tma_store_4d(&tmY, sm.M[1], 32, h, c0, b);
            bulk_commit();
            if (c + 2 < nc) load_x(c + 2, par);
            if (more) {
                tc_fence_after_sync();
                issue_z(true, c + 1 < nc - 1);
                mma_commit(&sm.bar_g);
            }
        }
        tot_cur = tot_nxt;
    }
    }

done:
    if (tid == 0) bulk_wait0();
    if (!ok && tid == 0) {
        abort_flag = 1;
        atomicOr(&g_device_error, 1u);
        // MMAs still in flight after a timeout: give them a bounded chance
        // to finish before the tensor memory is released.
        mma_commit(&sm.bar_fin);
        volatile int never = 0;
        (void)mbar_wait_bounded(&sm.bar_fin, 0, &never, 100000000ull);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Unidirectional kernel: eight math warps, an MMA-issuing warp, a copying warp
// ---------------------------------------------------------------------------
// The same computation as ssd_chunk_scan_kernel for the forward scan.  Eight
// math warps share every per-tile stage: warps w and w + 4 read TMEM lane
// quarter q = w % 4 (tile rows / state rows 32 q .. 32 q + 31) and split the
// work of those rows by column halves (hf = w / 4):
//   the decay mask: row quarter q has causal 32 x 32 blocks sb = 0..q; the
//     half-0 warp computes the diagonal block (direct exponentials), the
//     half-1 warp the blocks below it (products of two factors, cheaper), so
//     no warp has more than about one diagonal block's work;
//   the weighted x rows, the fp32 state update and its bf16 image, the
//     output rows y = Y + e^{cum} Zf: columns 32 hf .. 32 hf + 31.
// Per tile c the warps (1) weigh the x rows of tile c + 1 and compute its
// mask in registers while Y(c), S_c(c) run on the tensor core, (2) wait for
// them, update the state (the image of the state entering tile c + 1), store
// the mask of tile c + 1 into tensor memory -- so Zf(c + 1), Y(c + 1) and
// S_c(c + 1) start at once -- and (3) write the outputs of tile c while they
// run.  Two threads issue the tcgen05.mma products as soon as their inputs
// are ready -- warp 8 the G and Zf streams, warp 11 the Y and S_c products --
// and warp 9 (one thread) every TMA copy as soon as its buffer is free.  The mask M lives in tensor memory and is the A operand of Y = M X;
// D x rides on its diagonal.  Y and Zf have two accumulators (by tile
// parity) so the products of tile c + 1 run while the outputs of tile c are
// read; the weighted rows Xw are double-buffered, and once S_c(c) has run
// the outputs of tile c are staged in tile c's buffer and leave by TMA
// stores, so that no warp waits on its global stores.
namespace ws {

constexpr int kMath = 256;             // math threads (warps 0..7)
constexpr int kThreads = kMath + 128;  // + warpgroup 2: warp 8 issues G and Zf, warp 9 copies,
                                       //   warp 10 computes the per-tile vectors, warp 11
                                       //   issues Y and S_c
// Registers: the register file is split between the SM's four schedulers,
// one warp of each warpgroup per scheduler; the CTA is launched with 168 per
// thread (3 warps x 32 x 168 <= 16384 per scheduler) and setmaxnreg moves
// registers from the control warpgroup to the two math warpgroups.
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kCtrlRegs = 40;
constexpr uint32_t kMathRegs = 232;
static_assert(kCtrlRegs + 2 * kMathRegs <= 3 * kLaunchRegs,
              "the register split must fit in what the CTA is launched with");
constexpr int kSlots = 3;        // per-tile vectors in flight (tile c uses slot c % 3)
constexpr int kXBufs = 2;        // x tiles in flight (tile c uses buffer c % 2)

// Tensor-memory columns: G (fp32, 128), Y and Zf by tile parity (fp32, 64
// each), the chunk state S_c^T (fp32, 64) and the mask M (bf16 pairs, 64).
constexpr uint32_t kWsG = 0, kWsY0 = 128, kWsY1 = 192, kWsZ0 = 256, kWsZ1 = 320, kWsS = 384,
                   kWsM = 448;

template <int NB>
struct __align__(1024) Smem {
    uint8_t C[2][NB][kTile];    // C tiles (double buffered), K-major rows t
    uint8_t B[2][2][kTile];     // B tiles (double buffered); region 1 zero when N = 64
    uint8_t X[kXBufs][kTile];   // x tiles (MN-major B operand of Y), tile c in c % 2
    uint8_t Xw[2][kTile];       // weighted x rows of tile c in c % 2; then tile c's y staging
    uint8_t S[NB][kStateRegion];    // entering state image
    float cum[kSlots][kQ];
    float dtv[kSlots][kQ];
    float csf[kSlots][kQ];
    float tot[kSlots];
    uint64_t bar_c[2], bar_b[2], bar_x[kXBufs];      // TMA copies landed
    // Products finished and hand-offs.  A parity wait cannot tell phase k
    // from phase k + 2, so no barrier may complete twice before every waiter
    // has seen the first: bar_xw and bar_m2 are one per tile parity, because
    // the weighted rows of tile c + 1 are written before Y(c) is issued, and
    // the copying thread is the only waiter on bar_m2 that nothing else holds
    // back; each of the others completes again only after its waiters moved on.
    uint64_t bar_g, bar_m2[2], bar_z[2];
    uint64_t bar_gfree, bar_mfull[2], bar_xw[2], bar_st;   // bar_mfull[c & 1]: mask of tile c stored
    uint64_t bar_vec[kSlots];                        // vectors of a slot written
    uint64_t bar_pair[4];                            // the two warps of a lane quarter: their
                                                     //   output stores have read the staging
    uint64_t bar_fin[2];                             // error path (one per issuing thread)
    uint32_t tmem_base;
};

// Non-blocking test of whether the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Half `hf` (32 p) of row n of an MN-major bf16 state image (64 p, 128-byte
// swizzle) from the 32 fp32 values a thread holds.
__device__ __forceinline__ void put_state_half(uint8_t *img, int n, int hf, const float (&s)[32]) {
    uint8_t *rowp = img + n * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4 *>(rowp + (((4 * hf + j) ^ (n & 7)) << 4)) =
            make_uint4(pack_bf16(s[8 * j], s[8 * j + 1]), pack_bf16(s[8 * j + 2], s[8 * j + 3]),
                       pack_bf16(s[8 * j + 4], s[8 * j + 5]), pack_bf16(s[8 * j + 6], s[8 * j + 7]));
}

// silu(z) = z sigmoid(z), sigmoid(z) = (1 + tanh(z / 2)) / 2: one
// special-function instruction (the hardware tanh approximation, relative
// error about 2^-11) instead of an exponential and a reciprocal.  The gate
// multiplies an fp32 output that came through bf16 operands.
__device__ __forceinline__ float silu_tanh(float z) {
    float th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * z));
    return z * fmaf(0.5f, th, 0.5f);
}

// a * b for two packed fp32 pairs (one instruction on sm_100-family cores).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)),
          "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&r);
}

template <int NB>
struct Ctx {
    Smem<NB> &sm;
    const Params &prm;
    int b, h, grp, bh, L, nc;
    float Ah, Dh, dbias;
    uint32_t tmem;
    volatile int *abort;
    const CUtensorMap *tmY;   // y (fp32), box 16 p x 32 rows, 64-byte swizzle
};

#define WS_WAIT(bar, ph)                                                                  \
    do {                                                                                  \
        if (!mbar_wait_bounded(&(bar), (ph), cx.abort, kWaitLimitNs)) return false;       \
        (ph) ^= 1u;                                                                       \
    } while (0)
// The same for barrier i of an array whose phases are the bits of `bits`
// (a register, where an array indexed at run time would go to local memory).
#define WS_WAIT_I(bar, bits, i)                                                           \
    do {                                                                                  \
        if (!mbar_wait_bounded(&(bar), ((bits) >> (i)) & 1u, cx.abort, kWaitLimitNs))    \
            return false;                                                                 \
        (bits) ^= 1u << (i);                                                              \
    } while (0)

// ---- the issuing thread -------------------------------------------------------------
template <int NB, bool EXT>
__device__ __forceinline__ bool issuer_role(Ctx<NB> &cx, bool has_h0) {
    constexpr int N = NB * 64;
    auto &sm = cx.sm;
    const int nc = cx.nc;
    const uint32_t tmem = cx.tmem;
    constexpr uint32_t idG = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idZ = idesc_bf16_f32(128, 64, false, true);
    uint32_t ph_c = 0, ph_b = 0;              // phase bits, one per buffer
    uint32_t ph_gfree = 0, ph_st = 0;

    auto issue_g = [&](int buf) {
        const uint32_t sC = smem_addr(sm.C[buf]), sB = smem_addr(sm.B[buf]);
#pragma unroll
        for (int kk = 0; kk < N / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kTile + (kk & 3) * 32;
            mma_bf16_ss(tmem + kWsG, smem_desc(sC + koff, 16, 1024, kSwizzle128B),
                        smem_desc(sB + koff, 16, 1024, kSwizzle128B), idG, kk > 0);
        }
    };
    auto issue_z = [&](int buf) {    // Zf of the tile whose parity is buf
        const uint32_t sC = smem_addr(sm.C[buf]), sS = smem_addr(sm.S);
        const uint32_t zcol = buf ? kWsZ1 : kWsZ0;
#pragma unroll
        for (int kk = 0; kk < N / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kTile + (kk & 3) * 32;
            mma_bf16_ss(tmem + zcol, smem_desc(sC + koff, 16, 1024, kSwizzle128B),
                        smem_desc(sS + kk * 2048, kTile, 1024, kSwizzle128B), idZ, kk > 0);
        }
    };
    WS_WAIT_I(sm.bar_c[0], ph_c, 0);
    WS_WAIT_I(sm.bar_b[0], ph_b, 0);
    tc_fence_after_sync();
    issue_g(0);
    mma_commit(&sm.bar_g);
    WS_WAIT(sm.bar_st, ph_st);                  // the initial state image (if any)
    if (has_h0) {
        tc_fence_after_sync();
        issue_z(0);
    }
    mma_commit(&sm.bar_z[0]);
    // Two streams of products, each issued as soon as its inputs are ready
    // (non-blocking polls, so that a late input of one stream does not hold
    // up the other); Y(c) and S_c(c) are issued by another thread:
    //   G(c):         G(c - 1) read by the math warps, C(c) and B(c) landed;
    //   Zf(c):        state image of tile c written (C(c) landed: G(c) issued);
    //                 its end is signalled on its own barrier, bar_z.
    int g_next = 1, z_next = 1;
    uint64_t t_idle = 0;
    uint32_t idle_passes = 0;
    while (g_next < nc || z_next < nc) {
        bool progress = false;
        if (z_next < nc && g_next > z_next && mbar_test_wait(&sm.bar_st, ph_st)) {
            ph_st ^= 1u;
            tc_fence_after_sync();
            issue_z(z_next & 1);
            mma_commit(&sm.bar_z[z_next & 1]);
            ++z_next;
            progress = true;
        }
        if (g_next < nc && mbar_test_wait(&sm.bar_gfree, ph_gfree) &&
            mbar_test_wait(&sm.bar_c[g_next & 1], (ph_c >> (g_next & 1)) & 1u) &&
            mbar_test_wait(&sm.bar_b[g_next & 1], (ph_b >> (g_next & 1)) & 1u)) {
            ph_gfree ^= 1u;
            ph_c ^= 1u << (g_next & 1);
            ph_b ^= 1u << (g_next & 1);
            tc_fence_after_sync();
            issue_g(g_next & 1);
            mma_commit(&sm.bar_g);
            ++g_next;
            progress = true;
        }
        if (progress) {
            t_idle = 0;
            idle_passes = 0;
        } else if ((++idle_passes & 255u) == 0) {
            // the wall clock is read only now and then: it is slow to read,
            // and a slow poll answers late to the math warps' hand-offs
            const uint64_t now = globaltimer_ns();
            if (t_idle == 0) t_idle = now;
            else if (now - t_idle > kWaitLimitNs || *cx.abort) return false;
        }
    }
    return true;
}

// ---- the thread issuing Y and S_c ---------------------------------------------------------
// Y(c), S_c(c) once mask(c) is stored, the weighted rows of tile c are
// written and x(c) has landed.  The math warps store mask(c) after reading
// G(c), so G(c) has ended by then, and the end of Y(c), S_c(c) also means
// the end of G(c).  (A thread of its own: the mask hand-off is on the
// per-tile chain, and a thread that also polls the other streams answers
// it late.)
template <int NB, bool EXT>
__device__ __forceinline__ bool issuer_ys_role(Ctx<NB> &cx) {
    auto &sm = cx.sm;
    const int nc = cx.nc;
    const uint32_t tmem = cx.tmem;
    constexpr uint32_t idY = idesc_bf16_f32(128, 64, false, true);
    constexpr uint32_t idS = idesc_bf16_f32(128, 64, true, true);
    uint32_t ph_mfull = 0, ph_xw = 0, ph_x = 0;   // one bit per buffer
    for (int c = 0; c < nc; ++c) {
        const int xb = c % kXBufs, yp = c & 1;
        WS_WAIT_I(sm.bar_mfull[yp], ph_mfull, yp);
        WS_WAIT_I(sm.bar_xw[yp], ph_xw, yp);
        WS_WAIT_I(sm.bar_x[xb], ph_x, xb);
        tc_fence_after_sync();
        // Y = M X: A = the mask in tensor memory (row t, 8 columns = 16 s per
        // K step), B = the x tile (MN-major: rows s, 64 p)
        const uint32_t sX = smem_addr(sm.X[xb]);
        const uint32_t dcol = (c & 1) ? kWsY1 : kWsY0;
#pragma unroll
        for (int kk = 0; kk < kQ / 16; ++kk)
            mma_bf16_ts(tmem + dcol, tmem + kWsM + kk * 8,
                        smem_desc(sX + kk * 2048, kTile, 1024, kSwizzle128B), idY, kk > 0);
        // S_c^T = B^T (w x): A = B tile read MN-major (128 n rows), B = the weighted x rows
        const uint32_t sB = smem_addr(sm.B[c & 1]), sXw = smem_addr(sm.Xw[c & 1]);
#pragma unroll
        for (int kk = 0; kk < kQ / 16; ++kk)
            mma_bf16_ss(tmem + kWsS, smem_desc(sB + kk * 2048, kTile, 1024, kSwizzle128B),
                        smem_desc(sXw + kk * 2048, kTile, 1024, kSwizzle128B), idS, kk > 0);
        mma_commit(&sm.bar_m2[yp]);
    }
    return true;
}

// ---- the copying thread --------------------------------------------------------------
// Every TMA copy, each into a buffer whose previous contents have been used:
// the end of Y(c), S_c(c) means the end of G(c) too (issued before them),
// Zf(c) signals its own end, and the math warps are done with x(c) once
// they have weighed it (S_c(c) reads the weighted rows).
template <int NB, bool EXT>
__device__ __forceinline__ bool loader_role(Ctx<NB> &cx, const CUtensorMap *tmC, const CUtensorMap *tmB,
                                            const CUtensorMap *tmX) {
    auto &sm = cx.sm;
    const int nc = cx.nc, b = cx.b, h = cx.h, grp = cx.grp;
    uint32_t ph_m2 = 0, ph_z = 0;   // one bit per parity
    auto load_b = [&](int c, int buf) {
        mbar_arrive_expect_tx(&sm.bar_b[buf], NB * kTile);
#pragma unroll
        for (int r = 0; r < NB; ++r)
            tma_load_4d(sm.B[buf][r], tmB, &sm.bar_b[buf], r * 64, grp, c * kQ, b);
    };
    auto load_c = [&](int c, int buf) {
        mbar_arrive_expect_tx(&sm.bar_c[buf], NB * kTile);
#pragma unroll
        for (int r = 0; r < NB; ++r) tma_load_4d(sm.C[buf][r], tmC, &sm.bar_c[buf], r * 64, grp, c * kQ, b);
    };
    auto load_x = [&](int c) {
        const int xb = c % kXBufs;
        mbar_arrive_expect_tx(&sm.bar_x[xb], kTile);
        tma_load_4d(sm.X[xb], tmX, &sm.bar_x[xb], 0, h, c * kQ, b);
    };
    load_c(0, 0);
    load_b(0, 0);
    load_x(0);
    if (nc > 1) {
        load_c(1, 1);
        load_b(1, 1);
        load_x(1);
    }
    for (int c = 0; c < nc; ++c) {
        WS_WAIT_I(sm.bar_m2[c & 1], ph_m2, c & 1);   // G(c), Y(c), S_c(c) done
        if (c + 2 < nc) {
            load_x(c + 2);
            load_b(c + 2, c & 1);
        }
        WS_WAIT_I(sm.bar_z[c & 1], ph_z, c & 1);     // Zf(c) done: C(c) read
        if (c + 2 < nc) load_c(c + 2, c & 1);
    }
    return true;
}

// ---- the vector warp ------------------------------------------------------------------
// The per-tile vectors, up to two tiles ahead of the math warps: cumulative
// sums of dt A (log2 units) inside the tile, dt, the column factors of the
// off-diagonal mask blocks and the tile total.  Lane l holds rows 4 l ..
// 4 l + 3.  Slot c % 3 held tile c - 3, which the math warps last read right
// after m2(c - 3) and before their mask store of tile c - 2: the vectors of
// tile c are written once that store is complete everywhere.  The mask
// stores alternate between two barriers, so that this wait cannot alias: the
// barrier of tile c - 2 completes next with the store of tile c, which needs
// the vectors this warp is about to write.  (With one barrier a parity wait
// could: were this warp held up, by a slow dt load say, the stores of tiles
// c - 2 and c - 1 could both complete first, and the wait would then stand
// for the store of tile c.)
template <int NB, bool EXT>
__device__ __forceinline__ bool vector_role(Ctx<NB> &cx) {
    auto &sm = cx.sm;
    const int lane = threadIdx.x & 31;
    const int nc = cx.nc, L = cx.L, H = cx.prm.H;
    const __nv_bfloat16 *dtp = cx.prm.dt + (int64_t(cx.b) * L) * H + cx.h;
    uint32_t ph_mfull = 0;   // one bit per mask barrier
    float raw[4], nxt[4];
    auto load = [&](int c, float (&r)[4]) {    // raw dt of rows c kQ + 4 lane + k; past L: 0
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int row = c * kQ + 4 * lane + k;
            r[k] = row < L ? __bfloat162float(dtp[int64_t(row) * H]) : 0.0f;
        }
    };
    load(0, raw);
    for (int c = 0; c < nc; ++c) {
        if (c + 1 < nc) load(c + 1, nxt);
        if (c >= 2) WS_WAIT_I(sm.bar_mfull[c & 1], ph_mfull, c & 1);   // mask of tile c - 2 stored
        const int p = c % kSlots;
        float dv[4], cs[4], run = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float d = 0.0f;
            if (c * kQ + 4 * lane + k < L) {    // rows past L: no decay, no input
                d = raw[k];
                if (EXT) {
                    d += cx.dbias;
                    if (cx.prm.dt_softplus) d = softplus_fast(d);
                    if (cx.prm.dt_limit) d = fminf(fmaxf(d, cx.prm.dt_min), cx.prm.dt_max);
                }
            }
            dv[k] = d;
            run += d * cx.Ah;
            cs[k] = run;
        }
        float incl = run;      // inclusive scan of the lane totals
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        const float excl = incl - run;
#pragma unroll
        for (int k = 0; k < 4; ++k) cs[k] += excl;
        // column factor of row s: exp2(cum at the end of s's 32-row block - cum_s) dt_s
        const float end = __shfl_sync(0xffffffffu, cs[3], lane | 7);
        const float tot = __shfl_sync(0xffffffffu, cs[3], 31);
        reinterpret_cast<float4 *>(sm.cum[p])[lane] = make_float4(cs[0], cs[1], cs[2], cs[3]);
        reinterpret_cast<float4 *>(sm.dtv[p])[lane] = make_float4(dv[0], dv[1], dv[2], dv[3]);
        reinterpret_cast<float4 *>(sm.csf[p])[lane] =
            make_float4(ex2(end - cs[0]) * dv[0], ex2(end - cs[1]) * dv[1], ex2(end - cs[2]) * dv[2],
                        ex2(end - cs[3]) * dv[3]);
        if (lane == 0) sm.tot[p] = tot;
        mbar_arrive(&sm.bar_vec[p]);
#pragma unroll
        for (int k = 0; k < 4; ++k) raw[k] = nxt[k];
    }
    return true;
}

// ---- the eight math warps -------------------------------------------------------------
// Weighted x rows: half hf (32 p) of row s of the x tile scaled by w into the
// Xw tile (same swizzle, so 16-byte chunks map in place).
__device__ __forceinline__ void weigh_half(const uint8_t *X, uint8_t *Xw, int s, float w, int hf) {
    const uint4 *src = reinterpret_cast<const uint4 *>(X + s * 128);
    uint4 *dst = reinterpret_cast<uint4 *>(Xw + s * 128);
    const float2 ww = make_float2(w, w);
    uint4 v[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) v[jj] = src[(4 * hf + jj) ^ (s & 7)];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const float2 a = fmul2(unpack_bf16(v[jj].x), ww), b = fmul2(unpack_bf16(v[jj].y), ww);
        const float2 c = fmul2(unpack_bf16(v[jj].z), ww), d = fmul2(unpack_bf16(v[jj].w), ww);
        dst[(4 * hf + jj) ^ (s & 7)] =
            make_uint4(pack_bf16(a.x, a.y), pack_bf16(b.x, b.y), pack_bf16(c.x, c.y), pack_bf16(d.x, d.y));
    }
}

// a * x + y for packed fp32 pairs.
__device__ __forceinline__ float2 ffma2(float2 a, float2 x, float2 y) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)),
          "l"(*reinterpret_cast<unsigned long long *>(&x)),
          "l"(*reinterpret_cast<unsigned long long *>(&y)));
    return *reinterpret_cast<float2 *>(&r);
}

template <int NB, bool EXT, bool GATE>
__device__ __forceinline__ bool math_role(Ctx<NB> &cx, bool has_h0) {
    constexpr int N = NB * 64;
    auto &sm = cx.sm;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;             // TMEM lane quarter
    const int hf = warp >> 2;           // column half
    const int t = q * 32 + lane;        // tile row t, state row n, TMEM lane
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    const int nc = cx.nc, L = cx.L, b = cx.b, h = cx.h, H = cx.prm.H;
    const uint32_t tmem = cx.tmem;
    const bool is_state = q * 32 < N;   // state rows n = t exist (warp-uniform)
    // mask blocks of row quarter q: half 0 forms the diagonal block sb = q,
    // half 1 the blocks sb = 0 .. q - 1 below it
    uint32_t ph_g = 0, ph_m2 = 0, ph_z = 0, ph_x = 0, ph_vec = 0;   // ph_m2, ph_z, ph_x, ph_vec: bits

    // Weighted x rows of tile c: row s = t, columns of half hf.  The buffer
    // held the output staging of tile c - 2, whose rows 32 q .. 32 q + 31
    // both warps of this lane quarter used: each waits until its own stores
    // have read it, then for the other warp.
    uint32_t ph_pair = 0;
    auto weigh = [&](int c) -> bool {
        const int p = c % kSlots, xb = c % kXBufs;
        const float w = ex2(sm.tot[p] - sm.cum[p][t]) * sm.dtv[p][t];
        if (c >= 2) {
            if (lane == 0) {
                bulk_wait_read0();
                mbar_arrive(&sm.bar_pair[q]);
            }
            WS_WAIT(sm.bar_pair[q], ph_pair);
        }
        WS_WAIT_I(sm.bar_x[xb], ph_x, xb);
        weigh_half(sm.X[xb], sm.Xw[c & 1], t, w, hf);
        fence_proxy_async_smem();
        mbar_arrive(&sm.bar_xw[c & 1]);
        return true;
    };
    // Mask rows t of tile c, this warp's blocks, into registers (bf16 pairs);
    // the weighted rows of tile c are written while the G rows load.
    uint32_t mk[3][16];
    auto weigh_and_mask = [&](int c) -> bool {
        const int p = c % kSlots;
        WS_WAIT_I(sm.bar_vec[p], ph_vec, p);
        WS_WAIT(sm.bar_g, ph_g);
        tc_fence_after_sync();
        const float *cum = sm.cum[p];
        const float *dtv = sm.dtv[p];
        const float *csf = sm.csf[p];
        const float cum_t = cum[t];
        // The first G block of this warp (half 0: the diagonal block; half 1:
        // block 0, when the quarter has blocks below the diagonal) loads
        // while the x rows are weighed: one weighing call site for both halves.
        uint32_t ga[32];
        const bool ld0 = hf == 0 || q >= 1;
        if (ld0) tmem_ld32_async(tmem + lane_base + kWsG + (hf == 0 ? q * 32 : 0), ga);
        if (!weigh(c)) return false;
        if (ld0) tmem_wait_tie(ga);
        if (hf == 0) {
            tc_fence_before_sync();
            mbar_arrive(&sm.bar_gfree);     // G may be overwritten now
            // diagonal block: direct differences of cumulative sums; the
            // skip term rides on the diagonal: Y = (M + D_h I) X
            const float4 *c4 = reinterpret_cast<const float4 *>(cum + q * 32);
            const float4 *d4 = reinterpret_cast<const float4 *>(dtv + q * 32);
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
                const float4 cs = c4[j4], ds = d4[j4];
                const float csv[4] = {cs.x, cs.y, cs.z, cs.w};
                const float dsv[4] = {ds.x, ds.y, ds.z, ds.w};
                float m[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j = 4 * j4 + k;
                    const float w = (j <= lane) ? ex2(cum_t - csv[k]) : 0.0f;
                    float v = __uint_as_float(ga[j]) * (w * dsv[k]);
                    if (j == lane) v += cx.Dh;
                    m[k] = v;
                }
                mk[0][2 * j4] = pack_bf16(m[0], m[1]);
                mk[0][2 * j4 + 1] = pack_bf16(m[2], m[3]);
            }
        } else {
            // blocks below the diagonal: G * (row factor) * (column factor),
            // both <= 1; the G rows of block i + 1 load while block i is formed
            auto offdiag = [&](int i, const uint32_t (&g)[32]) {
                const float e = ex2(cum_t - cum[i * 32 + 31]);
                const float2 ee = make_float2(e, e);
                const float4 *f4 = reinterpret_cast<const float4 *>(csf + i * 32);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 f = f4[j4];
                    const float2 a = fmul2(fmul2(make_float2(__uint_as_float(g[4 * j4]), __uint_as_float(g[4 * j4 + 1])),
                                                 make_float2(f.x, f.y)), ee);
                    const float2 bq = fmul2(fmul2(make_float2(__uint_as_float(g[4 * j4 + 2]), __uint_as_float(g[4 * j4 + 3])),
                                                  make_float2(f.z, f.w)), ee);
                    mk[i][2 * j4] = pack_bf16(a.x, a.y);
                    mk[i][2 * j4 + 1] = pack_bf16(bq.x, bq.y);
                }
            };
            uint32_t gb[32];
            if (q >= 2) tmem_ld32_async(tmem + lane_base + kWsG + 32, gb);
            if (q < 2) {
                tc_fence_before_sync();
                mbar_arrive(&sm.bar_gfree);
            }
            if (q >= 1) offdiag(0, ga);
            if (q >= 2) {
                tmem_wait_tie(gb);
                if (q >= 3) tmem_ld32_async(tmem + lane_base + kWsG + 64, ga);
                if (q < 3) {
                    tc_fence_before_sync();
                    mbar_arrive(&sm.bar_gfree);
                }
                offdiag(1, gb);
            }
            if (q >= 3) {
                tmem_wait_tie(ga);
                tc_fence_before_sync();
                mbar_arrive(&sm.bar_gfree);
                offdiag(2, ga);
            }
        }
        return true;
    };
    // Store this warp's mask blocks into tensor memory (after Y of the
    // previous tile has read the mask) and hand the mask to the issuer.
    auto mask_store = [&](int c) {
        if (hf == 0) {
            tmem_st_32x32b_x16(tmem + lane_base + kWsM + q * 16, mk[0]);
        } else {
            if (q >= 1) tmem_st_32x32b_x16(tmem + lane_base + kWsM, mk[0]);
            if (q >= 2) tmem_st_32x32b_x16(tmem + lane_base + kWsM + 16, mk[1]);
            if (q >= 3) tmem_st_32x32b_x16(tmem + lane_base + kWsM + 32, mk[2]);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(&sm.bar_mfull[c & 1]);
    };
    const bool gate = GATE && cx.prm.z != nullptr;
    // gate row of tile c (bf16, 32 values = 64 bytes): prefetched into L1 in
    // iteration c after the mask of tile c + 1 is formed, and read in the
    // epilogue of tile c, so that no registers hold it through the state update
    auto gate_row = [&](int c) {
        return reinterpret_cast<const uint4 *>(cx.prm.z + ((size_t(b) * L + c * kQ + t) * H + h) * kP + hf * 32);
    };
    auto load_gate = [&](int c) {
        if (!gate || c * kQ + t >= L) return;
        asm volatile("prefetch.global.L1 [%0];" ::"l"(gate_row(c)));
    };
    // Output rows t of tile c, columns of half hf, from the loaded
    // accumulators: y = Y + e^{cum_t} Zf (Y already holds D x), out through
    // this warp's part of tile c's weighted-rows buffer (rows 32 q .. 32 q +
    // 31, the 16-byte chunks 4 hf .. 4 hf + 3 of each, swizzled as the tile:
    // 32 rows x 16 columns at a time), so that each store instruction writes
    // 8 rows x 64 contiguous bytes.
    auto epilogue = [&](int c, const uint32_t (&yv)[32], const uint32_t (&zf)[32], bool has_s,
                        float ef) -> bool {
        float out[32];
        if (has_s) {
            const float2 e2 = make_float2(ef, ef);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float2 r = ffma2(e2, make_float2(__uint_as_float(zf[2 * j]), __uint_as_float(zf[2 * j + 1])),
                                       make_float2(__uint_as_float(yv[2 * j]), __uint_as_float(yv[2 * j + 1])));
                out[2 * j] = r.x;
                out[2 * j + 1] = r.y;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) out[j] = __uint_as_float(yv[j]);
        }
        if (gate && c * kQ + t < L) {   // (rows past L are computed but not stored)
            const uint4 *zp = gate_row(c);
            uint4 zq[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) zq[j] = __ldg(zp + j);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t w4[4] = {zq[j].x, zq[j].y, zq[j].z, zq[j].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 zz = unpack_bf16(w4[k]);
                    out[8 * j + 2 * k] *= silu_tanh(zz.x);
                    out[8 * j + 2 * k + 1] *= silu_tanh(zz.y);
                }
            }
        }
        // Out by TMA stores: rows 32 q .. 32 q + 31 of tile c's weighted-rows
        // buffer (read by S_c(c), which has finished) hold two 2 KB boxes,
        // one per warp of the lane quarter: 32 rows x 16 columns (64-byte
        // rows, 64-byte swizzle: 16-byte chunk j of row r at j ^ (r / 2 % 4)),
        // written twice (columns 0..15, then 16..31 of the warp's half).
        // Rows past L are not written by the store.
        uint8_t *box = sm.Xw[c & 1] + q * 4096 + hf * 2048;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            if (hh == 1) {
                if (lane == 0) bulk_wait_read0();   // the first store has read the box
                __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<float4 *>(box + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                    make_float4(out[16 * hh + 4 * j], out[16 * hh + 4 * j + 1], out[16 * hh + 4 * j + 2],
                                out[16 * hh + 4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_4d(cx.tmY, box, hf * 32 + hh * 16, h, c * kQ + q * 32, b);
                bulk_commit();
            }
        }
        return true;
    };

    // ---- prologue -------------------------------------------------------------------
    if (hf == 0) {   // the mask blocks above the diagonal stay zero for every tile
        uint32_t zero[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) zero[j] = 0u;
        for (int sb = q + 1; sb < 4; ++sb) tmem_st_32x32b_x16(tmem + lane_base + kWsM + sb * 16, zero);
        tmem_wait_st();
    }
    float st[32];   // state rows n = t, columns p of half hf (fp32)
#pragma unroll
    for (int j = 0; j < 32; ++j) st[j] = 0.0f;
    if (has_h0 && is_state) {
        const float *src = cx.prm.h0 + size_t(cx.bh) * kP * N + size_t(hf * 32) * N + t;
#pragma unroll
        for (int j = 0; j < 32; ++j) st[j] = src[size_t(j) * N];
        put_state_half(&sm.S[0][0], t, hf, st);
    }
    fence_proxy_async_smem();
    mbar_arrive(&sm.bar_st);
    if (!weigh_and_mask(0)) return false;
    mask_store(0);

    for (int c = 0; c < nc; ++c) {
        const bool more = c + 1 < nc;
        if (more && !weigh_and_mask(c + 1)) return false;
        load_gate(c);
        WS_WAIT_I(sm.bar_m2[c & 1], ph_m2, c & 1);   // every product of tile c done
        tc_fence_after_sync();
        const int p = c % kSlots;
        const float e = ex2(sm.tot[p]), ef = ex2(sm.cum[p][t]);
        const bool has_s = c > 0 || has_h0;
        // the chunk state and Y of tile c in one round trip
        // (with N = 64 the lanes of quarters 2, 3 hold S_c rows 64..127, which
        // are exact zeros -- the B operand's upper rows are zero: their state
        // stays zero, and loading it keeps the code the same for every warp)
        uint32_t sv[32], yv[32], zf[32];
        tmem_ld32_async(tmem + lane_base + kWsS + hf * 32, sv);
        tmem_ld32_async(tmem + lane_base + ((c & 1) ? kWsY1 : kWsY0) + hf * 32, yv);
        tmem_wait_tie(yv);
        reg_tie(sv);
        // S_c(c) is in registers: Y(c + 1) and S_c(c + 1) may start
        if (more) mask_store(c + 1);
        WS_WAIT_I(sm.bar_z[c & 1], ph_z, c & 1);    // Zf(c) done: the state image is free
        tc_fence_after_sync();
        // state passing: rows n = t of S_in, columns of half hf
#pragma unroll
        for (int j = 0; j < 32; ++j) st[j] = fmaf(e, st[j], __uint_as_float(sv[j]));
        if (is_state && more) put_state_half(&sm.S[0][0], t, hf, st);
        if (more) {
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&sm.bar_st);            // Zf(c + 1) can start
        }
        if (has_s) {
            tmem_ld32_async(tmem + lane_base + ((c & 1) ? kWsZ1 : kWsZ0) + hf * 32, zf);
            tmem_wait_tie(zf);
        }
        if (!epilogue(c, yv, zf, has_s, ef)) return false;
    }
    if (EXT && cx.prm.h_final != nullptr && is_state) {
        float *dst = cx.prm.h_final + size_t(cx.bh) * kP * N + size_t(hf * 32) * N + t;
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[size_t(j) * N] = st[j];
    }
    return true;
}

// GATE (only with EXT): the silu gate z is compiled in (its rows, loaded a
// tile ahead, take registers the other options do not need).
template <int NB, bool EXT, bool GATE>
__global__ void __launch_bounds__(kThreads, 1)
ssd_ws_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
              const __grid_constant__ Params prm) {
    extern __shared__ uint8_t smem_raw[];
    Smem<NB> &sm = *reinterpret_cast<Smem<NB> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int bh = blockIdx.x;

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.bar_c[i], 1);
            mbar_init(&sm.bar_b[i], 1);
        }
        for (int i = 0; i < kXBufs; ++i) mbar_init(&sm.bar_x[i], 1);
        mbar_init(&sm.bar_g, 1);
        mbar_init(&sm.bar_m2[0], 1);
        mbar_init(&sm.bar_m2[1], 1);
        mbar_init(&sm.bar_fin[0], 1);
        mbar_init(&sm.bar_fin[1], 1);
        mbar_init(&sm.bar_gfree, kMath);
        for (int i = 0; i < 2; ++i) mbar_init(&sm.bar_mfull[i], kMath);
        mbar_init(&sm.bar_xw[0], kMath);
        mbar_init(&sm.bar_xw[1], kMath);
        mbar_init(&sm.bar_st, kMath);
        mbar_init(&sm.bar_z[0], 1);
        mbar_init(&sm.bar_z[1], 1);
        for (int i = 0; i < kSlots; ++i) mbar_init(&sm.bar_vec[i], 32);
        for (int i = 0; i < 4; ++i) mbar_init(&sm.bar_pair[i], 2);
        mbar_fence_init();
        prefetch_tmap(&tmC);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmY);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (NB == 1) {   // the n = 64..127 rows that S_c's A operand spans read as zeros
        for (int i = tid; i < int(kTile / 16); i += kThreads) {
            reinterpret_cast<uint4 *>(sm.B[0][1])[i] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4 *>(sm.B[1][1])[i] = make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    Ctx<NB> cx{sm, prm, bh / prm.H, bh % prm.H, 0, bh, prm.L, prm.nc, 0.0f, 0.0f, 0.0f,
               sm.tmem_base, &abort_flag, &tmY};
    cx.grp = cx.h / (prm.H / prm.G);
    cx.Ah = prm.A[cx.h] * SSM_LOG2E;
    cx.Dh = prm.D ? prm.D[cx.h] : 0.0f;
    cx.dbias = (EXT && prm.dt_bias) ? prm.dt_bias[cx.h] : 0.0f;
    const bool has_h0 = EXT && prm.h0 != nullptr;

    bool ok = true;
    if (warp < 8) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kMathRegs));
        ok = math_role<NB, EXT, GATE>(cx, has_h0);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
        if (tid == 256) ok = issuer_role<NB, EXT>(cx, has_h0);
        if (tid == 288) ok = loader_role<NB, EXT>(cx, &tmC, &tmB, &tmX);
        if (warp == 10) ok = vector_role<NB, EXT>(cx);
        if (tid == 352) ok = issuer_ys_role<NB, EXT>(cx);
    }
    if (warp < 8 && (tid & 31) == 0) bulk_wait0();   // the output stores are complete
    if (!ok) {
        abort_flag = 1;
        atomicOr(&g_device_error, 1u);
    }
    if (!ok && (tid == 256 || tid == 352)) {
        // products still in flight after a timeout: give each issuing
        // thread's a bounded chance to finish before the tensor memory is released
        uint64_t *fin = &sm.bar_fin[tid == 352];
        mma_commit(fin);
        volatile int never = 0;
        (void)mbar_wait_bounded(fin, 0, &never, 100000000ull);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(sm.tmem_base, kTmemCols);
    }
}
#undef WS_WAIT
#undef WS_WAIT_I

}  // namespace ws


// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// The driver's tensor-map encoder.  Only a successful lookup is kept: after
// a failed one the next call asks the driver again.
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_acquire);
    if (fn != nullptr) return fn;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cached.store(fn, std::memory_order_release);
    }
    return fn;
}

static bool make_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
                     const cuuint64_t *strides_bytes, const cuuint32_t *box,
                     CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, dtype, cuuint32_t(rank), const_cast<void *>(base),
                    dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int NB>
static cudaError_t launch_nb(const __nv_bfloat16 *x, const __nv_bfloat16 *dt, const float *A,
                             const __nv_bfloat16 *Bm, const __nv_bfloat16 *Cm, const float *D,
                             float *y, int64_t Bs, int64_t L, int64_t H, bool bidir,
                             cudaStream_t stream, uint8_t *fixed_scratch = nullptr,
                             const Options *opt = nullptr) {
    constexpr int N = NB * 64;
    CUtensorMap tmC, tmB, tmX, tmY;
    const int64_t G = (opt && opt->ngroups > 1) ? opt->ngroups : 1;
    // B, C: (Bs, L, G, N); one box is 64 n x 128 rows of one group
    const cuuint64_t dbc[4] = {cuuint64_t(N), cuuint64_t(G), cuuint64_t(L), cuuint64_t(Bs)};
    const cuuint64_t sbc[3] = {cuuint64_t(N) * 2, cuuint64_t(G) * N * 2, cuuint64_t(L) * G * N * 2};
    const cuuint32_t boxbc[4] = {64, 1, kQ, 1};
    const cuuint64_t dx[4] = {cuuint64_t(kP), cuuint64_t(H), cuuint64_t(L), cuuint64_t(Bs)};
    const cuuint64_t sx[3] = {cuuint64_t(kP) * 2, cuuint64_t(H) * kP * 2, cuuint64_t(L) * H * kP * 2};
    const cuuint32_t boxx[4] = {64, 1, kQ, 1};
    const cuuint64_t sy[3] = {cuuint64_t(kP) * 4, cuuint64_t(H) * kP * 4, cuuint64_t(L) * H * kP * 4};
    const cuuint32_t boxy[4] = {32, 1, kQ, 1};
    if (!make_map(&tmC, Cm, 4, dbc, sbc, boxbc) || !make_map(&tmB, Bm, 4, dbc, sbc, boxbc) ||
        !make_map(&tmX, x, 4, dx, sx, boxx) ||
        !make_map(&tmY, y, 4, dx, sy, boxy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
        return cudaErrorInvalidValue;

    Params prm;
    prm.dt = dt;
    prm.A = A;
    prm.D = D;
    prm.y = y;
    prm.rstate = nullptr;
    prm.L = int(L);
    prm.H = int(H);
    prm.nc = int((L + kQ - 1) / kQ);
    const Options none{};
    const Options &o = opt ? *opt : none;
    prm.dt_bias = o.dt_bias;
    prm.z = static_cast<const __nv_bfloat16 *>(o.z);
    prm.h0 = o.h0;
    prm.h_final = o.h_final;
    prm.dt_min = o.dt_min;
    prm.dt_max = o.dt_max;
    prm.dt_softplus = o.dt_softplus;
    prm.dt_limit = o.dt_limit;
    prm.G = int(G);
    const int64_t grid = Bs * H;
    if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;

    // The warp-specialised kernel takes the unidirectional scan.
    const bool use_ws = !bidir;
    size_t smem = sizeof(Smem<NB>) + 1024;
    static_assert(sizeof(Smem<NB>) + 1024 <= 227 * 1024, "shared memory of one CTA exceeds 227 KB");
    static_assert(sizeof(ws::Smem<NB>) + 1024 <= 227 * 1024, "shared memory of one CTA exceeds 227 KB");
    // the plain kernels unless an option is on (groups alone need none)
    const bool ext = opt && (opt->dt_bias || opt->dt_softplus || opt->dt_limit || opt->z ||
                             opt->h0 || opt->h_final);
    auto kern = ext ? ssd_chunk_scan_kernel<NB, true> : ssd_chunk_scan_kernel<NB, false>;
    using WsKern = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                            const Params);
    WsKern wkern = nullptr;
    if (use_ws) {
        wkern = !ext ? ws::ssd_ws_kernel<NB, false, false>
                     : (opt->z ? ws::ssd_ws_kernel<NB, true, true> : ws::ssd_ws_kernel<NB, true, false>);
        smem = sizeof(ws::Smem<NB>) + 1024;
    }
    cudaError_t err;
    // the warp-specialised kernel stores y in boxes of 16 p x 32 rows
    CUtensorMap tmYw;
    const cuuint32_t boxyw[4] = {16, 1, 32, 1};
    if (wkern && !make_map(&tmYw, y, 4, dx, sy, boxyw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                           CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    if (wkern) {
        err = cudaFuncSetAttribute(wkern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (err != cudaSuccess) return err;
        // setmaxnreg re-divides the registers the CTA was launched with; had
        // it been launched with fewer, the larger share could never be granted.
        cudaFuncAttributes fa;
        err = cudaFuncGetAttributes(&fa, wkern);
        if (err != cudaSuccess) return err;
        if (fa.numRegs < int(ws::kLaunchRegs)) return cudaErrorNotSupported;
    } else {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (err != cudaSuccess) return err;
    }

    void *scratch = nullptr;
    if (bidir && prm.nc > 1 && fixed_scratch != nullptr) {
        prm.rstate = fixed_scratch;   // caller-provided region, sized by the caller
    } else if (bidir && prm.nc > 1) {
        const size_t bytes = size_t(grid) * prm.nc * NB * kStateRegion;
        err = cudaMallocAsync(&scratch, bytes, stream);
        if (err != cudaSuccess) return err;
        prm.rstate = static_cast<uint8_t *>(scratch);
    }
    if (wkern)
        wkern<<<dim3(unsigned(grid)), dim3(ws::kThreads), smem, stream>>>(tmC, tmB, tmX, tmYw, prm);
    else
        kern<<<dim3(unsigned(grid)), dim3(kThreads), smem, stream>>>(tmC, tmB, tmX, tmY, prm);
    err = cudaGetLastError();
    if (scratch) {
        cudaError_t e2 = cudaFreeAsync(scratch, stream);
        if (err == cudaSuccess) err = e2;
    }
    return err;
}

cudaError_t launch(const __nv_bfloat16 *x, const __nv_bfloat16 *dt, const float *A_head,
                   const __nv_bfloat16 *Bm, const __nv_bfloat16 *Cm, const float *D, float *y,
                   int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N, int64_t chunk,
                   bool bidirectional, int num_sms, cudaStream_t stream, const Options *opt) {
    (void)chunk;
    if (P != kP) return cudaErrorNotSupported;
    // short bidirectional sequences: independent per-tile passes (ssd_bidir.cu)
    if (bidirectional && bidir::supported(L, P, N))
        return bidir::launch(x, dt, A_head, Bm, Cm, D, y, Bs, L, H, num_sms, opt, stream);
    if (N == 64)
        return launch_nb<1>(x, dt, A_head, Bm, Cm, D, y, Bs, L, H, bidirectional, stream, nullptr, opt);
    if (N == 128)
        return launch_nb<2>(x, dt, A_head, Bm, Cm, D, y, Bs, L, H, bidirectional, stream, nullptr, opt);
    return cudaErrorNotSupported;
}

// ---------------------------------------------------------------------------
// Variant that allocates nothing
// ---------------------------------------------------------------------------
// Callers that may not allocate device memory (for instance code running
// under an allocator that forbids it, or inside a region that must not touch
// the memory pool) get the reverse scan's entering states in this fixed
// module-scope array instead of a cudaMallocAsync buffer.  Every GPU that
// loads the library holds it until the process exits.  All calls share it:
// two such calls that overlap on the GPU race.  No part of it needs to start
// at zero -- every slot a call reads was written earlier by the same call.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDev = 64;
std::mutex g_na_mutex;
void *g_na_addr[kMaxDev];   // written once per device, only after a successful lookup
}  // namespace

// Bytes of the reverse states a bidirectional call keeps; SIZE_MAX when the
// product does not fit (the caller then rejects the size).
size_t noalloc_scratch_needed(int64_t Bs, int64_t L, int64_t H, int64_t N, bool bidirectional) {
    const int64_t nc = (L + kQ - 1) / kQ;
    if (!bidirectional || nc <= 1) return 0;
    const uint64_t f[5] = {uint64_t(Bs), uint64_t(H), uint64_t(nc), uint64_t(N / 64),
                           uint64_t(kStateRegion)};
    uint64_t bytes = 1;
    for (uint64_t v : f) {
        if (v != 0 && bytes > UINT64_MAX / v) return SIZE_MAX;
        bytes *= v;
    }
    return bytes > uint64_t(SIZE_MAX) ? SIZE_MAX : size_t(bytes);
}

// Device address of the array, looked up with the device current, since the
// host-side symbol is not a device address.  Only a successful lookup is
// kept: a call whose lookup failed (for example while an earlier
// asynchronous error was pending) returns that error, and the next call
// tries again.
static cudaError_t noalloc_scratch_address(uint8_t **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_na_mutex);
    if (g_na_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_na_addr[dev] = p;
    }
    *out = static_cast<uint8_t *>(g_na_addr[dev]);
    return cudaSuccess;
}

cudaError_t launch_noalloc(const __nv_bfloat16 *x, const __nv_bfloat16 *dt, const float *A_head,
                           const __nv_bfloat16 *Bm, const __nv_bfloat16 *Cm, const float *D,
                           float *y, int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                           bool bidirectional, cudaStream_t stream) {
    if (P != kP || (N != 64 && N != 128)) return cudaErrorNotSupported;
    if (noalloc_scratch_needed(Bs, L, H, N, bidirectional) > kNoAllocScratchBytes)
        return cudaErrorNotSupported;
    uint8_t *scratch = nullptr;
    cudaError_t e = noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    if (N == 64)
        return launch_nb<1>(x, dt, A_head, Bm, Cm, D, y, Bs, L, H, bidirectional, stream, scratch);
    return launch_nb<2>(x, dt, A_head, Bm, Cm, D, y, Bs, L, H, bidirectional, stream, scratch);
}

// Self-test of the timeout path: one thread waits on an mbarrier that
// nothing ever arrives on, with the kernels' bounded wait and a short limit,
// and reports through the same error word when the wait runs out.
__global__ void wait_timeout_probe_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    mbar_init(&bar, 1);
    mbar_fence_init();
    volatile int never = 0;
    if (!mbar_wait_bounded(&bar, 0, &never, limit_ns)) atomicOr(&g_device_error, 1u);
}

cudaError_t probe_wait_timeout(cudaStream_t st) {
    wait_timeout_probe_kernel<<<1, 1, 0, st>>>(20000000ull);   // 20 ms
    return cudaGetLastError();
}

// Read and clear the device error word (host side, synchronous).
cudaError_t take_device_error(unsigned int *out) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    *out = v;
    return e;
}

}  // namespace ssd
}  // namespace ssm
