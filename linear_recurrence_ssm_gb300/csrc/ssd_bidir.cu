// ssd_bidir.cu -- the bidirectional chunked scalar-decay scan for short
// sequences (N = 64 states, at most four 128-row tiles), as independent
// per-tile work on 5th-generation tensor cores (sm_103a).
//
// The bidirectional scan of "Some questions of Bi-Mamba2 and Hydra"
// (Bi-Mamba2 issue 1) is the sum of a forward and a backward SSM with shared
// x, dt, A, B, C, plus the skip term D x counted once:
//     y = F(x) + flip(F(flip(x))) + D x,   F: H_t = e^{dt_t A} H_{t-1} + dt_t x_t (outer) B_t,  y_t = H_t C_t.
// In chunked form (tile of Q = 128 rows, cum = inclusive prefix sum of
// dA = dt A inside the tile, excl = cum - dA, tot = cum at the tile's end,
// all in log2 units) every tile's output needs only the states entering it
// from the left (forward) and from the right (reverse):
//     y[t] = (M X)[t] + e^{cum_t} (C S_in^T)[t] + e^{tot - excl_t} (C R_in^T)[t],
//     M[t,s] = (C B^T)[t,s] dt_s (e^{cum_t - cum_s} [s <= t] + e^{excl_s - excl_t} [s >= t]) + D [s = t],
// and those states are decayed sums of the other tiles' chunk states
//     Sf(j) = B_j^T (w_f x_j), w_f = dt e^{tot - cum},   Sr(j) = B_j^T (w_r x_j), w_r = dt e^{excl},
//     S_in(i) = sum_{j < i} e^{tot_{j+1} + .. + tot_{i-1}} Sf(j),   R_in(i) = sum_{j > i} e^{tot_{i+1} + .. + tot_{j-1}} Sr(j).
// So the work splits into two passes over independent tiles instead of a
// serial walk per (batch, head):
//   pass 1 (bidir_state_kernel, persistent): every tile's Sf, Sr (one
//     tensor-core product, B^T [w_f x | w_r x], rounded to bf16 -- the
//     operand precision of the product they feed) and its total decay, to
//     scratch;
//   pass 2 (bidir_out_kernel, persistent): per tile, the entering states
//     combined in fp32 from the other tiles' chunk states, G = C B^T, the
//     two-sided mask, Y = M X and Z = C [S_in | R_in]^T on the tensor core,
//     and y.
// No reversed copy of any input is made; both directions read each tile in
// place.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "ssm_common.cuh"
#include "tc_ptx.cuh"

namespace ssm {
namespace bidir {

using namespace ssm::tc;

constexpr int kQ = 128;              // tile rows (MMA M)
constexpr int kP = 64;               // head dimension
constexpr int kN = 64;               // state size served here
constexpr int kMaxTiles = 4;         // tiles per sequence served here
constexpr uint32_t kTile = kQ * 128; // bytes of a 128-row x 128-byte tile
constexpr uint32_t kImg = kN * 128;  // bytes of a bf16 state image (rows n, 64 p)
constexpr uint32_t kState = kN * kP * 2;   // bytes of one chunk state (bf16)
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ unsigned int g_device_error;   // non-zero once a bounded wait ran out

struct Params {
    const __nv_bfloat16 *dt;
    const float *A;
    const float *D;
    float *y;
    uint8_t *chunk;    // [Bs*H][2][nc][N][P] bf16: Sf (direction 0), Sr (direction 1), rows n
                       // of 128 bytes, the 16-byte chunks of row n at chunk ^ (n % 8)
    float *tot;        // [Bs*H][kMaxTiles] decay total of each tile (log2 units)
    const float *dt_bias;
    const __nv_bfloat16 *z;
    float dt_min, dt_max;
    int dt_softplus, dt_limit;
    int L, H, nc, G, units;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t w) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&w);
    return __bfloat1622float2(v);
}
// a * b for two packed fp32 pairs.
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)),
          "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&r);
}
// dt of a row after the optional bias, softplus and clamp.
template <bool EXT>
__device__ __forceinline__ float prep_dt(float d, const Params &prm, float bias) {
    if (EXT) {
        d += bias;
        if (prm.dt_softplus) d = softplus_fast(d);
        if (prm.dt_limit) d = fminf(fmaxf(d, prm.dt_min), prm.dt_max);
    }
    return d;
}
// Programmatic dependent launch: this grid lets the next one start its
// prologue; the next one waits for this one's results before reading them.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ===========================================================================
// Pass 1: chunk states of every tile (one tile per CTA)
// ===========================================================================
struct __align__(1024) StateSmem {
    uint8_t Bt[kTile];         // B tile (rows s, 64 n)
    uint8_t X[kTile];          // x tile; weighted forward in place; then Sf staging
    uint8_t XR[kTile];         // x weighted reverse; then Sr staging
    float wsum[4];
    uint64_t bar_ld, bar_mma;
    uint32_t tmem_base;
};

// One CTA of 128 threads per tile (thread t owns tile row t and TMEM lane t),
// four per SM (about 50 KB of shared memory, 128 TMEM columns each), so that
// the copies of every tile of a wave are in flight at once.  D (128 x 128) =
// B^T [w_f x | w_r x] with A = the B tile read MN-major (rows n 0..63; rows
// 64..127 of A read the x tile -- they only feed rows of D that are never
// read), B = the two weighted x tiles (N = 128: p of the forward, then of the
// reverse direction); rows n < 64 of D go to scratch through bulk copies.
template <bool EXT>
__global__ void __launch_bounds__(128, 4)
bidir_state_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ Params prm) {
    extern __shared__ uint8_t smem_raw[];
    StateSmem &sm = *reinterpret_cast<StateSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int nc = prm.nc, L = prm.L, H = prm.H;
    const int bh = int(blockIdx.x) / nc, c = int(blockIdx.x) % nc;
    const int b = bh / H, h = bh % H;
    volatile int never = 0;
    // The output pass may be launched as soon as every CTA of this one has
    // started: what it does before its griddepcontrol.wait (barriers, tensor
    // memory, the first x, B, C copies) reads nothing this pass writes, and
    // that wait returns only once this grid has completed and its writes
    // (the bulk stores included) are visible.
    pdl_launch_dependents();

    if (t == 0) {
        mbar_init(&sm.bar_ld, 1);
        mbar_init(&sm.bar_mma, 1);
        mbar_fence_init();
        mbar_arrive_expect_tx(&sm.bar_ld, 2 * kTile);
        tma_load_4d(sm.Bt, &tmB, &sm.bar_ld, 0, h / (H / prm.G), c * kQ, b);
        tma_load_4d(sm.X, &tmX, &sm.bar_ld, 0, h, c * kQ, b);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 128);
        tmem_relinquish();
    }
    // the tile's cumulative sums (row t), rows past L: dt = 0
    const int r = c * kQ + t;
    const float dv = r < L ? prep_dt<EXT>(__bfloat162float(prm.dt[(int64_t(b) * L + r) * H + h]), prm,
                                          (EXT && prm.dt_bias) ? prm.dt_bias[h] : 0.0f)
                           : 0.0f;
    const float dA = dv * prm.A[h] * SSM_LOG2E;
    float v = dA;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) sm.wsum[warp] = v;
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    float off = 0.0f, tot = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        off += (w < warp) ? sm.wsum[w] : 0.0f;
        tot += sm.wsum[w];
    }
    const float cum = v + off, excl = cum - dA;
    bool ok = mbar_wait_bounded(&sm.bar_ld, 0, &never, kWaitLimitNs);
    if (ok) {
        // row t: the reverse weights into XR, the forward weights in place
        // (same swizzle: 16-byte chunks map one to one)
        const float wf = ex2(tot - cum) * dv, wr = ex2(excl) * dv;
        const float2 f2 = make_float2(wf, wf), r2 = make_float2(wr, wr);
        uint4 *src = reinterpret_cast<uint4 *>(sm.X + t * 128);
        uint4 *dst = reinterpret_cast<uint4 *>(sm.XR + t * 128);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int j = jj ^ (t & 7);      // (rows of a warp hit different banks)
            const uint4 x4 = src[j];
            const float2 a = unpack_bf16(x4.x), bb = unpack_bf16(x4.y), cc = unpack_bf16(x4.z),
                         dd = unpack_bf16(x4.w);
            float2 p0 = fmul2(a, r2), p1 = fmul2(bb, r2), p2 = fmul2(cc, r2), p3 = fmul2(dd, r2);
            dst[j] = make_uint4(pack_bf16(p0.x, p0.y), pack_bf16(p1.x, p1.y), pack_bf16(p2.x, p2.y),
                                pack_bf16(p3.x, p3.y));
            p0 = fmul2(a, f2), p1 = fmul2(bb, f2), p2 = fmul2(cc, f2), p3 = fmul2(dd, f2);
            src[j] = make_uint4(pack_bf16(p0.x, p0.y), pack_bf16(p1.x, p1.y), pack_bf16(p2.x, p2.y),
                                pack_bf16(p3.x, p3.y));
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    if (__syncthreads_or(!ok)) ok = false;
    bool issued = false;   // (thread 0)
    if (ok && t == 0) {
        issued = true;
        tc_fence_after_sync();
        constexpr uint32_t idS = idesc_bf16_f32(128, 128, true, true);
        const uint32_t sB = smem_addr(sm.Bt), sX = smem_addr(sm.X);
        const uint32_t lboA = smem_addr(sm.X) - sB, lboB = smem_addr(sm.XR) - sX;
#pragma unroll
        for (int kk = 0; kk < kQ / 16; ++kk)
            mma_bf16_ss(tmem, smem_desc(sB + kk * 2048, lboA, 1024, kSwizzle128B),
                        smem_desc(sX + kk * 2048, lboB, 1024, kSwizzle128B), idS, kk > 0);
        mma_commit(&sm.bar_mma);
    }
    if (ok) ok = mbar_wait_bounded(&sm.bar_mma, 0, &never, kWaitLimitNs);
    tc_fence_after_sync();
    if (__syncthreads_or(!ok)) ok = false;
    if (ok) {
        // lanes n = t < 64: Sf, Sr rows as bf16, staged (swizzled chunks) in
        // the x buffers (the product has read them), then two bulk copies of 8 KB
        if (warp < 2) {
            const uint32_t lb = uint32_t(warp * 32) << 16;
            uint32_t vv[2][32];
            tmem_ld32_async(tmem + lb, vv[0]);
            tmem_ld32_async(tmem + lb + 32, vv[1]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                tmem_wait_tie(vv[q & 1]);
                uint4 *row = reinterpret_cast<uint4 *>((q < 2 ? sm.X : sm.XR) + t * 128);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    row[((q & 1) * 4 + j) ^ (t & 7)] = make_uint4(
                        pack_bf16(__uint_as_float(vv[q & 1][8 * j]), __uint_as_float(vv[q & 1][8 * j + 1])),
                        pack_bf16(__uint_as_float(vv[q & 1][8 * j + 2]), __uint_as_float(vv[q & 1][8 * j + 3])),
                        pack_bf16(__uint_as_float(vv[q & 1][8 * j + 4]), __uint_as_float(vv[q & 1][8 * j + 5])),
                        pack_bf16(__uint_as_float(vv[q & 1][8 * j + 6]), __uint_as_float(vv[q & 1][8 * j + 7])));
                if (q < 2) tmem_ld32_async(tmem + lb + (q + 2) * 32, vv[q & 1]);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (t == 0) {
            bulk_store(prm.chunk + ((size_t(bh) * 2 + 0) * nc + c) * kState, sm.X, kState);
            bulk_store(prm.chunk + ((size_t(bh) * 2 + 1) * nc + c) * kState, sm.XR, kState);
            bulk_commit();
            prm.tot[size_t(bh) * kMaxTiles + c] = tot;
            bulk_wait_read0();            // the stores have read the staging (shared memory)
        }
    } else if (t == 0) {
        atomicOr(&g_device_error, 1u);
        // a product may still be in flight: give it a bounded chance to finish
        mma_commit(&sm.bar_mma);
        (void)mbar_wait_bounded(&sm.bar_mma, issued ? 1u : 0u, &never, 100000000ull);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 128);
    }
}

// ===========================================================================
// Pass 2: outputs of every tile (persistent)
// ===========================================================================
// Roles, as in the unidirectional kernel: eight math warps (warps w and w + 4
// read TMEM lane quarter q = w % 4: tile rows 32 q .. 32 q + 31, and split
// the work of those rows by column halves hf = w / 4), warp 8 issues every
// tcgen05.mma of G and Z, warp 11 those of Y, warp 9 every copy, warp 10
// computes the per-tile vectors.
// The CTA walks its tiles k = 0, 1, .. (tile blockIdx.x + k gridDim.x); the
// products of tile k + 1 run while the outputs of tile k are written.
constexpr int kMath = 256;
constexpr int kThreads = kMath + 128;
constexpr uint32_t kLaunchRegs = 168, kCtrlRegs = 40, kMathRegs = 232;
static_assert(kCtrlRegs + 2 * kMathRegs <= 3 * kLaunchRegs,
              "the register split must fit in what the CTA is launched with");
constexpr int kSlots = 3;
// Tensor-memory columns: G (128), Y by tile parity (64 each), Z = [Zf | Zr]
// (128), the mask M (bf16 pairs, 64).
constexpr uint32_t kColG = 0, kColY0 = 128, kColY1 = 192, kColZ = 256, kColM = 384;

struct __align__(1024) OutSmem {
    uint8_t C[2][kTile];             // C tile of tile k in k % 2 (K-major rows t, 64 n)
    uint8_t B[2][kTile];             // B tile, rows s
    uint8_t X[2][kTile];             // x tile (MN-major B operand of Y); then y staging
    uint8_t IMG[2][2][kImg];         // [tile parity][S_in, R_in]: bf16 images, rows n, 64 p
    uint8_t YS[8][32 * 128];         // per math warp: 32 rows x 32 fp32 of y (128-byte swizzle), out by TMA
    uint8_t SB[kMaxTiles - 1][kState];   // the chunk states one tile combines (bf16, swizzled rows)
    float TOT[kMaxTiles];            // the decay totals of its sequence's tiles
    float cum[kSlots][kQ];
    float excl[kSlots][kQ];
    float dtv[kSlots][kQ];
    float csf[kSlots][kQ];           // column factors of the forward off-diagonal blocks
    float csr[kSlots][kQ];           // column factors of the reverse off-diagonal blocks
    float tot[kSlots];
    // A parity wait cannot tell phase k from phase k + 2, so bar_st is one
    // per tile parity (the images of tile k + 1 are written right after the
    // outputs of tile k, before Z(k) need have been issued).
    uint64_t bar_c[2], bar_b[2], bar_x[2], bar_sb;       // copies landed
    uint64_t bar_g, bar_y[2], bar_z[2];                  // products finished
    uint64_t bar_gfree, bar_mfull, bar_zfree, bar_st[2], bar_sbfree;   // math -> issue / copy
    uint64_t bar_vec[kSlots], bar_fin[2];
    uint64_t bar_slot[kSlots];                           // math warps done with a vector slot
    uint32_t tmem_base;
};

struct Ctx {
    OutSmem &sm;
    const Params &prm;
    int nk;                 // tiles of this CTA
    float Dh_unused;
    uint32_t tmem;
    volatile int *abort;
};

// the k-th tile of this CTA: (batch * head, tile) and its batch, head, group
struct Unit {
    int bh, c, b, h, grp;
};
__device__ __forceinline__ Unit unit_of(const Params &prm, int k) {
    Unit un;
    const int u = blockIdx.x + k * gridDim.x;
    un.bh = u / prm.nc;
    un.c = u % prm.nc;
    un.b = un.bh / prm.H;
    un.h = un.bh % prm.H;
    un.grp = un.h / (prm.H / prm.G);
    return un;
}

__device__ __forceinline__ bool test_wait(uint64_t *bar, uint32_t parity) {
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
__device__ __forceinline__ void arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

#define BI_WAIT(bar, ph)                                                                  \
    do {                                                                                  \
        if (!mbar_wait_bounded(&(bar), (ph), cx.abort, kWaitLimitNs)) return false;       \
        (ph) ^= 1u;                                                                       \
    } while (0)
#define BI_WAIT_I(bar, bits, i)                                                           \
    do {                                                                                  \
        if (!mbar_wait_bounded(&(bar), ((bits) >> (i)) & 1u, cx.abort, kWaitLimitNs))    \
            return false;                                                                 \
        (bits) ^= 1u << (i);                                                              \
    } while (0)

// ---- the issuing threads ---------------------------------------------------------------
// Warp 8 issues G and Z, warp 11 issues Y, each stream as soon as its inputs
// are ready (two threads, so that the Y product -- the one the next tile's
// mask store waits for -- is not held up behind the other polls):
//   G(k):  C(k), B(k) landed and G(k - 1) read by the math warps;
//   Z(k):  the state images of tile k written, G(k) issued (C(k) landed) and
//          Z(k - 1) read by the math warps (one Z accumulator);
//   Y(k):  mask(k) stored -- which the math warps do after reading G(k), so
//          G(k) has ended -- and x(k) landed.
__device__ __forceinline__ bool issuer_gz_role(Ctx &cx) {
    auto &sm = cx.sm;
    const int nk = cx.nk;
    const uint32_t tmem = cx.tmem;
    constexpr uint32_t idG = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idZ = idesc_bf16_f32(128, 128, false, true);
    uint32_t ph_c = 0, ph_b = 0;             // one bit per buffer
    uint32_t ph_gfree = 0, ph_st = 0, ph_zfree = 0;   // ph_st: one bit per parity
    int g_next = 0, z_next = 0;
    uint64_t t_idle = 0;
    uint32_t idle_passes = 0;
    while (g_next < nk || z_next < nk) {
        bool progress = false;
        if (g_next < nk && (g_next == 0 || test_wait(&sm.bar_gfree, ph_gfree)) &&
            test_wait(&sm.bar_c[g_next & 1], (ph_c >> (g_next & 1)) & 1u) &&
            test_wait(&sm.bar_b[g_next & 1], (ph_b >> (g_next & 1)) & 1u)) {
            if (g_next > 0) ph_gfree ^= 1u;
            ph_c ^= 1u << (g_next & 1);
            ph_b ^= 1u << (g_next & 1);
            tc_fence_after_sync();
            const uint32_t sC = smem_addr(sm.C[g_next & 1]), sB = smem_addr(sm.B[g_next & 1]);
#pragma unroll
            for (int kk = 0; kk < kN / 16; ++kk)
                mma_bf16_ss(tmem + kColG, smem_desc(sC + kk * 32, 16, 1024, kSwizzle128B),
                            smem_desc(sB + kk * 32, 16, 1024, kSwizzle128B), idG, kk > 0);
            mma_commit(&sm.bar_g);
            ++g_next;
            progress = true;
        }
        if (z_next < nk && g_next > z_next &&
            test_wait(&sm.bar_st[z_next & 1], (ph_st >> (z_next & 1)) & 1u) &&
            (z_next == 0 || test_wait(&sm.bar_zfree, ph_zfree))) {
            ph_st ^= 1u << (z_next & 1);
            if (z_next > 0) ph_zfree ^= 1u;
            tc_fence_after_sync();
            // Z = C [S_in | R_in]^T: B operand = the two images side by side (N = 128)
            const uint32_t sC = smem_addr(sm.C[z_next & 1]), sI = smem_addr(sm.IMG[z_next & 1]);
#pragma unroll
            for (int kk = 0; kk < kN / 16; ++kk)
                mma_bf16_ss(tmem + kColZ, smem_desc(sC + kk * 32, 16, 1024, kSwizzle128B),
                            smem_desc(sI + kk * 2048, kImg, 1024, kSwizzle128B), idZ, kk > 0);
            mma_commit(&sm.bar_z[z_next & 1]);
            ++z_next;
            progress = true;
        }
        if (progress) {
            t_idle = 0;
            idle_passes = 0;
        } else if ((++idle_passes & 255u) == 0) {
            const uint64_t now = globaltimer_ns();
            if (t_idle == 0) t_idle = now;
            else if (now - t_idle > kWaitLimitNs || *cx.abort) return false;
        }
    }
    return true;
}
__device__ __forceinline__ bool issuer_y_role(Ctx &cx) {
    auto &sm = cx.sm;
    const int nk = cx.nk;
    const uint32_t tmem = cx.tmem;
    constexpr uint32_t idY = idesc_bf16_f32(128, 64, false, true);
    uint32_t ph_mfull = 0, ph_x = 0;          // ph_x: one bit per buffer
    for (int k = 0; k < nk; ++k) {
        const int xb = k & 1;
        BI_WAIT(sm.bar_mfull, ph_mfull);
        BI_WAIT_I(sm.bar_x[xb], ph_x, xb);
        tc_fence_after_sync();
        // Y = M X: A = the mask in tensor memory, B = the x tile (MN-major)
        const uint32_t sX = smem_addr(sm.X[xb]);
        const uint32_t dcol = (k & 1) ? kColY1 : kColY0;
#pragma unroll
        for (int kk = 0; kk < kQ / 16; ++kk)
            mma_bf16_ts(tmem + dcol, tmem + kColM + kk * 8,
                        smem_desc(sX + kk * 2048, kTile, 1024, kSwizzle128B), idY, kk > 0);
        mma_commit(&sm.bar_y[k & 1]);
    }
    return true;
}

// ---- the copying thread -----------------------------------------------------------------
// x, B, C of tile k + 2 into the buffers of tile k once its products are done
// (Y(k) ends after G(k): x(k), B(k) read; Z(k) reads C(k)); the chunk states
// tile k + 1 combines once the math warps have combined tile k's.
__device__ __forceinline__ bool loader_role(Ctx &cx, const CUtensorMap *tmC, const CUtensorMap *tmB,
                                            const CUtensorMap *tmX) {
    auto &sm = cx.sm;
    const Params &prm = cx.prm;
    const int nk = cx.nk, nc = prm.nc;
    uint32_t ph_y = 0, ph_z = 0, ph_sbfree = 0;   // ph_y, ph_z: one bit per parity
    auto load_bc = [&](int k) {
        const Unit un = unit_of(prm, k);
        const int buf = k & 1;
        mbar_arrive_expect_tx(&sm.bar_b[buf], kTile);
        tma_load_4d(sm.B[buf], tmB, &sm.bar_b[buf], 0, un.grp, un.c * kQ, un.b);
        mbar_arrive_expect_tx(&sm.bar_c[buf], kTile);
        tma_load_4d(sm.C[buf], tmC, &sm.bar_c[buf], 0, un.grp, un.c * kQ, un.b);
    };
    auto load_x = [&](int k) {
        const Unit un = unit_of(prm, k);
        const int buf = k & 1;
        mbar_arrive_expect_tx(&sm.bar_x[buf], kTile);
        tma_load_4d(sm.X[buf], tmX, &sm.bar_x[buf], 0, un.h, un.c * kQ, un.b);
    };
    // the states entering tile k: forward states of the tiles before it,
    // reverse states of the tiles after it (one contiguous run each), and
    // the decay totals of its sequence
    auto load_states = [&](int k) {
        const Unit un = unit_of(prm, k);
        const int nf = un.c, nr = nc - 1 - un.c;
        mbar_arrive_expect_tx(&sm.bar_sb, uint32_t(nf + nr) * kState + kMaxTiles * 4);
        if (nf > 0)
            bulk_load(sm.SB[0], prm.chunk + (size_t(un.bh) * 2 + 0) * nc * kState,
                      uint32_t(nf) * kState, &sm.bar_sb);
        if (nr > 0)
            bulk_load(sm.SB[nf], prm.chunk + ((size_t(un.bh) * 2 + 1) * nc + un.c + 1) * kState,
                      uint32_t(nr) * kState, &sm.bar_sb);
        bulk_load(sm.TOT, prm.tot + size_t(un.bh) * kMaxTiles, kMaxTiles * 4, &sm.bar_sb);
    };
    load_bc(0);
    load_x(0);
    if (nk > 1) {
        load_bc(1);
        load_x(1);
    }
    pdl_wait();                          // the chunk states of the first pass
    load_states(0);
    for (int k = 0; k < nk; ++k) {
        if (k + 1 < nk) {
            BI_WAIT(sm.bar_sbfree, ph_sbfree);     // tile k's states combined
            load_states(k + 1);
        }
        BI_WAIT_I(sm.bar_y[k & 1], ph_y, k & 1);   // G(k), Y(k) done: B(k), x(k) read
        if (k + 2 < nk) load_x(k + 2);
        BI_WAIT_I(sm.bar_z[k & 1], ph_z, k & 1);   // Z(k) done: C(k) read
        if (k + 2 < nk) load_bc(k + 2);
    }
    return true;
}

// ---- the vector warp --------------------------------------------------------------------
// Per-tile vectors up to two tiles ahead (lane l: rows 4 l .. 4 l + 3):
// cumulative sums of dt A (log2 units), their exclusive form, dt, the column
// factors of the off-diagonal mask blocks in both directions, the total.
// Slot k % 3 held tile k - 3: the math warps signal their last read of it on
// the slot's own barrier.  (A parity wait on the mask stores instead could
// alias: with this warp held up -- by a slow dt load, say -- the math warps
// could complete the stores of tiles k - 2 and k - 1 first, and the wait for
// the first would then wait for the store of tile k, which needs this warp.
// A slot's barrier cannot complete again before this warp writes the slot.)
template <bool EXT>
__device__ __forceinline__ bool vector_role(Ctx &cx) {
    auto &sm = cx.sm;
    const Params &prm = cx.prm;
    const int lane = threadIdx.x & 31;
    const int nk = cx.nk, L = prm.L, H = prm.H;
    uint32_t ph_slot = 0;   // one bit per slot
    float raw[4], nxt[4];
    auto load = [&](int k, float (&rr)[4]) {
        const Unit un = unit_of(prm, k);
        const __nv_bfloat16 *dtp = prm.dt + (int64_t(un.b) * L) * H + un.h;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int row = un.c * kQ + 4 * lane + j;
            rr[j] = row < L ? __bfloat162float(dtp[int64_t(row) * H]) : 0.0f;
        }
    };
    load(0, raw);
    for (int k = 0; k < nk; ++k) {
        if (k + 1 < nk) load(k + 1, nxt);
        const int p = k % kSlots;
        if (k >= kSlots) BI_WAIT_I(sm.bar_slot[p], ph_slot, p);   // tile k - 3 done with slot p
        const Unit un = unit_of(prm, k);
        const float Ah = prm.A[un.h] * SSM_LOG2E;
        const float bias = (EXT && prm.dt_bias) ? prm.dt_bias[un.h] : 0.0f;
        float dv[4], cs[4], da[4], run = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float d = (un.c * kQ + 4 * lane + j < L) ? prep_dt<EXT>(raw[j], prm, bias) : 0.0f;
            dv[j] = d;
            da[j] = d * Ah;
            run += da[j];
            cs[j] = run;
        }
        float incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        const float base = incl - run;
        float ex[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            cs[j] += base;
            ex[j] = cs[j] - da[j];
        }
        // block of 32 rows of row s: lanes 8 blk .. 8 blk + 7
        const float end = __shfl_sync(0xffffffffu, cs[3], lane | 7);      // cum at the block's end
        const float start = __shfl_sync(0xffffffffu, ex[0], lane & ~7);  // excl at its start
        const float tot = __shfl_sync(0xffffffffu, cs[3], 31);
        reinterpret_cast<float4 *>(sm.cum[p])[lane] = make_float4(cs[0], cs[1], cs[2], cs[3]);
        reinterpret_cast<float4 *>(sm.excl[p])[lane] = make_float4(ex[0], ex[1], ex[2], ex[3]);
        reinterpret_cast<float4 *>(sm.dtv[p])[lane] = make_float4(dv[0], dv[1], dv[2], dv[3]);
        reinterpret_cast<float4 *>(sm.csf[p])[lane] =
            make_float4(ex2(end - cs[0]) * dv[0], ex2(end - cs[1]) * dv[1], ex2(end - cs[2]) * dv[2],
                        ex2(end - cs[3]) * dv[3]);
        reinterpret_cast<float4 *>(sm.csr[p])[lane] =
            make_float4(ex2(ex[0] - start) * dv[0], ex2(ex[1] - start) * dv[1],
                        ex2(ex[2] - start) * dv[2], ex2(ex[3] - start) * dv[3]);
        if (lane == 0) sm.tot[p] = tot;
        arrive(&sm.bar_vec[p]);
#pragma unroll
        for (int j = 0; j < 4; ++j) raw[j] = nxt[j];
    }
    return true;
}

// Half hf (32 p) of row n of a bf16 state image (64 p, 128-byte swizzle).
__device__ __forceinline__ void put_image_half(uint8_t *img, int n, int hf, const float (&s)[32]) {
    uint8_t *rowp = img + n * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4 *>(rowp + (((4 * hf + j) ^ (n & 7)) << 4)) =
            make_uint4(pack_bf16(s[8 * j], s[8 * j + 1]), pack_bf16(s[8 * j + 2], s[8 * j + 3]),
                       pack_bf16(s[8 * j + 4], s[8 * j + 5]), pack_bf16(s[8 * j + 6], s[8 * j + 7]));
}

// ---- the eight math warps ----------------------------------------------------------------
template <bool EXT>
__device__ __forceinline__ bool math_role(Ctx &cx, const CUtensorMap *tmY) {
    auto &sm = cx.sm;
    const Params &prm = cx.prm;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, hf = warp >> 2;
    const int t = q * 32 + lane;
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    const int nk = cx.nk, L = prm.L, H = prm.H;
    const uint32_t tmem = cx.tmem;
    uint32_t ph_g = 0, ph_y = 0, ph_z = 0, ph_vec = 0, ph_sb = 0;   // ph_y, ph_z, ph_vec: bits
    const int nc = prm.nc;
    // combine part of this thread: state row n, direction d, columns of half hf
    const int cn = 32 * (warp & 1) + lane, cd = (warp >> 1) & 1;

    // The states entering tile k (in SB / TOT), combined in fp32 and written
    // as the bf16 images of tile k's parity; then the Z product may start.
    auto combine = [&](int k) -> bool {
        const Unit un = unit_of(prm, k);
        BI_WAIT(sm.bar_sb, ph_sb);
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
        const int nf = un.c, nr = nc - 1 - un.c;
        // forward: S_in = sum over j < c in order, acc <- e^{tot_j} acc + Sf(j);
        // reverse: R_in = sum over j > c from the last, acc <- e^{tot_j} acc + Sr(j)
        const int cnt = cd == 0 ? nf : nr;
        for (int i = 0; i < cnt; ++i) {
            const int j = cd == 0 ? i : nc - 1 - i;              // tile
            const int slot = cd == 0 ? i : nf + (j - un.c - 1);  // its state in SB
            const float e = ex2(sm.TOT[j]);
            const uint4 *src = reinterpret_cast<const uint4 *>(sm.SB[slot] + cn * 128);
            uint4 s4[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) s4[q4] = src[(hf * 4 + q4) ^ (cn & 7)];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const uint32_t w4[4] = {s4[q4].x, s4[q4].y, s4[q4].z, s4[q4].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 v2 = unpack_bf16(w4[i]);
                    acc[8 * q4 + 2 * i] = fmaf(e, acc[8 * q4 + 2 * i], v2.x);
                    acc[8 * q4 + 2 * i + 1] = fmaf(e, acc[8 * q4 + 2 * i + 1], v2.y);
                }
            }
        }
        arrive(&sm.bar_sbfree);          // the copying thread may refill SB / TOT
        put_image_half(sm.IMG[k & 1][cd], cn, hf, acc);
        fence_proxy_async_smem();
        arrive(&sm.bar_st[k & 1]);
        return true;
    };
    // Mask rows t of tile k into registers (bf16 pairs).  Row quarter q has
    // the diagonal block sb = q (direct exponentials of differences, both
    // triangles, the diagonal counted once per direction, plus D) and three
    // blocks off it (row factor x column factor, both <= 1): half 0 forms
    // columns 0..15 of the diagonal block and the first off-diagonal block,
    // half 1 columns 16..31 and the other two.
    uint32_t mkd[8], mk[2][16];
    // the off-diagonal blocks of quarter q, in increasing order
    const int ob0 = q == 0 ? 1 : 0, ob1 = q <= 1 ? 2 : 1, ob2 = q <= 2 ? 3 : 2;
    auto mask = [&](int k) -> bool {
        const int p = k % kSlots;
        BI_WAIT_I(sm.bar_vec[p], ph_vec, p);
        BI_WAIT(sm.bar_g, ph_g);
        tc_fence_after_sync();
        const float *cum = sm.cum[p];
        const float *excl = sm.excl[p];
        const float *dtv = sm.dtv[p];
        const float cum_t = cum[t], excl_t = excl[t];
        auto offdiag = [&](int i, int sb, const uint32_t (&g)[32]) {
            const bool fwd = sb < q;
            const float e = fwd ? ex2(cum_t - cum[sb * 32 + 31]) : ex2(excl[sb * 32] - excl_t);
            const float2 ee = make_float2(e, e);
            const float4 *f4 = reinterpret_cast<const float4 *>((fwd ? sm.csf[p] : sm.csr[p]) + sb * 32);
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
        uint32_t gd[16], ga[32];
        tmem_ld16_async(tmem + lane_base + kColG + q * 32 + hf * 16, gd);
        tmem_ld32_async(tmem + lane_base + kColG + (hf == 0 ? ob0 : ob1) * 32, ga);
        tmem_wait_tie(ga);
        reg_tie16(gd);
        uint32_t gb[32];
        if (hf == 1) tmem_ld32_async(tmem + lane_base + kColG + ob2 * 32, gb);
        {
            // columns j = 16 hf .. 16 hf + 15 of the diagonal block
            const Unit un = unit_of(prm, k);
            const float Dh = prm.D ? prm.D[un.h] : 0.0f;
            const float4 *c4 = reinterpret_cast<const float4 *>(cum + q * 32 + hf * 16);
            const float4 *e4 = reinterpret_cast<const float4 *>(excl + q * 32 + hf * 16);
            const float4 *d4 = reinterpret_cast<const float4 *>(dtv + q * 32 + hf * 16);
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
                const float4 cs = c4[j4], es = e4[j4], ds = d4[j4];
                const float csv[4] = {cs.x, cs.y, cs.z, cs.w};
                const float esv[4] = {es.x, es.y, es.z, es.w};
                const float dsv[4] = {ds.x, ds.y, ds.z, ds.w};
                float m[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = hf * 16 + 4 * j4 + i;
                    // one exponential: s < t forward, s > t reverse; s = t: 1 + 1
                    const float arg = (j < lane) ? cum_t - csv[i] : ((j > lane) ? esv[i] - excl_t : 0.0f);
                    const float w = ex2(arg) + ((j == lane) ? 1.0f : 0.0f);
                    float v = __uint_as_float(gd[4 * j4 + i]) * (w * dsv[i]);
                    if (j == lane) v += Dh;
                    m[i] = v;
                }
                mkd[2 * j4] = pack_bf16(m[0], m[1]);
                mkd[2 * j4 + 1] = pack_bf16(m[2], m[3]);
            }
        }
        // one call site for the first off-diagonal block of either half
        if (hf == 0) {
            tc_fence_before_sync();
            arrive(&sm.bar_gfree);
        }
        offdiag(0, hf == 0 ? ob0 : ob1, ga);
        if (hf == 1) {
            tmem_wait_tie(gb);
            tc_fence_before_sync();
            arrive(&sm.bar_gfree);
            offdiag(1, ob2, gb);
        }
        return true;
    };
    auto mask_store = [&]() {
        tmem_st_32x32b_x8(tmem + lane_base + kColM + q * 16 + hf * 8, mkd);
        tmem_st_32x32b_x16(tmem + lane_base + kColM + (hf == 0 ? ob0 : ob1) * 16, mk[0]);
        if (hf == 1) tmem_st_32x32b_x16(tmem + lane_base + kColM + ob2 * 16, mk[1]);
        tmem_wait_st();
        tc_fence_before_sync();
        arrive(&sm.bar_mfull);
    };
    const bool gate = EXT && prm.z != nullptr;

    if (!combine(0)) return false;
    if (!mask(0)) return false;
    mask_store();
    for (int k = 0; k < nk; ++k) {
        const bool more = k + 1 < nk;
        const Unit un = unit_of(prm, k);
        if (gate && un.c * kQ + t < L)   // the gate row of tile k, read by its epilogue below
            asm volatile("prefetch.global.L1 [%0];" ::"l"(
                prm.z + ((size_t(un.b) * L + un.c * kQ + t) * H + un.h) * kP + hf * 32));
        if (more && !mask(k + 1)) return false;
        BI_WAIT_I(sm.bar_y[k & 1], ph_y, k & 1);   // G(k), Y(k) done
        BI_WAIT_I(sm.bar_z[k & 1], ph_z, k & 1);   // Z(k) done
        tc_fence_after_sync();
        const int p = k % kSlots;
        const float ef = ex2(sm.cum[p][t]), er = ex2(sm.tot[p] - sm.excl[p][t]);
        arrive(&sm.bar_slot[p]);             // tile k's vectors are read for the last time
        uint32_t yv[32], zf[32], zr[32];
        tmem_ld32_async(tmem + lane_base + ((k & 1) ? kColY1 : kColY0) + hf * 32, yv);
        tmem_ld32_async(tmem + lane_base + kColZ + hf * 32, zf);
        tmem_ld32_async(tmem + lane_base + kColZ + 64 + hf * 32, zr);
        tmem_wait_tie(yv);
        reg_tie(zf);
        reg_tie(zr);
        tc_fence_before_sync();
        arrive(&sm.bar_zfree);               // Z may be overwritten now
        if (more) mask_store();              // Y(k + 1) may start
        // y rows t, columns of half hf: staged in this warp's tile (128-byte
        // swizzle, the layout of a 32-row x 32-float TMA box), one TMA store
        // (rows past L are clipped by the store)
        float out[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            out[j] = fmaf(er, __uint_as_float(zr[j]), fmaf(ef, __uint_as_float(zf[j]), __uint_as_float(yv[j])));
        const int row0 = un.c * kQ;
        if (gate && row0 + t < L) {
            const uint4 *zp = reinterpret_cast<const uint4 *>(prm.z + ((size_t(un.b) * L + row0 + t) * H + un.h) * kP + hf * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 zv = __ldg(zp + j);
                const uint32_t w4[4] = {zv.x, zv.y, zv.z, zv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 zz = unpack_bf16(w4[i]);
                    out[8 * j + 2 * i] *= silu_fast(zz.x);
                    out[8 * j + 2 * i + 1] *= silu_fast(zz.y);
                }
            }
        }
        uint8_t *stg = sm.YS[warp];
        if (lane == 0) bulk_wait_read0();    // the previous tile's store has read the tile
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4 *>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_float4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_4d(tmY, stg, hf * 32, un.h, row0 + q * 32, un.b);
            bulk_commit();
        }
        if (more && !combine(k + 1)) return false;   // then Z(k + 1) may start
    }
    if (lane == 0) bulk_wait0();         // the last stores have left the staging tile
    return true;
}

template <bool EXT>
__global__ void __launch_bounds__(kThreads, 1)
bidir_out_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                 const __grid_constant__ Params prm) {
    extern __shared__ uint8_t smem_raw[];
    OutSmem &sm = *reinterpret_cast<OutSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int nk = (prm.units - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x);

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.bar_c[i], 1);
            mbar_init(&sm.bar_b[i], 1);
            mbar_init(&sm.bar_x[i], 1);
            mbar_init(&sm.bar_y[i], 1);
            mbar_init(&sm.bar_z[i], 1);
        }
        mbar_init(&sm.bar_sb, 1);
        mbar_init(&sm.bar_g, 1);
        mbar_init(&sm.bar_gfree, kMath);
        mbar_init(&sm.bar_mfull, kMath);
        mbar_init(&sm.bar_zfree, kMath);
        mbar_init(&sm.bar_st[0], kMath);
        mbar_init(&sm.bar_st[1], kMath);
        mbar_init(&sm.bar_sbfree, kMath);
        mbar_init(&sm.bar_fin[0], 1);
        mbar_init(&sm.bar_fin[1], 1);
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&sm.bar_vec[i], 32);
            mbar_init(&sm.bar_slot[i], kMath);
        }
        mbar_fence_init();
        prefetch_tmap(&tmC);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmY);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    Ctx cx{sm, prm, nk, 0.0f, sm.tmem_base, &abort_flag};
    bool ok = true;
    if (warp < 8) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kMathRegs));
        ok = math_role<EXT>(cx, &tmY);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
        if (tid == 256) ok = issuer_gz_role(cx);
        if (tid == 288) ok = loader_role(cx, &tmC, &tmB, &tmX);
        if (warp == 10) ok = vector_role<EXT>(cx);
        if (tid == 352) ok = issuer_y_role(cx);
    }
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
        tmem_dealloc(sm.tmem_base, 512);
    }
}
#undef BI_WAIT
#undef BI_WAIT_I

// ===========================================================================
// Host side
// ===========================================================================
// The driver's tensor-map encoder.  Only a successful lookup is kept: after
// a failed one the next call asks the driver again.
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_acquire);
    if (fn != nullptr) return fn;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess) {
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cached.store(fn, std::memory_order_release);
    }
    return fn;
}

static bool make_map(CUtensorMap *m, const void *base, const cuuint64_t *dims,
                     const cuuint64_t *strides_bytes, const cuuint32_t *box,
                     CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, dtype, 4, const_cast<void *>(base), dims, strides_bytes,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool supported(int64_t L, int64_t P, int64_t N) {
    return P == kP && N == kN && L >= 1 && (L + kQ - 1) / kQ <= kMaxTiles;
}

size_t scratch_bytes(int64_t Bs, int64_t H, int64_t L) {
    const int64_t nc = (L + kQ - 1) / kQ;
    return size_t(Bs) * size_t(H) * (size_t(2 * nc) * kState + kMaxTiles * 4);
}

// The bidirectional scan of bf16 inputs with P = 64, N = 64 and at most
// four 128-row tiles: pass 1 then pass 2 (launched to overlap pass 1's tail).
cudaError_t launch(const __nv_bfloat16 *x, const __nv_bfloat16 *dt, const float *A_head,
                   const __nv_bfloat16 *Bm, const __nv_bfloat16 *Cm, const float *D, float *y,
                   int64_t Bs, int64_t L, int64_t H, int num_sms, const ScanOpts *opt,
                   cudaStream_t stream) {
    const int64_t G = (opt && opt->ngroups > 1) ? opt->ngroups : 1;
    const int nc = int((L + kQ - 1) / kQ);
    const int64_t units64 = Bs * H * nc;
    if (units64 > 0x7fffffff || nc > kMaxTiles) return cudaErrorNotSupported;
    CUtensorMap tmC, tmB, tmX, tmY;
    const cuuint64_t dbc[4] = {cuuint64_t(kN), cuuint64_t(G), cuuint64_t(L), cuuint64_t(Bs)};
    const cuuint64_t sbc[3] = {cuuint64_t(kN) * 2, cuuint64_t(G) * kN * 2, cuuint64_t(L) * G * kN * 2};
    const cuuint32_t box[4] = {64, 1, kQ, 1};
    const cuuint64_t dx[4] = {cuuint64_t(kP), cuuint64_t(H), cuuint64_t(L), cuuint64_t(Bs)};
    const cuuint64_t sx[3] = {cuuint64_t(kP) * 2, cuuint64_t(H) * kP * 2, cuuint64_t(L) * H * kP * 2};
    const cuuint64_t sy[3] = {cuuint64_t(kP) * 4, cuuint64_t(H) * kP * 4, cuuint64_t(L) * H * kP * 4};
    const cuuint32_t boxy[4] = {32, 1, 32, 1};
    if (!make_map(&tmC, Cm, dbc, sbc, box) || !make_map(&tmB, Bm, dbc, sbc, box) ||
        !make_map(&tmX, x, dx, sx, box) ||
        !make_map(&tmY, y, dx, sy, boxy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
        return cudaErrorInvalidValue;

    Params prm{};
    prm.dt = dt;
    prm.A = A_head;
    prm.D = D;
    prm.y = y;
    prm.L = int(L);
    prm.H = int(H);
    prm.nc = nc;
    prm.G = int(G);
    prm.units = int(units64);
    const ScanOpts none{};
    const ScanOpts &o = opt ? *opt : none;
    prm.dt_bias = o.dt_bias;
    prm.z = static_cast<const __nv_bfloat16 *>(o.z);
    prm.dt_min = o.dt_min;
    prm.dt_max = o.dt_max;
    prm.dt_softplus = o.dt_softplus;
    prm.dt_limit = o.dt_limit;

    void *scratch = nullptr;
    cudaError_t err = cudaMallocAsync(&scratch, scratch_bytes(Bs, H, L), stream);
    if (err != cudaSuccess) return err;
    prm.chunk = static_cast<uint8_t *>(scratch);
    prm.tot = reinterpret_cast<float *>(prm.chunk + size_t(Bs) * size_t(H) * 2 * nc * kState);

    // the plain kernels unless an option is on (groups alone need none)
    const bool ext = opt && (opt->dt_bias || opt->dt_softplus || opt->dt_limit || opt->z);
    auto kst = ext ? bidir_state_kernel<true> : bidir_state_kernel<false>;
    auto kout = ext ? bidir_out_kernel<true> : bidir_out_kernel<false>;
    const size_t smem_st = sizeof(StateSmem) + 1024, smem_out = sizeof(OutSmem) + 1024;
    static_assert(sizeof(OutSmem) + 1024 <= 227 * 1024, "shared memory of one CTA exceeds 227 KB");
    err = cudaFuncSetAttribute(kst, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_st));
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(kout, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_out));
    if (err == cudaSuccess) {
        // setmaxnreg re-divides the registers the CTA was launched with
        cudaFuncAttributes fa;
        err = cudaFuncGetAttributes(&fa, kout);
        if (err == cudaSuccess && fa.numRegs < int(kLaunchRegs)) err = cudaErrorNotSupported;
    }
    if (err == cudaSuccess) {
        // pass 1: one CTA per tile
        kst<<<dim3(unsigned(units64)), dim3(128), smem_st, stream>>>(tmB, tmX, prm);
        err = cudaGetLastError();
    }
    if (err == cudaSuccess) {
        const int grid = int(units64 < int64_t(num_sms) ? units64 : int64_t(num_sms));
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(unsigned(grid));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem_out;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, kout, tmC, tmB, tmX, tmY, prm);
    }
    cudaError_t e2 = cudaFreeAsync(scratch, stream);
    return err != cudaSuccess ? err : e2;
}

// Read and clear this unit's device error word (host side, synchronous).
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

}  // namespace bidir
}  // namespace ssm
