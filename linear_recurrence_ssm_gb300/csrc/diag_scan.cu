// diag_scan.cu -- the plain diagonal scan's entry into the kernels of
// diag_scan.cuh, and the work decomposition shared with the option variant.
#include "diag_scan.cuh"

#include <algorithm>

namespace ssm {
namespace diag {

// Work decomposition.  A warp owns 32/G channels for a time segment and
// keeps 16/G states per lane.  Measured on GB300: a single warp per
// scheduler leaves the MUFU / FMA pipes idle most of the time, two or more
// keep them busy, and the carry pass of a time split costs about a quarter
// of a segment pass.  So: 16 states per lane (G = 1) and no split when that
// already gives >= 1.5 warps per scheduler; otherwise the fewest time
// segments K (each >= 128 steps) that give >= 1.8 warps per scheduler, and
// fewer states per lane only if even 8 segments are not enough.  A plan that
// would need a second wave of CTAs is never chosen.
static int padded_states(int64_t N) {
    return N <= 16 ? 16 : (N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256)));
}

static Plan choose_plan(int64_t Bs, int64_t L, int64_t ED, int N, int num_sms, int max_ctas_per_sm) {
    const int NP = padded_states(N);
    const double schedulers = 4.0 * num_sms;
    auto make = [&](int s, int k) {
        int64_t seg = (L + k - 1) / k;
        seg = (seg + kTileT - 1) / kTileT * kTileT;
        return Plan{s, NP / s, int((L + seg - 1) / seg), int(seg)};
    };
    auto warps = [&](int s, int k) {
        const int g = NP / s;
        return double((Bs * ED * g + 31) / 32) * k;
    };
    auto fits = [&](int s, int k) {
        const int et = kThreads / (NP / s);
        const int64_t ctas = (ED + et - 1) / et * Bs * k;
        return (ctas + num_sms - 1) / num_sms <= max_ctas_per_sm;
    };
    if (warps(16, 1) >= 1.5 * schedulers || NP != 16) {
        // enough channels (or more than 16 states: no split): G = NP / 16
        return make(16, 1);
    }
    Plan best = make(16, 1);
    for (int s = 16; s >= 4; s /= 2) {
        for (int k = 1; k <= kMaxSeg; ++k) {
            const Plan p = make(s, k);
            if (p.K != k || (k > 1 && p.seg_len < 128)) break;
            if (!fits(s, k)) break;
            best = p;
            if (warps(s, k) >= 1.8 * schedulers) return best;
        }
    }
    return best;
}

// The decomposition used for a shape: (S, G, K) and the segment length.
Plan plan_for(int64_t Bs, int64_t L, int64_t ED, int64_t N, int esz, int num_sms) {
    const int NP = padded_states(N);
    // CTAs per SM allowed by shared memory (228 KB per SM, 1 KB reserved per
    // CTA) for the 16-states-per-thread split, capped at 16.
    const int et = kThreads / (NP / 16);
    const int smem = (kStages * 2 * kTileT * et + kStages * 2 * kTileT * NP) * esz +
                     2 * kTileT * NP * 4;
    return choose_plan(Bs, L, ED, int(N), num_sms, std::min(16, (228 * 1024) / (smem + 1024)));
}

template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                   const float *D, float *y, int64_t Bs, int64_t L, int64_t ED, int64_t N,
                   int num_sms, cudaStream_t st) {
    const Ext none{};
    return launch_impl<Tin, false>(x, dlt, A, Bm, Cm, D, y, Bs, L, ED, N, num_sms, none, st);
}

template cudaError_t launch<float>(const float *, const float *, const float *, const float *,
                                   const float *, const float *, float *, int64_t, int64_t, int64_t,
                                   int64_t, int, cudaStream_t);
template cudaError_t launch<__nv_bfloat16>(const __nv_bfloat16 *, const __nv_bfloat16 *,
                                           const float *, const __nv_bfloat16 *,
                                           const __nv_bfloat16 *, const float *, float *, int64_t,
                                           int64_t, int64_t, int64_t, int, cudaStream_t);

}  // namespace diag
}  // namespace ssm
