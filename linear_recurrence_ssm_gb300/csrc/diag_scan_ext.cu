// diag_scan_ext.cu -- the diagonal scan with its options (delta bias,
// softplus and clamp, silu output gate, initial and final state): the
// kernels of diag_scan.cuh instantiated with the option path compiled in.
#include "diag_scan.cuh"

namespace ssm {
namespace diag {

template <typename Tin>
cudaError_t launch_ext(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                       const float *D, float *y, int64_t Bs, int64_t L, int64_t ED, int64_t N,
                       int num_sms, const Ext &ex, cudaStream_t st) {
    return launch_impl<Tin, true>(x, dlt, A, Bm, Cm, D, y, Bs, L, ED, N, num_sms, ex, st);
}

template cudaError_t launch_ext<float>(const float *, const float *, const float *, const float *,
                                       const float *, const float *, float *, int64_t, int64_t,
                                       int64_t, int64_t, int, const Ext &, cudaStream_t);
template cudaError_t launch_ext<__nv_bfloat16>(const __nv_bfloat16 *, const __nv_bfloat16 *,
                                               const float *, const __nv_bfloat16 *,
                                               const __nv_bfloat16 *, const float *, float *,
                                               int64_t, int64_t, int64_t, int64_t, int,
                                               const Ext &, cudaStream_t);

}  // namespace diag
}  // namespace ssm
