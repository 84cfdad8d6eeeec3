// ssd_chunk_scan.cu -- chunked scalar-decay (SSD) scan for sm_103a.
#include "ssm_common.cuh"

namespace ssm {
namespace ssd {

cudaError_t launch(const __nv_bfloat16 *, const __nv_bfloat16 *, const float *,
                   const __nv_bfloat16 *, const __nv_bfloat16 *, const float *, float *, int64_t,
                   int64_t, int64_t, int64_t, int64_t, int64_t, bool, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace ssd
}  // namespace ssm
