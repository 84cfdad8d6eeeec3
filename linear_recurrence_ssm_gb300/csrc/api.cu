// api.cu -- the C ABI of libssmscan.so: argument validation, device checks
// and dispatch to the kernels.  See include/ssm_scan.h for the contract.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <limits.h>
#include <mutex>

#include "ssm_common.cuh"

namespace ssm {
namespace diag {
template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                   const float *D, float *y, int64_t Bs, int64_t L, int64_t ED, int64_t N,
                   int num_sms, cudaStream_t st);
template <typename Tin>
cudaError_t launch_ext(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                       const float *D, float *y, int64_t Bs, int64_t L, int64_t ED, int64_t N,
                       int num_sms, const ScanOpts &ex, cudaStream_t st);
struct Plan {
    int S, G, K, seg_len;
};
Plan plan_for(int64_t Bs, int64_t L, int64_t ED, int64_t N, int esz, int num_sms);
}  // namespace diag
namespace diag_bwd {
template <typename Tin>
cudaError_t launch_bwd(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                       const float *D, const float *dy, float *dx, float *ddelta, float *dA,
                       float *dB, float *dC, float *dD, int64_t Bs, int64_t L, int64_t ED,
                       int64_t N, int num_sms, cudaStream_t st);
}
namespace ssd_bwd {
bool supported(int64_t P, int64_t N);
template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dt, const float *A_head, const Tin *Bm, const Tin *Cm,
                   const float *D, const float *dy, float *dx, float *ddt, float *dA, float *dB,
                   float *dC, float *dD, int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                   int64_t G, bool bidir, cudaStream_t st);
}
namespace diag_bwd_ex {
template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dlt, const float *A, const Tin *Bm, const Tin *Cm,
                   const float *D, const float *dy, float *dx, float *ddelta, float *dA, float *dB,
                   float *dC, float *dD, float *dz, float *ddt_bias, float *dh0, int64_t Bs,
                   int64_t L, int64_t ED, int64_t N, const ScanOpts &o, int num_sms,
                   cudaStream_t st);
}
namespace ssd_bwd_ex {
template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dt, const float *A_head, const Tin *Bm, const Tin *Cm,
                   const float *D, const float *dy, float *dx, float *ddt, float *dA, float *dB,
                   float *dC, float *dD, float *dz, float *ddt_bias, float *dh0, int64_t Bs,
                   int64_t L, int64_t H, int64_t P, int64_t N, int64_t G, bool bidir,
                   const ScanOpts &o, int num_sms, cudaStream_t st);
}
namespace ssd_general {
bool supported(int64_t P, int64_t N);
template <typename Tin>
cudaError_t launch(const Tin *x, const Tin *dt, const float *A_head, const Tin *Bm, const Tin *Cm,
                   const float *D, float *y, int64_t Bs, int64_t L, int64_t H, int64_t P,
                   int64_t N, bool bidir, int num_sms, const ScanOpts *opt, cudaStream_t st);
}
namespace bidir {
cudaError_t take_device_error(unsigned int *out);
}
namespace ssd {
cudaError_t launch(const __nv_bfloat16 *x, const __nv_bfloat16 *dt, const float *A_head,
                   const __nv_bfloat16 *Bm, const __nv_bfloat16 *Cm, const float *D, float *y,
                   int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N, int64_t chunk,
                   bool bidirectional, int num_sms, cudaStream_t st, const ScanOpts *opt);
cudaError_t take_device_error(unsigned int *out);
cudaError_t probe_wait_timeout(cudaStream_t st);
size_t noalloc_scratch_needed(int64_t Bs, int64_t L, int64_t H, int64_t N, bool bidirectional);
cudaError_t launch_noalloc(const __nv_bfloat16 *x, const __nv_bfloat16 *dt, const float *A_head,
                           const __nv_bfloat16 *Bm, const __nv_bfloat16 *Cm, const float *D,
                           float *y, int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                           bool bidirectional, cudaStream_t stream);
}
}  // namespace ssm

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ok = false;
    int num_sms = 0;
};

std::mutex g_dev_mutex;
bool g_dev_known[kMaxDevices];   // set only once the attribute queries succeeded
DeviceInfo g_dev[kMaxDevices];

// Device attributes, kept per device once a query has succeeded.  A device that is not
// compute capability 10.3 cannot run this library's sm_103a code.
ssm_status_t current_device(DeviceInfo *out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SSM_ERR_NO_DEVICE;
    }
    {
        // a failed query is not kept: the next call asks again
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        if (!g_dev_known[dev]) {
            int major = 0, minor = 0, sms = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return SSM_ERR_NO_DEVICE;
            g_dev[dev].ok = major == 10 && minor == 3;
            g_dev[dev].num_sms = sms;
            g_dev_known[dev] = true;
        }
        *out = g_dev[dev];
    }
    return out->ok ? SSM_OK : SSM_ERR_NO_DEVICE;
}

bool mul_ok(int64_t a, int64_t b, int64_t *out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

// Every size >= 1 and the product of all of them fits in int64.
bool sizes_ok(std::initializer_list<int64_t> dims) {
    int64_t prod = 1;
    for (int64_t d : dims) {
        if (d < 1) return false;
        if (!mul_ok(prod, d, &prod)) return false;
    }
    return true;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ssm_status_t from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return SSM_OK;
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorNoDevice ||
        e == cudaErrorInsufficientDriver)
        return SSM_ERR_NO_DEVICE;
    if (e == cudaErrorInvalidConfiguration) return SSM_ERR_UNSUPPORTED;
    return SSM_ERR_CUDA;
}

// Options present, and their pointers aligned to `zsize` (z) / 4 bytes.
ssm_status_t check_options(const ssm_scan_options_t *o, size_t zsize) {
    if (!o) return SSM_OK;
    if ((o->z && !aligned(o->z, zsize)) || (o->dt_bias && !aligned(o->dt_bias, 4)) ||
        (o->h0 && !aligned(o->h0, 4)) || (o->h_final && !aligned(o->h_final, 4)))
        return SSM_ERR_ALIGNMENT;
    return SSM_OK;
}

template <typename Tin>
ssm_status_t diag_entry(const Tin *x, const Tin *delta, const float *A, const Tin *B, const Tin *C,
                        const float *D, float *y, int64_t Bs, int64_t L, int64_t ED, int64_t N,
                        void *stream, const ssm_scan_options_t *opts = nullptr) {
    if (!x || !delta || !A || !B || !C || !y) return SSM_ERR_INVALID_ARG;
    if (!sizes_ok({Bs, L, ED}) || !sizes_ok({Bs, L, N}) || !sizes_ok({ED, N}))
        return SSM_ERR_INVALID_ARG;
    if (N > 256) return SSM_ERR_UNSUPPORTED;
    if (L > INT_MAX || ED > INT_MAX) return SSM_ERR_UNSUPPORTED;
    const size_t es = sizeof(Tin);
    if (!aligned(x, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) ||
        !aligned(A, 4) || !aligned(y, 4) || (D && !aligned(D, 4)))
        return SSM_ERR_ALIGNMENT;
    if (opts && opts->ngroups > 1) return SSM_ERR_UNSUPPORTED;   // groups: SSD only
    ssm_status_t s = check_options(opts, es);
    if (s != SSM_OK) return s;
    DeviceInfo dev;
    s = current_device(&dev);
    if (s != SSM_OK) return s;
    // the plain kernels unless an option is on
    if (opts && (opts->dt_bias || opts->dt_softplus || opts->dt_limit || opts->z || opts->h0 ||
                 opts->h_final)) {
        const ssm::ScanOpts ex{opts->dt_bias, opts->z, opts->h0, opts->h_final,
                               opts->dt_min, opts->dt_max, opts->dt_softplus, opts->dt_limit, 1};
        return from_cuda(ssm::diag::launch_ext<Tin>(x, delta, A, B, C, D, y, Bs, L, ED, N,
                                                    dev.num_sms, ex,
                                                    static_cast<cudaStream_t>(stream)));
    }
    return from_cuda(ssm::diag::launch<Tin>(x, delta, A, B, C, D, y, Bs, L, ED, N, dev.num_sms,
                                            static_cast<cudaStream_t>(stream)));
}


// The chunked scan: validation, then the tensor-core kernel (bf16, P = 64,
// N in {64, 128}) or the CUDA-core kernel (every other supported shape and
// fp32 inputs).  `noalloc`: the reverse states' scratch comes from the fixed
// module array (the CUDA-core kernel needs none).
ssm_status_t ssd_entry(const void *x, const void *dt, const float *A_head, const void *B,
                       const void *C, const float *D, float *y, int64_t Bs, int64_t L, int64_t H,
                       int64_t P, int64_t N, int64_t chunk, int bidirectional, int input_bf16,
                       const ssm_scan_options_t *opts, void *stream, bool noalloc) {
    if (!x || !dt || !A_head || !B || !C || !y) return SSM_ERR_INVALID_ARG;
    if (!sizes_ok({Bs, L, H, P}) || !sizes_ok({Bs, L, N}) || chunk < 1) return SSM_ERR_INVALID_ARG;
    const bool tc = input_bf16 && P == 64 && (N == 64 || N == 128);
    if (!tc && !ssm::ssd_general::supported(P, N)) return SSM_ERR_UNSUPPORTED;
    if (chunk != 64 && chunk != 128 && chunk != 256) return SSM_ERR_UNSUPPORTED;
    if (L > INT_MAX || H > 65535 || Bs > INT_MAX) return SSM_ERR_UNSUPPORTED;
    if (opts) {
        if (bidirectional && (opts->h0 || opts->h_final)) return SSM_ERR_UNSUPPORTED;
        if (opts->ngroups < 0 || (opts->ngroups > 1 && H % opts->ngroups != 0))
            return SSM_ERR_INVALID_ARG;
        if (opts->ngroups > 1 && !sizes_ok({Bs, L, opts->ngroups, N})) return SSM_ERR_INVALID_ARG;
    }
    if (tc && noalloc &&
        ssm::ssd::noalloc_scratch_needed(Bs, L, H, N, bidirectional != 0) > SSM_NOALLOC_SCRATCH_BYTES)
        return SSM_ERR_UNSUPPORTED;
    const size_t es = input_bf16 ? 2 : 4;
    if (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(y, 16) ||
        !aligned(dt, es) || !aligned(A_head, 4) || (D && !aligned(D, 4)))
        return SSM_ERR_ALIGNMENT;
    ssm_status_t s = check_options(opts, 16);
    if (s != SSM_OK) return s;
    DeviceInfo dev;
    s = current_device(&dev);
    if (s != SSM_OK) return s;
    using bf = __nv_bfloat16;
    ssm::ScanOpts o{};
    if (opts)
        o = ssm::ScanOpts{opts->dt_bias, opts->z, opts->h0, opts->h_final, opts->dt_min,
                          opts->dt_max, opts->dt_softplus, opts->dt_limit, opts->ngroups};
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!tc) {
        if (input_bf16)
            return from_cuda(ssm::ssd_general::launch<bf>(
                static_cast<const bf *>(x), static_cast<const bf *>(dt), A_head,
                static_cast<const bf *>(B), static_cast<const bf *>(C), D, y, Bs, L, H, P, N,
                bidirectional != 0, dev.num_sms, opts ? &o : nullptr, st));
        return from_cuda(ssm::ssd_general::launch<float>(
            static_cast<const float *>(x), static_cast<const float *>(dt), A_head,
            static_cast<const float *>(B), static_cast<const float *>(C), D, y, Bs, L, H, P, N,
            bidirectional != 0, dev.num_sms, opts ? &o : nullptr, st));
    }
    if (noalloc)
        return from_cuda(ssm::ssd::launch_noalloc(static_cast<const bf *>(x),
                                                  static_cast<const bf *>(dt), A_head,
                                                  static_cast<const bf *>(B),
                                                  static_cast<const bf *>(C), D, y, Bs, L, H, P, N,
                                                  bidirectional != 0, st));
    return from_cuda(ssm::ssd::launch(static_cast<const bf *>(x), static_cast<const bf *>(dt),
                                      A_head, static_cast<const bf *>(B),
                                      static_cast<const bf *>(C), D, y, Bs, L, H, P, N, chunk,
                                      bidirectional != 0, dev.num_sms, st, opts ? &o : nullptr));
}
}  // namespace

extern "C" {

ssm_status_t ssm_scan_fwd(const float *x, const float *delta, const float *A, const float *B,
                          const float *C, const float *D, float *y, int64_t Bs, int64_t L,
                          int64_t ED, int64_t N, void *stream) {
    return diag_entry<float>(x, delta, A, B, C, D, y, Bs, L, ED, N, stream);
}

ssm_status_t ssm_scan_fwd_bf16(const void *x, const void *delta, const float *A, const void *B,
                               const void *C, const float *D, float *y, int64_t Bs, int64_t L,
                               int64_t ED, int64_t N, void *stream) {
    using bf = __nv_bfloat16;
    return diag_entry<bf>(static_cast<const bf *>(x), static_cast<const bf *>(delta), A,
                          static_cast<const bf *>(B), static_cast<const bf *>(C), D, y, Bs, L, ED,
                          N, stream);
}

ssm_status_t ssd_chunk_scan_fwd(const void *x, const void *dt, const float *A_head, const void *B,
                                const void *C, const float *D, float *y, int64_t Bs, int64_t L,
                                int64_t H, int64_t P, int64_t N, int64_t chunk, int bidirectional,
                                void *stream) {
    return ssd_entry(x, dt, A_head, B, C, D, y, Bs, L, H, P, N, chunk, bidirectional, 1, nullptr,
                     stream, false);
}

ssm_status_t ssd_chunk_scan_fwd_noalloc(const void *x, const void *dt, const float *A_head,
                                        const void *B, const void *C, const float *D, float *y,
                                        int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                                        int64_t chunk, int bidirectional, void *stream) {
    return ssd_entry(x, dt, A_head, B, C, D, y, Bs, L, H, P, N, chunk, bidirectional, 1, nullptr,
                     stream, true);
}

ssm_status_t ssm_scan_fwd_ex(const void *x, const void *delta, const float *A, const void *B,
                             const void *C, const float *D, float *y, int64_t Bs, int64_t L,
                             int64_t ED, int64_t N, int input_bf16,
                             const ssm_scan_options_t *opts, void *stream) {
    using bf = __nv_bfloat16;
    if (input_bf16)
        return diag_entry<bf>(static_cast<const bf *>(x), static_cast<const bf *>(delta), A,
                              static_cast<const bf *>(B), static_cast<const bf *>(C), D, y, Bs, L,
                              ED, N, stream, opts);
    return diag_entry<float>(static_cast<const float *>(x), static_cast<const float *>(delta), A,
                             static_cast<const float *>(B), static_cast<const float *>(C), D, y, Bs,
                             L, ED, N, stream, opts);
}

ssm_status_t ssd_chunk_scan_fwd_ex(const void *x, const void *dt, const float *A_head,
                                   const void *B, const void *C, const float *D, float *y,
                                   int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                                   int64_t chunk, int bidirectional, int input_bf16,
                                   const ssm_scan_options_t *opts, void *stream) {
    return ssd_entry(x, dt, A_head, B, C, D, y, Bs, L, H, P, N, chunk, bidirectional, input_bf16,
                     opts, stream, false);
}

ssm_status_t ssm_scan_bwd(const void *x, const void *delta, const float *A, const void *B,
                          const void *C, const float *D, const float *dy, float *dx,
                          float *ddelta, float *dA, float *dB, float *dC, float *dD, int64_t Bs,
                          int64_t L, int64_t ED, int64_t N, int input_bf16, void *stream) {
    if (!x || !delta || !A || !B || !C || !dy || !dx || !ddelta || !dA || !dB || !dC)
        return SSM_ERR_INVALID_ARG;
    if (!sizes_ok({Bs, L, ED}) || !sizes_ok({Bs, L, N}) || !sizes_ok({ED, N}))
        return SSM_ERR_INVALID_ARG;
    if (N > 256 || Bs > 65535 || L > INT_MAX || ED > INT_MAX) return SSM_ERR_UNSUPPORTED;
    const size_t es = input_bf16 ? 2 : 4;
    if (!aligned(x, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) ||
        !aligned(A, 4) || (D && !aligned(D, 4)) || !aligned(dy, 4) || !aligned(dx, 4) ||
        !aligned(ddelta, 4) || !aligned(dA, 4) || !aligned(dB, 4) || !aligned(dC, 4) ||
        (dD && !aligned(dD, 4)))
        return SSM_ERR_ALIGNMENT;
    DeviceInfo dev;
    ssm_status_t s = current_device(&dev);
    if (s != SSM_OK) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    using bf = __nv_bfloat16;
    if (input_bf16)
        return from_cuda(ssm::diag_bwd::launch_bwd<bf>(
            static_cast<const bf *>(x), static_cast<const bf *>(delta), A,
            static_cast<const bf *>(B), static_cast<const bf *>(C), D, dy, dx, ddelta, dA, dB, dC,
            dD, Bs, L, ED, N, dev.num_sms, st));
    return from_cuda(ssm::diag_bwd::launch_bwd<float>(
        static_cast<const float *>(x), static_cast<const float *>(delta), A,
        static_cast<const float *>(B), static_cast<const float *>(C), D, dy, dx, ddelta, dA, dB,
        dC, dD, Bs, L, ED, N, dev.num_sms, st));
}

ssm_status_t ssm_scan_bwd_ex(const void *x, const void *delta, const float *A, const void *B,
                             const void *C, const float *D, const float *dy, float *dx,
                             float *ddelta, float *dA, float *dB, float *dC, float *dD, float *dz,
                             float *ddt_bias, float *dh0, int64_t Bs, int64_t L, int64_t ED,
                             int64_t N, int input_bf16, const ssm_scan_options_t *opts,
                             void *stream) {
    if (!x || !delta || !A || !B || !C || !dy || !dx || !ddelta || !dA || !dB || !dC)
        return SSM_ERR_INVALID_ARG;
    if (!sizes_ok({Bs, L, ED}) || !sizes_ok({Bs, L, N}) || !sizes_ok({ED, N}))
        return SSM_ERR_INVALID_ARG;
    if (opts && opts->h_final) return SSM_ERR_INVALID_ARG;       // an output of the forward only
    if (opts && opts->z && !dz) return SSM_ERR_INVALID_ARG;
    if (opts && opts->ngroups > 1) return SSM_ERR_UNSUPPORTED;  // groups: SSD only
    if (N > 256 || Bs > 65535 || L > INT_MAX || ED > INT_MAX) return SSM_ERR_UNSUPPORTED;
    const size_t es = input_bf16 ? 2 : 4;
    if (!aligned(x, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) ||
        !aligned(A, 4) || (D && !aligned(D, 4)) || !aligned(dy, 4) || !aligned(dx, 4) ||
        !aligned(ddelta, 4) || !aligned(dA, 4) || !aligned(dB, 4) || !aligned(dC, 4) ||
        (dD && !aligned(dD, 4)) || (dz && !aligned(dz, 4)) || (ddt_bias && !aligned(ddt_bias, 4)) ||
        (dh0 && !aligned(dh0, 4)))
        return SSM_ERR_ALIGNMENT;
    ssm_status_t s = check_options(opts, es);
    if (s != SSM_OK) return s;
    DeviceInfo dev;
    s = current_device(&dev);
    if (s != SSM_OK) return s;
    ssm::ScanOpts o{};
    if (opts)
        o = ssm::ScanOpts{opts->dt_bias, opts->z, opts->h0, nullptr, opts->dt_min,
                          opts->dt_max, opts->dt_softplus, opts->dt_limit, 1};
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    using bf = __nv_bfloat16;
    float *dzo = o.z ? dz : nullptr;
    float *dbo = o.dt_bias ? ddt_bias : nullptr;
    float *dho = o.h0 ? dh0 : nullptr;
    if (input_bf16)
        return from_cuda(ssm::diag_bwd_ex::launch<bf>(
            static_cast<const bf *>(x), static_cast<const bf *>(delta), A,
            static_cast<const bf *>(B), static_cast<const bf *>(C), D, dy, dx, ddelta, dA, dB, dC,
            dD, dzo, dbo, dho, Bs, L, ED, N, o, dev.num_sms, st));
    return from_cuda(ssm::diag_bwd_ex::launch<float>(
        static_cast<const float *>(x), static_cast<const float *>(delta), A,
        static_cast<const float *>(B), static_cast<const float *>(C), D, dy, dx, ddelta, dA, dB,
        dC, dD, dzo, dbo, dho, Bs, L, ED, N, o, dev.num_sms, st));
}

ssm_status_t ssd_chunk_scan_bwd(const void *x, const void *dt, const float *A_head, const void *B,
                                const void *C, const float *D, const float *dy, float *dx,
                                float *ddt, float *dA_head, float *dB, float *dC, float *dD,
                                int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                                int64_t ngroups, int bidirectional, int input_bf16, void *stream) {
    if (!x || !dt || !A_head || !B || !C || !dy || !dx || !ddt || !dA_head || !dB || !dC)
        return SSM_ERR_INVALID_ARG;
    if (ngroups < 1 || !sizes_ok({Bs, L, H, P}) || !sizes_ok({Bs, L, ngroups, N}) ||
        !sizes_ok({Bs, H, L, P, N}))
        return SSM_ERR_INVALID_ARG;
    if (!ssm::ssd_bwd::supported(P, N) || H % ngroups != 0 || Bs * H > INT_MAX || L > INT_MAX)
        return SSM_ERR_UNSUPPORTED;
    const size_t es = input_bf16 ? 2 : 4;
    if (!aligned(x, es) || !aligned(dt, es) || !aligned(B, es) || !aligned(C, es) ||
        !aligned(A_head, 4) || (D && !aligned(D, 4)) || !aligned(dy, 4) || !aligned(dx, 4) ||
        !aligned(ddt, 4) || !aligned(dA_head, 4) || !aligned(dB, 4) || !aligned(dC, 4) ||
        (dD && !aligned(dD, 4)))
        return SSM_ERR_ALIGNMENT;
    DeviceInfo dev;
    ssm_status_t s = current_device(&dev);
    if (s != SSM_OK) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    using bf = __nv_bfloat16;
    if (input_bf16)
        return from_cuda(ssm::ssd_bwd::launch<bf>(
            static_cast<const bf *>(x), static_cast<const bf *>(dt), A_head,
            static_cast<const bf *>(B), static_cast<const bf *>(C), D, dy, dx, ddt, dA_head, dB,
            dC, dD, Bs, L, H, P, N, ngroups, bidirectional != 0, st));
    return from_cuda(ssm::ssd_bwd::launch<float>(
        static_cast<const float *>(x), static_cast<const float *>(dt), A_head,
        static_cast<const float *>(B), static_cast<const float *>(C), D, dy, dx, ddt, dA_head, dB,
        dC, dD, Bs, L, H, P, N, ngroups, bidirectional != 0, st));
}

ssm_status_t ssd_chunk_scan_bwd_ex(const void *x, const void *dt, const float *A_head,
                                   const void *B, const void *C, const float *D, const float *dy,
                                   float *dx, float *ddt, float *dA_head, float *dB, float *dC,
                                   float *dD, float *dz, float *ddt_bias, float *dh0, int64_t Bs,
                                   int64_t L, int64_t H, int64_t P, int64_t N, int bidirectional,
                                   int input_bf16, const ssm_scan_options_t *opts, void *stream) {
    if (!x || !dt || !A_head || !B || !C || !dy || !dx || !ddt || !dA_head || !dB || !dC)
        return SSM_ERR_INVALID_ARG;
    const int64_t G = (opts && opts->ngroups > 1) ? opts->ngroups : 1;
    if ((opts && opts->ngroups < 0) || !sizes_ok({Bs, L, H, P}) || !sizes_ok({Bs, L, G, N}) ||
        !sizes_ok({Bs, H, L, P, N}))
        return SSM_ERR_INVALID_ARG;
    if (opts && opts->h_final) return SSM_ERR_INVALID_ARG;       // an output of the forward only
    if (opts && opts->z && !dz) return SSM_ERR_INVALID_ARG;
    if (bidirectional && opts && opts->h0) return SSM_ERR_UNSUPPORTED;
    if (!ssm::ssd_bwd::supported(P, N) || H % G != 0 || Bs * H > INT_MAX || L > INT_MAX)
        return SSM_ERR_UNSUPPORTED;
    const size_t es = input_bf16 ? 2 : 4;
    if (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(dt, es) ||
        !aligned(A_head, 4) || (D && !aligned(D, 4)) || !aligned(dy, 4) || !aligned(dx, 4) ||
        !aligned(ddt, 4) || !aligned(dA_head, 4) || !aligned(dB, 4) || !aligned(dC, 4) ||
        (dD && !aligned(dD, 4)) || (dz && !aligned(dz, 4)) || (ddt_bias && !aligned(ddt_bias, 4)) ||
        (dh0 && !aligned(dh0, 4)))
        return SSM_ERR_ALIGNMENT;
    ssm_status_t s = check_options(opts, es);
    if (s != SSM_OK) return s;
    DeviceInfo dev;
    s = current_device(&dev);
    if (s != SSM_OK) return s;
    ssm::ScanOpts o{};
    if (opts)
        o = ssm::ScanOpts{opts->dt_bias, opts->z, opts->h0, nullptr, opts->dt_min,
                          opts->dt_max, opts->dt_softplus, opts->dt_limit, opts->ngroups};
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    using bf = __nv_bfloat16;
    float *dzo = o.z ? dz : nullptr;
    float *dbo = o.dt_bias ? ddt_bias : nullptr;
    float *dho = o.h0 ? dh0 : nullptr;
    if (input_bf16)
        return from_cuda(ssm::ssd_bwd_ex::launch<bf>(
            static_cast<const bf *>(x), static_cast<const bf *>(dt), A_head,
            static_cast<const bf *>(B), static_cast<const bf *>(C), D, dy, dx, ddt, dA_head, dB, dC,
            dD, dzo, dbo, dho, Bs, L, H, P, N, G, bidirectional != 0, o, dev.num_sms, st));
    return from_cuda(ssm::ssd_bwd_ex::launch<float>(
        static_cast<const float *>(x), static_cast<const float *>(dt), A_head,
        static_cast<const float *>(B), static_cast<const float *>(C), D, dy, dx, ddt, dA_head, dB,
        dC, dD, dzo, dbo, dho, Bs, L, H, P, N, G, bidirectional != 0, o, dev.num_sms, st));
}

ssm_status_t ssm_scan_fwd_plan(int64_t Bs, int64_t L, int64_t ED, int64_t N, int input_bf16,
                               int32_t *states_per_thread, int32_t *lanes_per_channel,
                               int32_t *time_segments) {
    if (!states_per_thread || !lanes_per_channel || !time_segments) return SSM_ERR_INVALID_ARG;
    if (!sizes_ok({Bs, L, ED}) || !sizes_ok({Bs, L, N}) || !sizes_ok({ED, N}))
        return SSM_ERR_INVALID_ARG;
    if (N > 256) return SSM_ERR_UNSUPPORTED;
    if (L > INT_MAX || ED > INT_MAX) return SSM_ERR_UNSUPPORTED;
    DeviceInfo dev;
    ssm_status_t s = current_device(&dev);
    if (s != SSM_OK) return s;
    const ssm::diag::Plan p = ssm::diag::plan_for(Bs, L, ED, N, input_bf16 ? 2 : 4, dev.num_sms);
    *states_per_thread = p.S;
    *lanes_per_channel = p.G;
    *time_segments = p.K;
    return SSM_OK;
}

ssm_status_t ssm_check_device_errors(void *stream) {
    DeviceInfo dev;
    ssm_status_t s = current_device(&dev);
    if (s != SSM_OK) return s;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SSM_ERR_CUDA;
    unsigned int flag = 0, flag_bi = 0;
    if (ssm::ssd::take_device_error(&flag) != cudaSuccess) return SSM_ERR_CUDA;
    if (ssm::bidir::take_device_error(&flag_bi) != cudaSuccess) return SSM_ERR_CUDA;
    return (flag | flag_bi) ? SSM_ERR_DEVICE_TIMEOUT : SSM_OK;
}

ssm_status_t ssm_selftest_wait_timeout(void *stream) {
    DeviceInfo dev;
    ssm_status_t s = current_device(&dev);
    if (s != SSM_OK) return s;
    return from_cuda(ssm::ssd::probe_wait_timeout(static_cast<cudaStream_t>(stream)));
}

const char *ssm_status_string(ssm_status_t status) {
    switch (status) {
        case SSM_OK: return "SSM_OK";
        case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG: null pointer or size < 1 / overflow";
        case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED: size outside the supported set";
        case SSM_ERR_ALIGNMENT: return "SSM_ERR_ALIGNMENT: pointer not aligned as required";
        case SSM_ERR_CUDA: return "SSM_ERR_CUDA: a CUDA call or kernel launch failed";
        case SSM_ERR_DEVICE_TIMEOUT: return "SSM_ERR_DEVICE_TIMEOUT: a bounded device wait ran out";
        case SSM_ERR_NO_DEVICE: return "SSM_ERR_NO_DEVICE: no sm_103 CUDA device is current";
    }
    return "unknown ssm_status_t";
}

int ssm_version(void) { return 100; }

}  // extern "C"
