/*
 * ssm_scan.h -- C ABI of the GB300 (sm_103a) selective-scan library
 * (libssmscan.so).
 *
 * The library computes the forward linear recurrence at the core of
 * Mamba-style state-space layers, in two forms:
 *
 *   ssm_scan_fwd / ssm_scan_fwd_bf16  -- diagonal A (one decay per channel
 *       and state).  Shape API of selective_scan / selective_scan_seq in
 *       "scan output is different between sequential and parallel
 *       versions" (mamba.py issue 26, the test script's comment block):
 *       x, delta (Bs, L, ED); A (ED, N); B, C (Bs, L, N); D (ED);
 *       y (Bs, L, ED).  Per channel (b, e) and state n, with h_{-1} = 0:
 *         h_t[n] = exp(delta_t * A[e,n]) * h_{t-1}[n] + delta_t * B_t[n] * x_t
 *         y_t    = sum_n C_t[n] * h_t[n] + D[e] * x_t
 *
 *   ssd_chunk_scan_fwd  -- one scalar decay per head (chunked "SSD" form),
 *       argument subset (x, dt, A, B, C, chunk_size, D) of the chunked scan
 *       in "Some questions of Bi-Mamba2 and Hydra" (Bi-Mamba2 issue 1, the
 *       MambaChunkScanCombinedFn.forward signature), with z, dt_bias and
 *       dt_softplus off and one group of B, C shared by all heads (the
 *       _ex entry points below add those options and state I/O).
 *       x (Bs, L, H, P); dt (Bs, L, H); A_head (H); B, C (Bs, L, N) -- the
 *       same memory as (Bs, L, 1, N); D (H); y (Bs, L, H, P).  Per (b, h):
 *         H_t = exp(dt_t * A_h) * H_{t-1} + dt_t * x_t (outer) B_t   (P x N)
 *         y_t = H_t C_t + D_h * x_t
 *       With bidirectional != 0 the reversed scan (same x, dt, A, B, C, the
 *       time axis walked from the end) is added, and D x once: the page
 *       describes Bi-Mamba2 as the sum of two SSMs with shared weights plus
 *       the skip term.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, dense
 *     row-major with the last index fastest.  Inputs are only read; y is
 *     fully overwritten (never accumulated into).  The library keeps no
 *     pointer after the call returns.
 *   - A, A_head and D are fp32.  D may be NULL (read as D = 0).  y is fp32.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work
 *     is enqueued on it and the call never synchronises; faults raised by
 *     the kernels surface at the caller's next synchronisation.
 *   - Errors are returned as ssm_status_t; nothing is launched when the
 *     status is not SSM_OK.  No entry point aborts or throws.
 *   - Calls are reentrant and thread-safe; the only global state is a
 *     per-device cache of attributes.
 *   - Sizes are int64; every size must be >= 1 and every tensor's element
 *     count must fit in int64.
 *   - Results are deterministic: the same inputs give bitwise-equal y.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,     /* NULL pointer, size < 1, size overflow */
    SSM_ERR_UNSUPPORTED = 2,     /* a size outside what the kernels handle */
    SSM_ERR_ALIGNMENT = 3,       /* a pointer not aligned to its element size */
    SSM_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed */
    SSM_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device wait ran out (see ssm_check_device_errors) */
    SSM_ERR_NO_DEVICE = 6        /* no CUDA device, or not an sm_103 device */
} ssm_status_t;

/*
 * Diagonal selective scan, fp32 x / delta / B / C.
 *   x, delta : (Bs, L, ED) fp32        A : (ED, N) fp32
 *   B, C     : (Bs, L, N)  fp32        D : (ED) fp32 or NULL
 *   y        : (Bs, L, ED) fp32 output
 * Supported: 1 <= N <= 256.  Every pointer must be 4-byte aligned
 * (SSM_ERR_ALIGNMENT otherwise).  Any Bs, L, ED >= 1.
 */
SSM_API ssm_status_t ssm_scan_fwd(const float *x, const float *delta, const float *A,
                          const float *B, const float *C, const float *D,
                          float *y, int64_t Bs, int64_t L, int64_t ED,
                          int64_t N, void *stream);

/*
 * Diagonal selective scan, bf16 x / delta / B / C (passed as raw 16-bit
 * bfloat16 storage); A, D fp32; state and y fp32.  Same shapes and rules as
 * ssm_scan_fwd; x, delta, B, C must be 2-byte aligned.
 */
SSM_API ssm_status_t ssm_scan_fwd_bf16(const void *x, const void *delta,
                               const float *A, const void *B, const void *C,
                               const float *D, float *y, int64_t Bs,
                               int64_t L, int64_t ED, int64_t N,
                               void *stream);

/*
 * How ssm_scan_fwd / ssm_scan_fwd_bf16 (input_bf16 != 0) decompose a shape
 * on the current device: states held per thread, lanes sharing a channel, and
 * the number of time segments scanned in parallel.  With time_segments > 1 a
 * call launches two kernels (the segments, then a pass that carries each
 * segment's entering state into its first outputs) and takes stream-ordered
 * scratch of time_segments*Bs*ED*18*4 bytes; otherwise one kernel and no
 * scratch.  Same argument rules as ssm_scan_fwd; output pointers must be
 * non-NULL.
 */
SSM_API ssm_status_t ssm_scan_fwd_plan(int64_t Bs, int64_t L, int64_t ED,
                                       int64_t N, int input_bf16,
                                       int32_t *states_per_thread,
                                       int32_t *lanes_per_channel,
                                       int32_t *time_segments);

/*
 * Chunked scalar-decay (SSD) scan, bf16 x / dt / B / C (raw bfloat16
 * storage), fp32 A_head, D, state and y.
 *   x  : (Bs, L, H, P) bf16        dt : (Bs, L, H) bf16
 *   A_head : (H) fp32              B, C : (Bs, L, N) bf16 (one group)
 *   D  : (H) fp32 or NULL          y  : (Bs, L, H, P) fp32 output
 *   chunk : time-chunk length Q of the chunked algorithm.
 *   bidirectional : 0 = forward scan; != 0 = forward + reversed scan + D x.
 * Supported: P and N in {16, 32, 64, 128, 256}; chunk in {64, 128, 256};
 * any Bs, L, H >= 1 (L need not be
 * a multiple of chunk).  x, B, C and y must be 16-byte aligned, dt aligned
 * to its element size (SSM_ERR_ALIGNMENT otherwise).  bf16 inputs with
 * P == 64 and N in {64, 128} run on the tensor cores (tcgen05); every other
 * supported shape, and fp32 inputs (ssd_chunk_scan_fwd_ex), on CUDA cores.
 * The chunked result equals the recurrence for every chunk length (up to
 * rounding).  The tensor-core kernel passes the state between 128-row tiles
 * -- the tensor-core tile height -- so a chunk of 256 rows is computed as
 * two 128-row tiles and a chunk of 64 as half of one; `chunk` is validated
 * and does not change the result beyond rounding.
 * Bidirectional calls of the tensor-core kernel with L > 128 take a
 * stream-ordered scratch buffer of Bs*H*ceil(L/128)*P*N*2 bytes
 * (cudaMallocAsync / cudaFreeAsync on `stream`) for the reverse scan's
 * entering states; the CUDA-core kernel needs none.
 */
SSM_API ssm_status_t ssd_chunk_scan_fwd(const void *x, const void *dt,
                                const float *A_head, const void *B,
                                const void *C, const float *D, float *y,
                                int64_t Bs, int64_t L, int64_t H, int64_t P,
                                int64_t N, int64_t chunk, int bidirectional,
                                void *stream);

/*
 * Same computation, arguments and rules as ssd_chunk_scan_fwd, for callers
 * that cannot allocate device memory -- code running where cudaMalloc and
 * stream-ordered allocation are unavailable or forbidden (a custom
 * allocator owns all device memory, or the call sits in a region that must
 * not touch the memory pool).  It allocates nothing and calls no
 * allocating routine: the scratch that bidirectional calls need for the
 * reverse scan's entering states lives in one fixed array inside the
 * library, SSM_NOALLOC_SCRATCH_BYTES long, which every GPU that loads the
 * library holds until the process exits.  The pages have no counterpart to
 * this entry point; it exists for such callers only.
 *   - Calls needing more than SSM_NOALLOC_SCRATCH_BYTES of scratch, i.e.
 *     bidirectional with Bs*H*ceil(L/128)*P*N*2 > SSM_NOALLOC_SCRATCH_BYTES,
 *     return SSM_ERR_UNSUPPORTED and launch nothing.  Unidirectional calls
 *     need no scratch.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it once the lookup succeeds; make
 *     that first call before any stream capture.  A lookup that fails
 *     returns SSM_ERR_CUDA, caches nothing, and the next call tries again.
 *   - Every call shares the one array: calls that overlap on the GPU (on
 *     different streams, or from different threads) race and give wrong
 *     results.  The array keeps the last call's contents; no call depends
 *     on it starting at zero.
 */
#define SSM_NOALLOC_SCRATCH_BYTES (16ull << 20)
SSM_API ssm_status_t ssd_chunk_scan_fwd_noalloc(const void *x, const void *dt,
                                        const float *A_head, const void *B,
                                        const void *C, const float *D, float *y,
                                        int64_t Bs, int64_t L, int64_t H, int64_t P,
                                        int64_t N, int64_t chunk, int bidirectional,
                                        void *stream);

/*
 * Options of the scans: the remaining arguments of the chunked scan's
 * argument list in "Some questions of Bi-Mamba2 and Hydra" (Bi-Mamba2
 * issue 1, MambaChunkScanCombinedFn.forward: dt_bias, dt_softplus,
 * dt_limit, z, initial and returned final states), read the Mamba way.
 * A zero-initialised structure means no option.  Applied in this order:
 *   delta <- delta + dt_bias[channel]          if dt_bias != NULL
 *   delta <- log(1 + exp(delta))               if dt_softplus != 0
 *   delta <- min(max(delta, dt_min), dt_max)   if dt_limit != 0
 *   (the scan, from h_{-1} = h0 when h0 != NULL, else 0)
 *   y     <- (scan + D x) * z / (1 + exp(-z))  if z != NULL   (silu gate)
 *   h_final <- the state after the last step   if h_final != NULL
 * "channel" is e for the diagonal scan and the head h for SSD.
 *   dt_bias : fp32, (ED) or (H)
 *   z       : same shape and element type as x (fp32 or bf16)
 *   h0, h_final : fp32 device arrays, (Bs, ED, N) for the diagonal scan,
 *             (Bs, H, P, N) for SSD (state matrix per head: row p, column
 *             n); caller-owned; h_final is fully written.
 *   ngroups : SSD only -- B and C have shape (Bs, L, ngroups, N) and head h
 *             reads group h / (H / ngroups) (ngroups must divide H, else
 *             SSM_ERR_INVALID_ARG); 0 or 1 = one group shared by all heads.
 *             The diagonal scan returns SSM_ERR_UNSUPPORTED for ngroups > 1.
 * State input/output belongs to a single direction: ssd_chunk_scan_fwd_ex
 * with bidirectional != 0 and h0 or h_final set returns
 * SSM_ERR_UNSUPPORTED.
 */
typedef struct ssm_scan_options {
    const float *dt_bias;
    int32_t dt_softplus;
    int32_t dt_limit;
    float dt_min;
    float dt_max;
    const void *z;
    const float *h0;
    float *h_final;
    int32_t ngroups;
} ssm_scan_options_t;

/*
 * ssm_scan_fwd / ssm_scan_fwd_bf16 with options.  input_bf16 selects the
 * element type of x, delta, B, C and z (0 = fp32, else bf16); `opts` may be
 * NULL (no option).  Alignment: x, delta, B, C, z to their element size;
 * dt_bias, h0, h_final to 4 bytes (SSM_ERR_ALIGNMENT otherwise).
 */
SSM_API ssm_status_t ssm_scan_fwd_ex(const void *x, const void *delta, const float *A,
                                     const void *B, const void *C, const float *D,
                                     float *y, int64_t Bs, int64_t L, int64_t ED,
                                     int64_t N, int input_bf16,
                                     const ssm_scan_options_t *opts, void *stream);

/*
 * ssd_chunk_scan_fwd with options and a choice of input type: input_bf16
 * selects the element type of x, dt, B, C and z (0 = fp32, else bf16).
 * Same arguments, support and scratch rules otherwise; z is 16-byte aligned;
 * `opts` may be NULL.
 */
SSM_API ssm_status_t ssd_chunk_scan_fwd_ex(const void *x, const void *dt,
                                           const float *A_head, const void *B,
                                           const void *C, const float *D, float *y,
                                           int64_t Bs, int64_t L, int64_t H, int64_t P,
                                           int64_t N, int64_t chunk, int bidirectional,
                                           int input_bf16, const ssm_scan_options_t *opts,
                                           void *stream);

/*
 * Gradients of the diagonal scan (ssm_scan_fwd without options): given dy,
 * the gradient of a loss with respect to y, writes the gradients with
 * respect to every input (the backward pass of the chunked scan's function
 * in "Some questions of Bi-Mamba2 and Hydra", Bi-Mamba2 issue 1, for the
 * diagonal form):
 *   dx, ddelta : (Bs, L, ED) fp32, overwritten
 *   dA         : (ED, N) fp32,  dB, dC : (Bs, L, N) fp32,  dD : (ED) fp32
 *                (zeroed by the call, then accumulated; dD may be NULL)
 * x, delta, B, C are fp32 (input_bf16 == 0) or bf16; A, D, dy are fp32.
 * Supported: N <= 256 (SSM_ERR_UNSUPPORTED otherwise), Bs <= 65535.  More
 * than 16 states are taken in groups of 16 (the recurrence is separate per
 * state): one gradient pass per group, dx and ddelta summed over the groups.
 * dx and ddelta are deterministic; dA, dB, dC, dD are sums formed with
 * atomic additions, so their last bits may differ between runs.  Takes a
 * stream-ordered scratch buffer of ceil(L/16)*Bs*ED*64 bytes for the
 * re-computation checkpoints, and for N > 16 another of about
 * (2 Bs L ED + 2 Bs L 16 + 2 ED 16) * 4 + 2 Bs L 16 * elem bytes for one
 * group's columns and its dx, ddelta.
 * Alignment: every pointer to its element size; dy, dx, ddelta, dA, dB, dC,
 * dD to 4 bytes.
 */
SSM_API ssm_status_t ssm_scan_bwd(const void *x, const void *delta, const float *A,
                                  const void *B, const void *C, const float *D,
                                  const float *dy, float *dx, float *ddelta, float *dA,
                                  float *dB, float *dC, float *dD, int64_t Bs, int64_t L,
                                  int64_t ED, int64_t N, int input_bf16, void *stream);

/*
 * Gradients of the diagonal scan with its options (the scan of
 * ssm_scan_fwd_ex): besides the outputs of ssm_scan_bwd,
 *   dz       : (Bs, L, ED) fp32, overwritten -- required when opts->z is set
 *   ddt_bias : (ED) fp32, overwritten when opts->dt_bias is set (may be NULL)
 *   dh0      : (Bs, ED, N) fp32, overwritten when opts->h0 is set (may be NULL)
 * delta is given before the options (bias, softplus, clamp) and ddelta is the
 * gradient with respect to it (0 where the clamp is active); the chain rule
 * as for ssd_chunk_scan_bwd_ex, per channel.  opts->h_final must be NULL
 * (SSM_ERR_INVALID_ARG); groups are an SSD option (SSM_ERR_UNSUPPORTED).
 * Support and the remaining rules as ssm_scan_bwd (N <= 256).  Computed on
 * CUDA cores by composition: the options' elementwise steps, the forward scan
 * without z (for the ungated output), the plain gradients and one kernel for
 * the terms of h0; bf16 inputs are widened to fp32 first.  Takes
 * stream-ordered scratch of about (2 + [bf16] 1 + [z] 2 + [h0] 1) Bs L ED * 4
 * (+ [bf16] 2 Bs L N * 4) bytes besides that of ssm_scan_bwd.  ddt_bias is
 * summed in a fixed order; dA, dB, dC, dD are formed with atomic additions.
 */
SSM_API ssm_status_t ssm_scan_bwd_ex(const void *x, const void *delta, const float *A,
                                     const void *B, const void *C, const float *D,
                                     const float *dy, float *dx, float *ddelta, float *dA,
                                     float *dB, float *dC, float *dD, float *dz,
                                     float *ddt_bias, float *dh0, int64_t Bs, int64_t L,
                                     int64_t ED, int64_t N, int input_bf16,
                                     const ssm_scan_options_t *opts, void *stream);

/*
 * Gradients of the chunked scalar-decay scan (ssd_chunk_scan_fwd_ex without
 * options; unidirectional or bidirectional, groups of B, C): given dy, the
 * gradient of a loss with respect to y, writes the gradients with respect to
 * every input -- the outputs of the chunked backward pass named in "Some
 * questions of Bi-Mamba2 and Hydra" (Bi-Mamba2 issue 1):
 *   dx      : (Bs, L, H, P) fp32,  ddt : (Bs, L, H) fp32, overwritten
 *   dA_head : (H) fp32,  dB, dC : (Bs, L, G, N) fp32,  dD : (H) fp32
 *             (zeroed by the call, then accumulated; dD may be NULL)
 * x, dt, B, C are fp32 (input_bf16 == 0) or bf16; A_head, D, dy are fp32;
 * B, C are (Bs, L, G, N) with G = ngroups dividing H (head h reads group
 * h / (H / G)).  Supported (SSM_ERR_UNSUPPORTED otherwise): P in {16, 32,
 * 64, 128}, N in {32, 64, 128, 256}, P * N <= 8192.  Computed on CUDA cores
 * from the recurrence step by step (a correctness path, not tuned): takes a
 * stream-ordered scratch buffer of Bs*H*L*P*N*4 bytes (every state of one
 * direction).  dx and ddt are deterministic; dA_head, dB, dC, dD are sums
 * formed with atomic additions, so their last bits may differ between runs.
 * Alignment: every pointer to its element size.
 */
SSM_API ssm_status_t ssd_chunk_scan_bwd(const void *x, const void *dt, const float *A_head,
                                        const void *B, const void *C, const float *D,
                                        const float *dy, float *dx, float *ddt, float *dA_head,
                                        float *dB, float *dC, float *dD, int64_t Bs, int64_t L,
                                        int64_t H, int64_t P, int64_t N, int64_t ngroups,
                                        int bidirectional, int input_bf16, void *stream);

/*
 * Gradients of the chunked scalar-decay scan with its options (the scan of
 * ssd_chunk_scan_fwd_ex): besides the outputs of ssd_chunk_scan_bwd, the
 * gradients the chunked backward of "Some questions of Bi-Mamba2 and Hydra"
 * (Bi-Mamba2 issue 1) returns for its options:
 *   dz       : (Bs, L, H, P) fp32, overwritten -- required when opts->z is set
 *   ddt_bias : (H) fp32, overwritten when opts->dt_bias is set (may be NULL)
 *   dh0      : (Bs, H, P, N) fp32, overwritten when opts->h0 is set (may be NULL)
 * dt is given before the options (bias, softplus, clamp) and ddt is the
 * gradient with respect to it; where the clamp is active ddt is 0.  With
 * v = dt + dt_bias, s = softplus(v) (or v), dte = clamp(s) (or s),
 * u = scan(dte) + D x and y = u silu(z): dz = dy u silu'(z), the scan's
 * gradients are taken for dy silu(z) from h0, and ddt = d dte [lo <= s <= hi]
 * sig(v).  opts->ngroups gives the groups of B, C; opts->h_final must be NULL
 * (SSM_ERR_INVALID_ARG); h0 with the bidirectional scan: SSM_ERR_UNSUPPORTED.
 * Support and the remaining rules as ssd_chunk_scan_bwd; x, B, C must be
 * 16-byte aligned, z aligned to its element size.  Computed on CUDA cores by
 * composition: the options' elementwise steps, the forward scan without z
 * (for u), the plain gradients and one kernel for the terms of h0; bf16
 * inputs are widened to fp32 first.  Takes stream-ordered scratch of about
 * (2 Bs L H + [bf16] Bs L H P + 2 Bs L G N + [z] 2 Bs L H P + [h0] Bs H L) * 4
 * bytes besides that of ssd_chunk_scan_bwd.  ddt_bias is summed in a fixed
 * order; dA_head, dB, dC, dD are formed with atomic additions.
 */
SSM_API ssm_status_t ssd_chunk_scan_bwd_ex(const void *x, const void *dt, const float *A_head,
                                           const void *B, const void *C, const float *D,
                                           const float *dy, float *dx, float *ddt,
                                           float *dA_head, float *dB, float *dC, float *dD,
                                           float *dz, float *ddt_bias, float *dh0, int64_t Bs,
                                           int64_t L, int64_t H, int64_t P, int64_t N,
                                           int bidirectional, int input_bf16,
                                           const ssm_scan_options_t *opts, void *stream);

/*
 * Synchronise `stream` and report whether a kernel of this library running on
 * the current device gave up a bounded wait (SSM_ERR_DEVICE_TIMEOUT) since
 * the previous check; the record is cleared by the call.  Kernels never hang
 * or trap: a wait that runs out abandons the kernel's work (y is then
 * unspecified) and is reported here.  Also returns SSM_ERR_CUDA if the
 * stream holds an earlier asynchronous CUDA error.
 */
SSM_API ssm_status_t ssm_check_device_errors(void *stream);

/*
 * Self-test of the timeout path: enqueues on `stream` a one-thread kernel
 * whose bounded mbarrier wait (the kernels' own wait, 20 ms limit) cannot
 * complete; it gives up and records the timeout, so the next
 * ssm_check_device_errors on that stream returns SSM_ERR_DEVICE_TIMEOUT (and
 * the one after it SSM_OK).  No fault, trap or hang is involved; the context
 * stays usable.
 */
SSM_API ssm_status_t ssm_selftest_wait_timeout(void *stream);

/* Static, human-readable name of a status code. */
SSM_API const char *ssm_status_string(ssm_status_t status);

/* Version of the library as MAJOR * 10000 + MINOR * 100 + PATCH. */
SSM_API int ssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
