/*
 * libmuon: the Muon optimizer step on one GB300 (sm_103a), C ABI.
 *
 * The step (HyperParallel FSDP Muon RFC, mindspore hyper-parallel issue
 * "HyperParallel FSDP Muon优化器性能优化 RFC"):
 *   1. momentum   M' = beta*M + G;  V = G + beta*M' (Nesterov) or V = M'
 *                 (section 1(1): the orthogonalised matrix is the gradient
 *                 momentum M_t);
 *   2. normalise  X0 = V / (||V||_F + eps) per matrix slice;
 *   3. Newton-Schulz, T steps on the slice, worked on transposed when M > N
 *                 (sections 1 and 2: needs the whole matrix, depends only on
 *                 the last two dims):
 *                   A = X X^T;  B = b*A + c*A*A;  X <- a*X + B*X;
 *   4. update     W' = W*(1 - lr*wd) - lr*s*O,  s = sqrt(max(1, M/N))
 *                 (section 6: AdamW-style decoupled weight decay).
 * Slices whose trailing dims agree are regrouped into one batch and each
 * [E, M, N] tensor contributes E independent slices (sections 2 and 3).
 *
 * Ownership: the caller allocates and owns every device buffer (parameters,
 * gradients, momentum, workspace).  A plan owns host memory only.  muon_step
 * is asynchronous on the given stream, allocates nothing and never
 * synchronises the host.
 *
 * Errors: every call returns a muon_status; nothing aborts or throws.
 * Arguments are validated before any launch.  Launch failures return
 * MUON_ERR_CUDA.  A device-side wait that runs out of its iteration budget
 * writes an error word into the workspace header; muon_workspace_error reads
 * it.  Every kernel of a step checks that word when it starts and returns
 * at once when it is set, and a kernel whose own wait gave up stores no
 * parameter and no momentum after that point: such a step leaves the
 * parameters of the slices not yet updated as they were (momenta may have
 * advanced).  The word stays set until the caller clears it.
 *
 * Environment (read by the library at each call):
 *   MUON_LOG=1        muon_plan prints the plan to stderr (one line per
 *                     group: dims, dtype, slices, tr, scale, kernel, chunk,
 *                     workspace).
 *   MUON_FAULT=alloc  muon_plan fails as if host memory ran out
 *                     (MUON_ERR_NOMEM), before allocating anything.
 *   MUON_FAULT=launch the step calls fail as if the first launch had
 *                     failed (MUON_ERR_CUDA), after validating their
 *                     arguments and before any device work.
 *   MUON_FAULT=timeout every bounded device wait of the step kernels gives
 *                     up at once (budget of zero polls): the step records
 *                     MUON_ERR_DEVICE_TIMEOUT in the error word; each kernel
 *                     still waits, with the normal budget, for the copies it
 *                     has in flight before it returns.
 * These fault switches exist to test the callers' error paths; unset, they
 * cost one getenv per call.
 */
#ifndef MUON_H_
#define MUON_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MUON_API __attribute__((visibility("default")))
#else
#define MUON_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MUON_OK = 0,
  MUON_ERR_INVALID_ARG = -1,       /* null pointer, bad count, bad option   */
  MUON_ERR_UNSUPPORTED_SHAPE = -2, /* ndim not in {2,3}, a zero dimension    */
  MUON_ERR_DTYPE = -3,             /* dtype not MUON_BF16 / MUON_F32         */
  MUON_ERR_ALIGNMENT = -4,         /* workspace not 256-byte aligned         */
  MUON_ERR_CUDA = -5,              /* a CUDA runtime call failed             */
  MUON_ERR_DEVICE_TIMEOUT = -6,    /* a bounded device wait gave up          */
  MUON_ERR_WORKSPACE = -7,         /* workspace smaller than the plan needs  */
  MUON_ERR_NOMEM = -8              /* host memory allocation failed          */
} muon_status;

/* element types of parameters and gradients (momentum is always fp32) */
enum { MUON_BF16 = 0, MUON_F32 = 1 };

/* arithmetic of the Newton-Schulz products */
enum {
  /* 16-bit tensor-core operands, fp32 accumulation.  Dense groups iterate
   * in fp16: the iterates are normalised (spectral norm <= 1.21), so fp16
   * cannot overflow and carries three more mantissa bits than bf16.  The
   * fused kernel of skinny groups keeps V in bf16 and runs the m x m
   * recursion in fp32; its two products take bf16 operands. */
  MUON_MODE_TC16 = 0,
  /* fp32 operands and accumulation throughout (accuracy mode) */
  MUON_MODE_FP32 = 1
};

/* which kernel family a group runs on (reported by muon_plan_group) */
enum { MUON_KERNEL_SKINNY = 0, MUON_KERNEL_DENSE = 1 };

/* One parameter: [M, N] (ndim 2) or [E, M, N] (ndim 3), row-major,
 * contiguous.  dims[k] for k >= ndim is ignored. */
typedef struct {
  int ndim;
  int64_t dims[3];
  int dtype; /* MUON_BF16 or MUON_F32 */
} muon_shape;

typedef struct {
  int mode;             /* MUON_MODE_TC16 (default) or MUON_MODE_FP32        */
  float eps;            /* normalisation eps, default 1e-7                   */
  size_t workspace_cap; /* bytes; 0 = no cap.  Dense groups are processed in
                           chunks of slices that fit the cap; chunking never
                           changes results (slices are independent).        */
  int skinny_max_m;     /* groups with min(M,N) <= this run on the fused
                           skinny kernel when they fit on chip (default 64,
                           0 or negative disables the skinny kernel)        */
  int scale_mode;       /* update scale s of a [M, N] slice (the RFC does
                           not fix it): MUON_SCALE_SQRT_RATIO (default) or
                           MUON_SCALE_RMS_MATCH                             */
} muon_options;

/* update scale s in W' = W (1 - lr wd) - lr s O, rounded once to float */
enum {
  MUON_SCALE_SQRT_RATIO = 0, /* s = sqrt(max(1, M/N))                          */
  MUON_SCALE_RMS_MATCH = 1   /* s = 0.2 sqrt(max(M, N)): an update whose RMS is
                                about 0.2, like a typical AdamW step          */
};

typedef struct muon_plan_s muon_plan_t;

typedef struct {
  int64_t M, N;   /* slice dims as stored                                 */
  int64_t m, n;   /* working dims: m = min(M,N), n = max(M,N)             */
  int dtype;
  int count;      /* slices in the group                                   */
  int tr;         /* 1 when M > N: the slice is worked on transposed       */
  float scale;    /* update scale s of the options' scale_mode (float)     */
  int kernel;     /* MUON_KERNEL_SKINNY or MUON_KERNEL_DENSE               */
  int cluster;    /* skinny: CTAs per slice (thread-block cluster size)    */
  int chunk;      /* dense: slices per chunk under the workspace cap       */
} muon_group_info;

/* Fill *opt with the defaults listed above. */
MUON_API void muon_options_default(muon_options* opt);

/*
 * Build a plan (host only; no device call).  RFC section 3: slices are
 * grouped by key (M, N, dtype) in order of first appearance while walking
 * parameters in call order and slices e = 0..E-1 within each; a slice's
 * index in its group is its order of encounter.  shapes: n entries, host.
 * opt may be null (defaults).  On success *out receives a plan to be freed
 * with muon_plan_destroy.
 */
MUON_API muon_status muon_plan(const muon_shape* shapes, int n, const muon_options* opt,
                      muon_plan_t** out);

/* Device workspace bytes muon_step needs for this plan (>= 256). */
MUON_API muon_status muon_plan_workspace_bytes(const muon_plan_t* plan, size_t* out);
MUON_API muon_status muon_plan_num_groups(const muon_plan_t* plan, int* out);
MUON_API muon_status muon_plan_num_slices(const muon_plan_t* plan, int* out);
MUON_API muon_status muon_plan_group(const muon_plan_t* plan, int g, muon_group_info* out);
/* group id and index within the group of slice `slice` of parameter `param` */
MUON_API muon_status muon_plan_slice(const muon_plan_t* plan, int param, int slice,
                            int* group, int* index);

/*
 * One Muon step for every parameter of the plan, enqueued on `stream`
 * (a cudaStream_t; null = legacy default stream).
 *   params[p]   device, dtype of shape p, updated in place (RNE rounding)
 *   grads[p]    device, same dtype and shape, read only
 *   momentum[p] device, fp32, same shape, updated in place
 *   coeffs      host, 3 floats (a, b, c); null = (3.4445, -4.7750, 2.0315)
 *   ns_steps    T >= 0
 *   workspace   device, 256-byte aligned, >= muon_plan_workspace_bytes.
 *               Any content is valid on entry.  Passing the same workspace
 *               to the next step of the same plan keeps, per dense slice, the
 *               power of two that scales its first iterate; when it still
 *               fits, the step skips one pass over that slice.  The results
 *               do not depend on it.
 * Parameter, gradient and momentum buffers must not overlap one another.
 */
MUON_API muon_status muon_step(const muon_plan_t* plan, void* const* params,
                      const void* const* grads, float* const* momentum,
                      float lr, float beta, float wd, int nesterov,
                      int ns_steps, const float* coeffs, void* workspace,
                      size_t ws_bytes, void* stream);

/*
 * muon_step that also writes the orthogonalised momentum O (fp32, the
 * parameter's own shape and layout) of every slice into ortho[p], a device
 * buffer per parameter.  Used to check O itself against a reference.
 */
MUON_API muon_status muon_step_ortho(const muon_plan_t* plan, void* const* params,
                            const void* const* grads, float* const* momentum,
                            float lr, float beta, float wd, int nesterov,
                            int ns_steps, const float* coeffs, void* workspace,
                            size_t ws_bytes, void* stream, float* const* ortho);

/*
 * muon_step on loss-scaled gradients (mixed-precision training with a loss
 * scaler; the Paddle Muon sharding PR's review of its AMP GradScaler path
 * shows the Muon step running behind such a scaler).
 *   grads hold S * G for a loss scale S; the step uses G = grads * inv_scale
 *   (the multiply is fused into the momentum update, no extra pass).
 *   found_inf: device int.  Before any state changes, every gradient value of
 *   every parameter is checked; *found_inf is set to 1 when one is inf or NaN,
 *   and then no parameter and no momentum is modified (the step is skipped),
 *   else *found_inf is set to 0 and the step runs.  The check reads every
 *   gradient once more (2 bytes per bf16 element).
 * inv_scale must be finite.  Other arguments are those of muon_step.
 */
MUON_API muon_status muon_step_amp(const muon_plan_t* plan, void* const* params,
                                   const void* const* grads, float* const* momentum,
                                   float lr, float beta, float wd, int nesterov,
                                   int ns_steps, const float* coeffs, float inv_scale,
                                   int* found_inf, void* workspace, size_t ws_bytes,
                                   void* stream);

/*
 * AdamW for the parameters Muon does not orthogonalise (1-D biases and norm
 * scales, or any tensor the caller keeps off the Muon path; the Paddle Muon
 * sharding PR keeps separate 2-D and 1-D gradient buffers because the two
 * kinds take different update rules).  Standard AdamW, bias-corrected, with
 * decoupled weight decay, step t >= 1:
 *   m' = b1*m + (1-b1)*g;  v' = b2*v + (1-b2)*g^2
 *   W' = W*(1 - lr*wd) - lr * (m'/(1-b1^t)) / (sqrt(v'/(1-b2^t)) + eps)
 *   n tensors, each contiguous with numel[i] elements (any shape): params[i]
 *   and grads[i] of `dtype`, exp_avg[i] and exp_avg_sq[i] fp32 (updated in
 *   place).  All device pointers; one launch per 256 tensors.
 * Returns MUON_ERR_INVALID_ARG for null pointers, t < 1, betas outside [0,1),
 * negative eps or non-finite hyper-parameters.
 */
MUON_API muon_status muon_adamw_step(int n, void* const* params, const void* const* grads,
                                     float* const* exp_avg, float* const* exp_avg_sq,
                                     const int64_t* numel, int dtype, float lr, float beta1,
                                     float beta2, float eps, float wd, int step, void* stream);

/*
 * Read the device error word of a workspace after synchronising `stream`.
 * *code receives MUON_OK or the first device-side error recorded
 * (MUON_ERR_DEVICE_TIMEOUT); when clear != 0 the word is reset to zero.
 */
MUON_API muon_status muon_workspace_error(const void* workspace, void* stream, int clear,
                                 int* code);

/*
 * muon_step without a workspace argument, for callers that cannot allocate
 * device memory: a host runtime that hands nearly all of the GPU's memory to
 * its own pooled allocator at start-up, leaving none for a library's
 * cudaMalloc, or a latency-bound caller that cannot afford a cudaMalloc,
 * which may block and synchronise the device.  The RFC has no counterpart of
 * this call.
 *
 * The scratch is one static device array of MUON_STATIC_WORKSPACE_BYTES,
 * held by every GPU that loads the library until the process exits; no call
 * allocates or frees anything.  Plans whose muon_plan_workspace_bytes exceed
 * that size are rejected with MUON_ERR_WORKSPACE before any device work.
 * The first call on each device, with that device current, looks up the
 * array's device address and caches it; make that first call before any
 * stream capture.  The cache assumes the device is not reset
 * (cudaDeviceReset) while the library is loaded.  `stream` must belong to the
 * current device (else MUON_ERR_INVALID_ARG).  Every call shares the array
 * and finds the previous call's contents there: the device error word is
 * cleared at each call, everything else is written before it is read.  Calls
 * whose work overlaps on the GPU (streams with no ordering between them) race
 * on the array.  A device-side wait that gave up during the step is reported
 * by muon_static_error, not by the return code.  Other arguments are those of
 * muon_step.
 */
#define MUON_STATIC_WORKSPACE_BYTES (32u << 20)
MUON_API muon_status muon_step_static(const muon_plan_t* plan, void* const* params,
                                      const void* const* grads, float* const* momentum,
                                      float lr, float beta, float wd, int nesterov,
                                      int ns_steps, const float* coeffs, void* stream);

/*
 * The device error word that the last muon_step_static on the current device
 * left in the static array, read after synchronising `stream` (which must
 * belong to the current device): *code receives MUON_OK or
 * MUON_ERR_DEVICE_TIMEOUT; when clear != 0 the word is reset to zero.  Call
 * it before the next muon_step_static, which clears the word.  Allocates
 * nothing.  The RFC has no counterpart of this call.
 */
MUON_API muon_status muon_static_error(void* stream, int clear, int* code);

/* kernel classes of muon_step_timed */
enum {
  MUON_KC_SKINNY = 0,  /* fused on-chip kernel of the skinny groups              */
  MUON_KC_FRONT = 1,   /* dense path: momentum, V, partial sums of V^2           */
  MUON_KC_NORM = 2,    /* dense path: 1/(||V|| + eps) and the 16-bit X0          */
  MUON_KC_GEMM = 3,    /* dense path: the tcgen05 (or fp32) Newton-Schulz products */
  MUON_KC_UPDATE = 4,  /* dense path: separate update kernel (O requested)       */
  MUON_KC_CHECK = 5,   /* loss-scaled step: non-finite check of the gradients    */
  MUON_KC_COUNT = 6
};
typedef struct {
  float ms[MUON_KC_COUNT];   /* device time summed over the launches of a class  */
  int launches[MUON_KC_COUNT];
} muon_kernel_times;

/*
 * muon_step with a CUDA event recorded on `stream` before every kernel
 * launch and after the last one; synchronises `stream` and writes the device
 * time of each kernel class into *times (host).  An event between two
 * launches keeps a kernel from overlapping its predecessor's tail, so the
 * classes can sum to slightly more than a muon_step of the same plan takes.
 * For measurement: it creates and destroys its events (host-side driver
 * objects, no device memory).  Other arguments are those of muon_step.
 */
MUON_API muon_status muon_step_timed(const muon_plan_t* plan, void* const* params,
                                     const void* const* grads, float* const* momentum,
                                     float lr, float beta, float wd, int nesterov, int ns_steps,
                                     const float* coeffs, void* workspace, size_t ws_bytes,
                                     void* stream, muon_kernel_times* times);

/*
 * muon_step on parameters, gradients and momenta held in HOST memory (an
 * optimizer whose state lives in host memory; on a Grace-Blackwell node the
 * GPU reaches it over NVLink-C2C).  `staging` is cut into
 * nbuf = staging_bytes / unit_bytes buffers (2 to 16) and the plan's slices
 * into units of whole slices that fit one; each unit's parameters, gradients
 * and momenta are copied to the device, stepped by the kernels of muon_step,
 * and its parameters and momenta copied back, the copies of one unit
 * overlapping the kernels of its neighbours (two copy streams of the call's
 * own).  The kernels do not wait as long as a unit's copies in and out take
 * at most about nbuf - 1 times as long as its kernels.
 *   params, grads, momentum  host pointers (page-locked memory gives full
 *                            copy bandwidth, and muon_host_alloc's keeps it
 *                            when the state is cold; pageable memory works,
 *                            slower), shapes and dtypes as for muon_step
 *   workspace, ws_bytes      device, as for muon_step
 *   staging, staging_bytes   device, 256-byte aligned
 *   unit_bytes               staging bytes of one unit, at least
 *                            muon_plan_host_unit_bytes; larger units mean
 *                            fewer launches and a longer pipeline fill and
 *                            drain
 * Asynchronous: the work is ordered before any later work on `stream`;
 * synchronise `stream` before reading the host buffers.  Returns
 * MUON_ERR_WORKSPACE when one slice does not fit unit_bytes or the staging
 * holds fewer than two units.  Other arguments are those of muon_step.  The
 * RFC has no counterpart of this call.
 */
MUON_API muon_status muon_step_host(const muon_plan_t* plan, void* const* params,
                                    const void* const* grads, float* const* momentum, float lr,
                                    float beta, float wd, int nesterov, int ns_steps,
                                    const float* coeffs, void* workspace, size_t ws_bytes,
                                    void* staging, size_t staging_bytes, size_t unit_bytes,
                                    void* stream);
/* smallest unit_bytes of muon_step_host: the largest slice's parameter,
 * gradient and momentum, each 256-byte aligned (host only, no device call) */
MUON_API muon_status muon_plan_host_unit_bytes(const muon_plan_t* plan, size_t* out);

/*
 * Page-locked host memory for the state muon_step_host streams: `bytes`
 * rounded up to the kernel's transparent-huge-page size (the PMD size, read
 * from sysfs; 2 MiB if it cannot be read), mapped at an address aligned to
 * it, advised for huge pages, faulted in and registered with the CUDA driver
 * (portable).  Huge pages keep the device's reads of state it has not touched
 * for a while at full speed; with the base pages of the ordinary allocators,
 * such cold reads ran at a fraction of the link's bandwidth on some
 * allocations.  Where the kernel has no transparent huge pages the memory is
 * still page-locked, on base pages.  *out (host) receives the address (NULL
 * on failure); the memory reads as zeros.  Returns MUON_ERR_INVALID_ARG for
 * bytes == 0 or out == NULL, MUON_ERR_NOMEM when the mapping fails (or under
 * MUON_FAULT=alloc), MUON_ERR_CUDA when the registration fails (no device,
 * or the driver refuses); nothing is held then.  Ownership: the caller's,
 * until muon_host_free.
 */
MUON_API muon_status muon_host_alloc(size_t bytes, void** out);
/* Unregisters and unmaps memory from muon_host_alloc.  NULL is a no-op;
 * MUON_ERR_INVALID_ARG for an address muon_host_alloc did not return (or
 * already freed).  No device work may still use the memory. */
MUON_API muon_status muon_host_free(void* p);

/* Kernel launches muon_step makes for this plan and ns_steps, for a step
 * without O outputs (for accounting; no device call). */
MUON_API muon_status muon_plan_launches(const muon_plan_t* plan, int ns_steps, int* out);

/*
 * Assignment of the plan's slices to `world` replicas that all hold every
 * parameter (HyperParallel FSDP Muon RFC, section 4, HSDP grouped
 * computation: each replica group orthogonalises only the parameters that a
 * greedy algorithm assigns to it for an even compute load, then the updated
 * parameters are broadcast; section 2: the E slices of an [E, M, N] tensor
 * are independent, so the unit of assignment is a slice).  Host only, no
 * device call; the result depends only on the plan's shapes and the
 * arguments, so every replica computes the same assignment without
 * communicating.
 *
 * Load of a slice (seconds on the roofline of one GPU):
 *   max(T (4 m^2 n + 2 m^3) / flops_per_s,  m n (3 es + 8) / bytes_per_s)
 * with m = min(M, N), n = max(M, N), T = ns_steps, es = 2 (bf16) or 4 (fp32):
 * standard Newton-Schulz flop count, and the optimizer state touched once
 * (gradient read, parameter read and written, fp32 momentum read and
 * written).  Greedy longest first: slices in decreasing load (equal loads:
 * lower global slice id first), each to the replica with the least summed
 * load so far (equal sums: lower rank).
 *   owner      host, muon_plan_num_slices ints, written: owner[s] is the rank
 *              of global slice s (parameters in plan order, slices e = 0..E-1
 *              of each)
 *   rank_load  host, `world` doubles, written, or null: summed load per rank
 * Errors: MUON_ERR_INVALID_ARG for a null plan or owner, world < 1,
 * ns_steps < 0, or a rate that is not finite and positive.
 */
MUON_API muon_status muon_plan_partition(const muon_plan_t* plan, int world, int ns_steps,
                                         double flops_per_s, double bytes_per_s, int* owner,
                                         double* rank_load);

MUON_API void muon_plan_destroy(muon_plan_t* plan);
MUON_API const char* muon_status_string(muon_status s);

#ifdef __cplusplus
}
#endif

#endif /* MUON_H_ */
